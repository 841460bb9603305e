"""bench.py's accounting, on CPU: the flop count its TFLOP/s figures divide by (4 B H Nq Nk d for the
forward, 2.5 times that for the backward, halved under a causal mask), the visible-pair count, and the
config object of the JSON line."""
import bench
from exact_head_attention_gb300 import workloads


def test_flops_of_the_bench_workload():
    w = workloads.WORKLOADS["long8k_causal_bf16"]
    fwd, bwd = bench.step_flops(w)
    assert fwd == 4 * 1 * 12 * 8192 * 8192 * 128 / 2 == 206158430208
    assert bwd == 2.5 * fwd
    assert bench.config_dict(w)["flops_per_step"] == fwd + bwd == 721554505728


def test_flops_without_a_mask_are_not_halved():
    w = workloads.WORKLOADS["self1k_bf16"]
    fwd, bwd = bench.step_flops(w)
    assert fwd == 4 * 8 * 16 * 1024 * 1024 * 64 and bwd == 2.5 * fwd


def test_visible_pairs_by_mask():
    assert bench.visible_pairs(workloads.custom(1, 1, 5, 7, 64, "bf16", False)) == 35
    assert bench.visible_pairs(workloads.custom(1, 1, 5, 5, 64, "bf16", True)) == 15          # 1 + 2 + ... + 5
    assert bench.visible_pairs(workloads.custom(1, 1, 3, 5, 64, "bf16", "bottom_right")) == 12  # 3 + 4 + 5
    assert bench.visible_pairs(workloads.custom(1, 1, 5, 3, 64, "bf16", "bottom_right")) == 6   # 0 + 0 + 1 + 2 + 3


def test_config_names_the_workload_and_no_model():
    c = bench.config_dict(workloads.WORKLOADS["long8k_causal_bf16"], {"parallelism": "single GPU"})
    assert c["workload"] == "long8k_causal_bf16" and c["parallelism"] == "single GPU"
    assert "model" not in c
    assert (c["B"], c["H"], c["Nq"], c["Nk"], c["d"], c["causal"]) == (1, 12, 8192, 8192, 128, True)
