"""Seeded synthetic attention workloads.

This module holds only shapes, distributions and random-number generation: it
contains none of the attention arithmetic, and it is the one piece of code that
both the CUDA path's tests/benchmark and the CPU oracle consume, so the same
bits reach both.

Recipe: every tensor is drawn on the CPU from its own ``torch.Generator``
seeded ``1000 * config_index + tensor_index + seed_offset`` as fp32 normal
samples times the tensor's standard deviation, then rounded (round to nearest
even) to the workload dtype.  Tensor indices: q=0, k=1, v=2, dO=3.

The workloads are the long-sequence / small-batch regime of "Fast Transformer
training with long sequences" (attention layer benchmark: H = 12, d = 128,
sequence 8k) and the encoder-decoder MHA of SparkAttention (arXiv 2502.12784),
Figure 1 (masked decoder self-attention and encoder-decoder cross-attention).
The two decoding workloads are the small-query regime the StreamKL summary
names for its split-K variant (autoregressive decoding, N_Q = 1, long
contexts): one new token, or a chunk of 64, attending to a long cache with the
bottom-right causal mask, on the heads of the 8k benchmark (H = 12, d = 128)
and of the SparkAttention decoder (H = 16, d = 64).
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int          # seed family
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    dtype: str          # "bf16" | "fp16"
    causal: bool | str  # False, True (top-left) or "bottom_right"
    sigma_qk: float = 1.0
    sigma_v: float = 1.0
    sigma_do: float = 1.0
    kind: str = "train"  # "train": forward + backward; "decode": forward only (split-KV); "kl": attention KL

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self) -> torch.dtype:
        return {"bf16": torch.bfloat16, "fp16": torch.float16}[self.dtype]

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five training workload families (two have a causal and a non-causal / d variant) and two
# decoding workloads.
WORKLOADS = {
    "tiny_fp16": Workload("tiny_fp16", 1, 1, 2, 128, 128, 64, "fp16", False),
    "self1k_bf16": Workload("self1k_bf16", 2, 8, 16, 1024, 1024, 64, "bf16", False),
    "self1k_causal_bf16": Workload("self1k_causal_bf16", 2, 8, 16, 1024, 1024, 64, "bf16", True),
    "dec_self512_fp16": Workload("dec_self512_fp16", 3, 16, 16, 512, 512, 64, "fp16", True),
    "dec_cross512x1024_fp16": Workload("dec_cross512x1024_fp16", 3, 16, 16, 512, 1024, 64, "fp16", False),
    "long8k_causal_bf16": Workload("long8k_causal_bf16", 4, 1, 12, 8192, 8192, 128, "bf16", True,
                                   sigma_qk=1.5),
    "ctx32k_d128_causal_bf16": Workload("ctx32k_d128_causal_bf16", 5, 1, 8, 32768, 32768, 128, "bf16", True),
    "ctx32k_d64_causal_bf16": Workload("ctx32k_d64_causal_bf16", 5, 1, 8, 32768, 32768, 64, "bf16", True),
    # decoding (split-KV forward)
    "decode_q1_kv32k_d128_bf16": Workload("decode_q1_kv32k_d128_bf16", 6, 8, 12, 1, 32768, 128, "bf16",
                                          "bottom_right", kind="decode"),
    "chunk_q64_kv16k_d64_fp16": Workload("chunk_q64_kv16k_d64_fp16", 8, 4, 16, 64, 16384, 64, "fp16",
                                         "bottom_right", kind="decode"),
    # attention KL divergence (teacher and student attention of one layer)
    "kl8k_causal_bf16": Workload("kl8k_causal_bf16", 9, 1, 12, 8192, 8192, 128, "bf16", True, kind="kl"),
}

# Student queries and keys of the KL workloads: the teacher's plus noise of this standard deviation.
KL_STUDENT_NOISE = 0.5

# The workload the throughput metric is quoted on.
HEADLINE = "long8k_causal_bf16"


def _normal(shape, seed: int, sigma: float, dtype: torch.dtype) -> torch.Tensor:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if sigma != 1.0:
        x = x * sigma
    return x.to(dtype)


def make_inputs(w: Workload, seed_offset: int = 0, with_grad_out: bool = True) -> dict:
    """CPU tensors q, k, v (and dO) in the workload dtype, layout [B, H, N, d]."""
    base = 1000 * w.index + seed_offset
    dt = w.torch_dtype
    out = {
        "q": _normal((w.B, w.H, w.Nq, w.d), base + 0, w.sigma_qk, dt),
        "k": _normal((w.B, w.H, w.Nk, w.d), base + 1, w.sigma_qk, dt),
        "v": _normal((w.B, w.H, w.Nk, w.d), base + 2, w.sigma_v, dt),
    }
    if with_grad_out:
        out["do"] = _normal((w.B, w.H, w.Nq, w.d), base + 3, w.sigma_do, dt)
    return out


def make_kl_inputs(w: Workload, seed_offset: int = 0) -> dict:
    """CPU tensors q1, k1 (teacher), q2, k2 (student) in the workload dtype and the upstream gradient g (fp32).

    The student's queries and keys are the teacher's plus independent noise (a student close to its
    teacher, as in attention distillation), drawn before rounding to the dtype.  Tensor indices: q1=0,
    k1=1, noise of q2=2, noise of k2=3, g=4."""
    base = 1000 * w.index + seed_offset
    dt = w.torch_dtype
    q1 = _normal((w.B, w.H, w.Nq, w.d), base + 0, w.sigma_qk, torch.float32)
    k1 = _normal((w.B, w.H, w.Nk, w.d), base + 1, w.sigma_qk, torch.float32)
    q2 = q1 + _normal((w.B, w.H, w.Nq, w.d), base + 2, KL_STUDENT_NOISE, torch.float32)
    k2 = k1 + _normal((w.B, w.H, w.Nk, w.d), base + 3, KL_STUDENT_NOISE, torch.float32)
    g = _normal((w.B, w.H, w.Nq), base + 4, 1.0, torch.float32)
    return {"q1": q1.to(dt), "k1": k1.to(dt), "q2": q2.to(dt), "k2": k2.to(dt), "g": g}


def custom(B: int, H: int, Nq: int, Nk: int, d: int, dtype: str = "bf16", causal: bool | str = False,
           index: int = 7, sigma_qk: float = 1.0) -> Workload:
    """An ad-hoc workload (ragged and edge-case shapes in the tests)."""
    mask = "br" if causal == "bottom_right" else ("c" if causal else "nc")
    name = f"custom_B{B}_H{H}_q{Nq}_k{Nk}_d{d}_{dtype}_{mask}"
    return Workload(name, index, B, H, Nq, Nk, d, dtype, causal, sigma_qk=sigma_qk)
