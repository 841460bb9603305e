"""CPU checks of the GPU tests' own helpers: the half-ulp allowance of the O comparison agrees with torch's
rounding to bf16 and fp16, and the relative-L2 floor behaves as documented."""
import numpy as np
import torch

from parity import half_ulp, rel_l2


def test_half_ulp_bounds_round_to_nearest_and_is_attained():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.uniform(-6, 6, 200000), rng.uniform(-1e-3, 1e-3, 20000), [2.0, 4.0, -4.0, 1.0]])
    for dtype, tdt in (("bf16", torch.bfloat16), ("fp16", torch.float16)):
        # torch rounds fp64 -> fp32 -> 16 bits: the first step adds at most 2^-24 |x|
        r = torch.from_numpy(x).to(tdt).double().numpy()
        err = np.abs(r - x)
        assert (err <= half_ulp(x, dtype) + 2.0 ** -23 * np.abs(x)).all(), dtype
        # a value halfway between two neighbours (one ulp apart at 2.0..4.0) is off by exactly half an ulp
        ulp = 2.0 ** (1 - (7 if dtype == "bf16" else 10))
        mid = 2.0 + ulp / 2
        assert abs(float(torch.tensor(mid, dtype=torch.float64).to(tdt)) - mid) == half_ulp(mid, dtype)


def test_rel_l2_floor():
    b = np.zeros(100)
    a = np.full(100, 2e-5)
    assert abs(rel_l2(a, b) - 2e-2) < 1e-12   # RMS error 2e-5 against a zero reference sits at the bound
    b = np.ones(100)
    assert abs(rel_l2(b * 1.01, b) - 1e-2) < 1e-12
