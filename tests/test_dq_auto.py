"""The rule ATTN_DQ_AUTO follows (attn_bwd_auto_dq_mode), checked on CPU with GB300's SM count and L2
size passed explicitly: each case is a shape whose two backward modes were timed on a GB300, and the
expected mode is the one that measured faster (atomic where they tied)."""
import pytest

from exact_head_attention_gb300 import exattn

SMS, L2 = 152, 126 << 20

CASES = [
    # B, H, N, d, causal, faster mode on GB300
    ((16, 16, 2048, 128, False), "deterministic"),   # 256 MiB accumulator, one head per SM or more
    ((32, 16, 1024, 128, False), "deterministic"),
    ((16, 16, 4096, 128, False), "deterministic"),
    ((64, 16, 512, 128, False), "atomic"),           # 4 key blocks per head
    ((8, 16, 2048, 128, False), "atomic"),           # 128 heads: a head's key blocks run in the same waves
    ((4, 16, 8192, 128, False), "atomic"),
    ((2, 16, 8192, 128, False), "atomic"),
    ((4, 16, 4096, 128, False), "atomic"),
    ((16, 16, 2048, 64, False), "atomic"),           # d = 64
    ((32, 16, 2048, 64, False), "atomic"),
    ((16, 16, 2048, 128, True), "atomic"),           # causal: half the revisits (the two modes tie)
    ((32, 16, 2048, 128, True), "atomic"),
    ((64, 16, 1024, 128, True), "atomic"),
    ((1, 12, 8192, 128, True), "atomic"),            # the bench workload
    ((1, 8, 32768, 128, True), "atomic"),
    ((4, 16, 16384, 128, True), "atomic"),
    ((1, 1, 65536, 128, False), "atomic"),           # one head: every key block adds into the same rows at once
]


@pytest.mark.parametrize("shape,want", CASES, ids=[str(c[0]) for c in CASES])
def test_auto_matches_the_faster_measured_mode(shape, want):
    B, H, N, d, causal = shape
    assert exattn.auto_dq_mode(B, H, N, N, d, causal, SMS, L2) == want


def test_auto_rejects_invalid_sizes():
    with pytest.raises(ValueError):
        exattn.auto_dq_mode(0, 1, 128, 128, 64, False, SMS, L2)
    with pytest.raises(ValueError):
        exattn.auto_dq_mode(1, 1, 128, 128, 96, False, SMS, L2)
