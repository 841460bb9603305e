"""The rule ATTN_DQ_AUTO follows (attn_bwd_auto_dq_mode), checked on CPU: the reductions on every shape
whose two backward modes were timed on a GB300 (the reductions measured faster on all of them), and
-1 (ValueError here) for sizes the backward rejects."""
import pytest

from exact_head_attention_gb300 import exattn

MEASURED = [
    # B, H, N, d, causal: 48 MiB to 512 MiB of fp32 accumulator, both launch orders, d = 64 and 128
    (1, 12, 8192, 128, True), (2, 16, 8192, 128, True), (16, 16, 2048, 128, True), (32, 16, 2048, 128, True),
    (64, 16, 1024, 128, True), (4, 16, 16384, 128, True), (2, 16, 8192, 128, False), (4, 16, 4096, 128, False),
    (8, 16, 2048, 128, False), (64, 16, 512, 128, False), (16, 16, 2048, 64, False), (32, 16, 2048, 64, False),
    (16, 16, 2048, 128, False), (32, 16, 1024, 128, False), (16, 16, 4096, 128, False), (4, 16, 8192, 128, False),
]


@pytest.mark.parametrize("shape", MEASURED, ids=str)
def test_auto_takes_the_reductions(shape):
    B, H, N, d, causal = shape
    assert exattn.auto_dq_mode(B, H, N, N, d, causal) == "atomic"
    assert exattn.auto_dq_mode(B, H, N, N, d, "bottom_right" if causal else False) == "atomic"


@pytest.mark.parametrize("dims", [(0, 1, 128, 128, 64), (1, 0, 128, 128, 64), (1, 1, 0, 128, 64), (1, 1, 128, 0, 64),
                                  (1, 1, 128, 128, 96), (-1, 1, 128, 128, 128)], ids=str)
def test_auto_rejects_invalid_sizes(dims):
    with pytest.raises(ValueError):
        exattn.auto_dq_mode(*dims, False)
