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


SMS, L2 = 152, 135528448  # GB300: SM count and the L2 size the device reports

# (B, H, N, d, causal) -> heads per launch group of the reducing backward, as in the measured table
GROUPS = [
    ((1, 12, 8192, 128, True), 12),    # 48 MiB accumulator, causal: heads fastest
    ((1, 8, 32768, 64, True), 8),      # 64 MiB, at most half of L2
    ((1, 8, 32768, 128, True), 2),     # 16 MiB per head: one fits in L2/16, but 256 key blocks need 2 heads
    ((2, 16, 8192, 128, True), 5),     # 4 MiB per head: 2 fit; 64 key blocks need 5
    ((16, 16, 2048, 128, True), 19),   # 1 MiB: 8 fit; 16 key blocks need 19
    ((32, 16, 2048, 128, True), 19),
    ((64, 16, 1024, 128, True), 38),
    ((4, 16, 16384, 128, True), 3),
    ((1, 1, 32768, 128, False), 1),    # one head
    ((1, 1, 65536, 128, False), 1),
    ((2, 16, 8192, 128, False), 2),    # no mask: as many heads as fit in L2/16
    ((4, 16, 4096, 128, False), 4),
    ((8, 16, 2048, 128, False), 8),
    ((16, 16, 2048, 64, False), 16),
    ((4, 16, 8192, 128, False), 2),
    ((16, 16, 2048, 128, False), 8),
    ((32, 16, 1024, 128, False), 16),
    ((64, 16, 512, 128, False), 32),
    ((32, 16, 2048, 64, False), 16),
    ((16, 16, 4096, 128, False), 4),
    ((8, 16, 1024, 64, False), 128),   # 32 MiB, within a quarter of L2: heads fastest
]


@pytest.mark.parametrize("shape,want", GROUPS, ids=[str(g[0]) for g in GROUPS])
def test_launch_group_rule(shape, want):
    B, H, N, d, causal = shape
    assert exattn.head_group(B, H, N, N, d, causal, SMS, L2) == want


def test_launch_group_limits():
    # the quarter / half of L2 thresholds, one byte either side
    rows = 8192  # one head of 8192 rows, d = 128: 4 MiB of accumulator
    per_head = rows * 128 * 4
    assert exattn.head_group(1, 8, rows, rows, 128, False, SMS, 8 * per_head * 4) == 8
    assert exattn.head_group(1, 8, rows, rows, 128, False, SMS, 8 * per_head * 4 - 1) < 8
    assert exattn.head_group(1, 8, rows, rows, 128, True, SMS, 8 * per_head * 2) == 8
    assert exattn.head_group(1, 8, rows, rows, 128, True, SMS, 8 * per_head * 2 - 1) < 8
    # never above B*H, never below 1; a ragged Nq counts its padded rows
    assert exattn.head_group(1, 3, 2048, 2048, 128, True, SMS, 1 << 20) == 3  # the causal floor, 19, capped at B*H
    assert exattn.head_group(4, 16, 8192, 8192, 128, False, SMS, 1 << 20) == 1
    assert exattn.head_group(1, 64, 129, 129, 64, False, SMS, 64 * 256 * 64 * 4 * 4) == 64
    for bad in ((0, 1, 128, 128, 64), (1, 1, 128, 128, 96), (1 << 16, 1 << 8, 128, 1 << 14, 64)):
        with pytest.raises(ValueError):
            exattn.head_group(*bad, False, SMS, L2)
