"""How the causal forward is spread over the SMs (attn_fwd_schedule), checked on CPU with the SM count
passed explicitly: where the launch order would leave SMs idle, the blocks are packed into one list
per SM, each block on exactly one list, and the busiest list carries less causal work than the
heaviest-first spread of the launch order does."""
import heapq

import pytest

from exact_head_attention_gb300 import exattn

SMS = 152


def block_work(Nq, Nk, causal_off):
    """Causal work of each 256-row query block: the (128-row query tile, 128-row key tile) pairs it visits,
    a tile pair counted when some query row of the tile sees some key of the key tile."""
    nkv = -(-Nk // 128)
    work = []
    for qb in range(-(-Nq // 256)):
        w = 0
        for t in range(2):
            last_row = min(Nq, qb * 256 + (t + 1) * 128) - 1
            if qb * 256 + t * 128 >= Nq:
                last_row = qb * 256 + t * 128 + 127  # a padding tile still runs its key tiles
            w += max(0, min(nkv, (last_row + causal_off) // 128 + 1))
        work.append(w)
    return work


def heaviest_first(costs, sms):
    loads = [0] * sms
    heap = [(0, i) for i in range(sms)]
    for c in sorted(costs, reverse=True):
        load, i = heapq.heappop(heap)
        loads[i] = load + c
        heapq.heappush(heap, (loads[i], i))
    return max(loads)


@pytest.mark.parametrize("shape", [(1, 12, 8192, 8192, 128, True), (1, 12, 8192, 8192, 64, True),
                                   (2, 6, 8192, 8192, 128, True), (1, 12, 8100, 8100, 128, True)], ids=str)
def test_coarse_causal_grids_are_packed(shape):
    B, H, Nq, Nk, d, causal = shape
    lists = exattn.fwd_schedule(B, H, Nq, Nk, d, causal, SMS)
    assert lists is not None and len(lists) == SMS
    nqb = -(-Nq // 256)
    flat = sorted(b for lst in lists for b in lst)
    assert flat == list(range(B * H * nqb)), "every block on exactly one list"
    assert all(lst for lst in lists)
    work = block_work(Nq, Nk, 0)
    busiest = max(sum(work[b % nqb] for b in lst) for lst in lists)
    assert busiest < heaviest_first([work[b % nqb] for b in range(B * H * nqb)], SMS)


@pytest.mark.parametrize("shape", [
    (1, 12, 8192, 8192, 128, False),    # no mask: equal blocks
    (1, 4, 8192, 8192, 128, True),      # 128 blocks: one wave
    (1, 8, 32768, 32768, 128, True),    # 6-7 blocks per SM: the launch order is already even
    (2, 16, 8192, 8192, 128, True),
    (8, 16, 1024, 1024, 64, True),      # d = 64 over at most 2048 keys: one query tile per CTA, two per SM
    (1, 12, 2048, 2048, 64, True),
    (2, 8, 512, 2048, 64, "bottom_right"),
    (4, 16, 16384, 16384, 128, True),   # 4096 blocks: more than a list holds
], ids=str)
def test_other_grids_keep_the_launch_order(shape):
    assert exattn.fwd_schedule(*shape, SMS) is None


def test_bottom_right_mask_and_other_sm_counts():
    for sms in (132, 148, SMS):
        for (Nq, Nk) in ((8192, 8192), (8000, 9000)):
            lists = exattn.fwd_schedule(1, 12, Nq, Nk, 128, "bottom_right", sms)
            if lists is None:
                continue
            assert len(lists) == sms
            assert sorted(b for lst in lists for b in lst) == list(range(12 * (-(-Nq // 256))))


def test_invalid_sizes():
    for bad in ((0, 1, 128, 128, 64, True), (1, 1, 128, 128, 96, True)):
        with pytest.raises(ValueError):
            exattn.fwd_schedule(*bad, SMS)
