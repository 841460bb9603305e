"""C-ABI boundary checks that need no GPU: the library loads, exports every
function include/exattn.h declares, and rejects bad arguments before touching
the device (fake, never-dereferenced pointers are used)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from exact_head_attention_gb300 import build, exattn
    build.build()
    return exattn.load()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "exattn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert {"attn_fwd", "attn_bwd", "attn_bwd_workspace_size", "attn_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    from exact_head_attention_gb300 import exattn
    for code in range(8):
        assert exattn.status_string(code)
    assert exattn.status_string(99) == "unknown status"


def test_workspace_size(lib):
    from exact_head_attention_gb300 import exattn
    # fp32 dQ accumulator over 128-row padded queries + two fp32 row vectors, each 256-byte aligned
    assert exattn.workspace_size(1, 12, 8192, 128) == 12 * 8192 * 128 * 4 + 2 * 12 * 8192 * 4
    rows = 2 * 3 * 256
    assert exattn.workspace_size(2, 3, 129, 64) == rows * 64 * 4 + 2 * ((rows * 4 + 255) // 256 * 256)
    for bad in ((0, 1, 1, 64), (1, 0, 1, 64), (1, 1, 0, 64), (1, 1, 1, 96)):
        assert exattn.workspace_size(*bad) == 0


FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation happens first


def _fwd(lib, B=1, H=1, Nq=128, Nk=128, d=64, causal=0, scale=0.125, dtype=0, ptrs=None):
    p = ptrs or [FAKE] * 5
    return lib.attn_fwd(*[ctypes.c_void_p(x) if x is not None else None for x in p],
                        B, H, Nq, Nk, d, causal, scale, dtype, None)


@pytest.mark.parametrize("kw,code", [
    (dict(B=0), 1), (dict(H=-1), 1), (dict(Nq=0), 1), (dict(Nk=0), 1),
    (dict(scale=0.0), 1), (dict(scale=-1.0), 1), (dict(scale=float("nan")), 1), (dict(scale=float("inf")), 1),
    (dict(dtype=7), 1), (dict(d=96), 2), (dict(d=256), 2), (dict(Nq=65536 * 256), 1),
    (dict(ptrs=[FAKE, None, FAKE, FAKE, FAKE]), 1),
    (dict(ptrs=[FAKE, FAKE, FAKE + 8, FAKE, FAKE]), 3),
    (dict(ptrs=[FAKE, FAKE, FAKE, FAKE, FAKE + 4]), 3),
])
def test_fwd_rejects_bad_arguments(lib, kw, code):
    assert _fwd(lib, **kw) == code


def _bwd(lib, ws=FAKE, ws_bytes=None, ptrs=None, d=64, **kw):
    B, H, Nq, Nk = kw.get("B", 1), kw.get("H", 1), kw.get("Nq", 128), kw.get("Nk", 128)
    need = lib.attn_bwd_workspace_size(B, H, Nq, d)
    p = ptrs or [FAKE] * 9
    return lib.attn_bwd(*[ctypes.c_void_p(x) if x is not None else None for x in p],
                        B, H, Nq, Nk, d, 0, 0.125, 0, ctypes.c_void_p(ws) if ws else None,
                        need if ws_bytes is None else ws_bytes, None)


def test_bwd_rejects_bad_arguments(lib):
    assert _bwd(lib, B=0) == 1
    assert _bwd(lib, d=80) == 2
    assert _bwd(lib, ptrs=[FAKE] * 8 + [None]) == 1
    assert _bwd(lib, ws=None) == 6
    assert _bwd(lib, ws_bytes=100) == 6
    assert _bwd(lib, ptrs=[FAKE] * 6 + [FAKE + 2] + [FAKE] * 2) == 3
    assert _bwd(lib, ws=FAKE + 16) == 3  # workspace must be 256-byte aligned
    # launch limits: 65535 key blocks per head, and B*H*key blocks numbered in an int
    assert _bwd(lib, Nk=65535 * 128 + 1) == 1
    assert _bwd(lib, B=1 << 16, H=1 << 8, Nk=1 << 14) == 1
    assert _bwd(lib, B=1 << 16, H=1 << 8, Nk=(1 << 14) - 128, ws=FAKE + 16) == 3  # one block fewer: size accepted


@pytest.mark.parametrize("causal,code", [(3, 1), (-1, 1), (100, 1)])
def test_rejects_unknown_mask(lib, causal, code):
    assert _fwd(lib, causal=causal) == code
    p = [ctypes.c_void_p(FAKE)] * 9
    need = lib.attn_bwd_workspace_size(1, 1, 128, 64)
    assert lib.attn_bwd(*p, 1, 1, 128, 128, 64, causal, 0.125, 0, ctypes.c_void_p(FAKE), need, None) == code


def _strided_fwd(lib, strides, B=2, H=3, Nq=128, Nk=128, d=64, causal=0, lse=FAKE + 4):
    # The LSE pointer is misaligned on purpose: a call that passes every other check stops there
    # (ATTN_ERR_MISALIGNED, after the stride checks) and never launches on the fake pointers.
    from exact_head_attention_gb300.exattn import Strides
    args = []
    for st in strides:
        args += [ctypes.c_void_p(FAKE), Strides(*st)]
    return lib.attn_fwd_strided(*args, ctypes.c_void_p(lse), B, H, Nq, Nk, d, causal, 0.125, 0, None)


@pytest.mark.parametrize("bad", [
    (3 * 128 * 64, 128 * 64, 32),         # row stride below d
    (3 * 128 * 64, 128 * 64, 68),         # row stride not a multiple of 8 elements
    (3 * 128 * 64, 100, 64),              # head stride not a multiple of 8
    (0, 128 * 64, 64),                    # zero batch stride with B > 1
    (3 * 128 * 64, -128 * 64, 64),        # negative head stride
    (1 << 40, 128 * 64, 64),              # byte stride beyond 2^40
])
def test_strided_rejects_bad_strides(lib, bad):
    good = (3 * 128 * 64, 128 * 64, 64)
    for i in range(4):
        strides = [good] * 4
        strides[i] = bad
        assert _strided_fwd(lib, strides) == 1, (i, bad)


def test_strided_accepts_valid_layouts(lib):
    B, H, N, d = 2, 3, 128, 64
    bhnd, bnhd = (H * N * d, N * d, d), (N * H * d, d, H * d)
    assert _strided_fwd(lib, [bhnd] * 4) == 3
    assert _strided_fwd(lib, [bnhd] * 4) == 3
    assert _strided_fwd(lib, [bnhd, bhnd, bnhd, bhnd]) == 3
    # B = H = 1: the batch and head strides address nothing and are not checked
    assert _strided_fwd(lib, [(0, 0, 64)] * 4, B=1, H=1) == 3


def test_splitkv_heuristic(lib):
    from exact_head_attention_gb300 import exattn
    # query tiles alone fill the SMs: no split
    assert exattn.splitkv_num_splits(1, 12, 8192, 8192, 128, sm_count=152) == 1
    assert exattn.splitkv_num_splits(8, 16, 1024, 1024, 64, sm_count=152) == 1
    # one key tile: nothing to divide
    assert exattn.splitkv_num_splits(1, 1, 1, 128, 64, sm_count=152) == 1
    # decoding: 96 rows over 256 key tiles -> 3 slices (288 blocks in 2 waves of 86 tiles)
    assert exattn.splitkv_num_splits(8, 12, 1, 32768, 128, sm_count=152) == 3
    for shape in [(4, 16, 64, 16384, 64), (1, 8, 1, 524288, 128), (2, 2, 1, 1000, 128)]:
        s = exattn.splitkv_num_splits(*shape, sm_count=152)
        assert 1 < s <= 256
    assert exattn.splitkv_num_splits(0, 1, 1, 1, 64, sm_count=152) == 0

    def documented_rule(B, H, Nq, Nk, d, sms):
        """(waves over sms SMs with two resident blocks at d = 64, one at d = 128) x (tiles per block + 1),
        a split kept only when it wins by more than 2 %; 1 once the query tiles alone fill the SMs."""
        base, nkv = B * H * -(-Nq // 128), -(-Nk // 128)
        if base >= sms:
            return 1
        slots = sms * (2 if d == 64 else 1)
        best, best_cost = 1, None
        for s in range(1, min(nkv, 256) + 1):
            cost = -(-(base * s) // slots) * (-(-nkv // s) + 1)
            if s == 1 or cost < best_cost * 0.98:
                best, best_cost = s, cost
        return best

    for shape in [(4, 16, 64, 16384, 64), (8, 12, 1, 32768, 128), (2, 3, 100, 5000, 64), (1, 8, 1, 524288, 128),
                  (1, 1, 1, 65536, 64)]:
        assert exattn.splitkv_num_splits(*shape, sm_count=152) == documented_rule(*shape, 152), shape
    # the 64-query chunk over a 16k cache (d = 64): two slice blocks per SM
    assert exattn.splitkv_num_splits(4, 16, 64, 16384, 64, sm_count=152) == 9
    # workspace: fp32 O and LSE of every slice, each 256-byte aligned
    rows = 3 * 8 * 12 * 1
    assert lib.attn_fwd_splitkv_workspace_size(8, 12, 1, 32768, 128, 3) == \
        (rows * 128 * 4 + 255) // 256 * 256 + (rows * 4 + 255) // 256 * 256
    assert lib.attn_fwd_splitkv_workspace_size(8, 12, 1, 32768, 128, 257) == 0


def test_splitkv_rejects_bad_arguments(lib):
    p = [ctypes.c_void_p(FAKE)] * 5
    need = lib.attn_fwd_splitkv_workspace_size(1, 2, 1, 1000, 64, 4)
    call = lambda splits, ws=FAKE, nbytes=need, causal=0: lib.attn_fwd_splitkv(  # noqa: E731
        *p, 1, 2, 1, 1000, 64, causal, 0.125, 0, splits, ctypes.c_void_p(ws) if ws else None, nbytes, None)
    assert call(-1) == 1
    assert call(257) == 1
    assert call(4, causal=5) == 1
    assert call(4, ws=None) == 6
    assert call(4, nbytes=need - 1) == 6
    assert call(4, ws=FAKE + 16) == 3


def test_bwd_ex_rejects_unknown_dq_mode(lib):
    p = [ctypes.c_void_p(FAKE)] * 9
    need = lib.attn_bwd_workspace_size(1, 1, 128, 64)
    for mode in (-1, 3, 17):
        assert lib.attn_bwd_ex(*p, 1, 1, 128, 128, 64, 0, 0.125, 0, mode, ctypes.c_void_p(FAKE), need, None) == 1
    # a valid mode still stops at the misaligned workspace, before any launch
    assert lib.attn_bwd_ex(*p, 1, 1, 128, 128, 64, 0, 0.125, 0, 1, ctypes.c_void_p(FAKE + 16), need, None) == 3


def test_kl_rejects_bad_arguments(lib):
    p4 = [ctypes.c_void_p(FAKE)] * 4
    f3 = [ctypes.c_void_p(FAKE)] * 3
    assert lib.attn_kl_fwd(*p4, *f3, 0, 1, 128, 128, 64, 0, 0.125, 0, None) == 1
    assert lib.attn_kl_fwd(*p4, *f3, 1, 1, 128, 128, 96, 0, 0.125, 0, None) == 2
    assert lib.attn_kl_fwd(*p4, ctypes.c_void_p(FAKE + 4), *f3[1:], 1, 1, 128, 128, 64, 0, 0.125, 0, None) == 3
    assert lib.attn_kl_fwd(*p4, *f3, 1, 1, 128, 128, 64, 3, 0.125, 0, None) == 1
    g = [ctypes.c_void_p(FAKE)] * 4  # KL, LSE1, LSE2, G
    out = [ctypes.c_void_p(FAKE)] * 2
    for setting in (0, 3, -1):
        assert lib.attn_kl_bwd(*p4, *g, setting, *out, 1, 1, 128, 128, 64, 0, 0.125, 0, None) == 1
    assert lib.attn_kl_bwd(*p4, *g, 1, ctypes.c_void_p(FAKE + 2), out[1], 1, 1, 128, 128, 64, 0, 0.125, 0, None) == 3


def test_kl_bwd_ex_rejects_bad_arguments(lib):
    B, H, Nq, Nk, d = 2, 3, 200, 300, 64
    rows = B * H * 256  # Nq padded to whole 128-row tiles
    align = lambda x: (x + 255) // 256 * 256  # noqa: E731
    need = lib.attn_kl_bwd_workspace_size(B, H, Nq, d)
    assert need == align(rows * d * 4) + align(3 * rows * 4)
    assert lib.attn_kl_bwd_workspace_size(0, H, Nq, d) == 0
    assert lib.attn_kl_bwd_workspace_size(B, H, Nq, 96) == 0
    p4, g, out = [ctypes.c_void_p(FAKE)] * 4, [ctypes.c_void_p(FAKE)] * 4, [ctypes.c_void_p(FAKE)] * 2
    call = lambda mode, ws=FAKE, nbytes=need, setting=1: lib.attn_kl_bwd_ex(  # noqa: E731
        *p4, *g, setting, *out, B, H, Nq, Nk, d, 0, 0.125, 0, mode, ctypes.c_void_p(ws) if ws else None, nbytes, None)
    for mode in (-1, 3):
        assert call(mode) == 1
    assert call(0, setting=0) == 1
    for mode in (0, 2):  # the one-pass modes need the workspace
        assert call(mode, ws=None) == 6
        assert call(mode, nbytes=need - 1) == 6
        assert call(mode, ws=FAKE + 16) == 3


def test_selftest_rejects_bad_timeout(lib):
    for ms in (0, -5, 10001):
        assert lib.attn_selftest_wait_timeout(ms, None) == 1


def test_kl_splitkv_rejects_bad_arguments(lib):
    p = [ctypes.c_void_p(FAKE)] * 7
    need = lib.attn_kl_fwd_splitkv_workspace_size(1, 2, 1, 1000, 64, 4)
    assert need == ((5 * 4 * 2 * 1 * 4 + 255) // 256) * 256
    call = lambda splits, ws=FAKE, nbytes=need: lib.attn_kl_fwd_splitkv(  # noqa: E731
        *p, 1, 2, 1, 1000, 64, 0, 0.125, 0, splits, ctypes.c_void_p(ws) if ws else None, nbytes, None)
    assert call(-1) == 1
    assert call(300) == 1
    assert call(4, ws=None) == 6
    assert call(4, nbytes=need - 1) == 6
    assert call(4, ws=FAKE + 8) == 3


def _declaration_comments():
    """(function name, the comment block directly above its declaration) for every function in the header;
    declarations grouped under one comment share it."""
    text = open(os.path.join(ROOT, "include", "exattn.h")).read()
    out, last_comment, pos = [], "", 0
    for m in re.finditer(r"/\*.*?\*/|\b(attn_[a-z_0-9]+)\s*\(", text, flags=re.S):
        if m.group(0).startswith("/*"):
            last_comment = m.group(0)
        elif text[pos:m.start()].count(";") or not out or out[-1][0] != m.group(1):
            # a declaration (not a call inside a comment): the name starts a statement
            line_start = text.rfind("\n", 0, m.start()) + 1
            if re.match(r"\s*(attn_status|size_t|int|const char\*)\s", text[line_start:m.start()]):
                out.append((m.group(1), last_comment))
        pos = m.end()
    return out


def test_every_entry_point_is_documented_with_its_source():
    """Each declaration carries a comment that cites the pages (by title) or says the pages have no
    counterpart, or points to the documented entry point it varies."""
    pages = ("SparkAttention", "StreamKL", "Fast Transformer training", "CANN")
    decls = _declaration_comments()
    names = {n for n, _ in decls}
    assert {"attn_fwd", "attn_bwd", "attn_bwd_noalloc", "attn_status_string"} <= names
    for name, comment in decls:
        assert comment, f"{name}: no comment"
        comment = re.sub(r"\s*\n\s*\*?\s*", " ", comment)  # one line, without the leading stars
        cites = any(p in comment for p in pages) or "no counterpart" in comment
        refers = any(other in comment for other in names if other != name)
        assert cites or refers, f"{name}: its comment neither cites a page nor refers to a documented entry point"
