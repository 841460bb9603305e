"""attn_bwd_noalloc: the backward for callers that cannot allocate device memory.

Some callers may not allocate while they run -- a plugin inside an engine that
owns all device memory, or a latency-bound loop that cannot risk an allocator
call or its failure.  attn_bwd_noalloc serves them by taking its scratch from a
fixed array built into the library; the caller passes only inputs and outputs.

These tests call it through the C ABI and compare it with attn_bwd (the entry
point that takes a caller-supplied workspace) on two calls in a row (the array
keeps the previous call's contents, so the second call checks that whatever
must start at zero is cleared).  dK and dV are the same bits on every run of
the backward, so they must equal attn_bwd's bit for bit; dQ's fp32 reductions
run in no fixed order, so it must agree within 1e-3 relative L2 (the bound the
repeatability test of the regular backward uses), far inside the 2e-2 parity
tolerance against the oracle.  The file is named to be collected last: a run that stops at its
first failure has already run every other test.  It also passes on its own.
"""
import ctypes

import pytest

from exact_head_attention_gb300 import build, exattn, workloads

MAX_BYTES = 64 << 20  # ATTN_BWD_NOALLOC_MAX_WORKSPACE_BYTES in include/exattn.h


def _lib():
    build.build()
    lib = exattn.load()
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.attn_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
    lib.attn_bwd_noalloc.restype = i
    return lib


def test_noalloc_rejects_shapes_beyond_the_builtin_scratch():
    """Checked before the device is touched: fake pointers are never dereferenced."""
    lib = _lib()
    B, H, Nq, Nk, d = 1, 64, 8192, 8192, 128
    assert exattn.workspace_size(B, H, Nq, d) > MAX_BYTES
    fake = [ctypes.c_void_p(0x10000)] * 9
    st = lib.attn_bwd_noalloc(*fake, B, H, Nq, Nk, d, 1, 0.088, exattn.ATTN_BF16, None)
    assert st == 6  # ATTN_ERR_WORKSPACE
    assert "built-in maximum" in exattn.last_error()
    # invalid sizes are reported exactly as attn_bwd reports them
    assert lib.attn_bwd_noalloc(*fake, 0, H, Nq, Nk, d, 1, 0.088, exattn.ATTN_BF16, None) == 1


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(2, 3, 333, 271, 128, "bf16", True), (1, 4, 1000, 1200, 64, "fp16", False),
                                   (1, 12, 2048, 2048, 128, "bf16", True)])
def test_noalloc_matches_attn_bwd_on_two_calls(shape):
    import torch

    from parity import rel_l2

    lib = _lib()
    B, H, Nq, Nk, d, dt, causal = shape
    w = workloads.custom(B, H, Nq, Nk, d, dt, causal)
    assert exattn.workspace_size(B, H, Nq, d) <= MAX_BYTES
    x = workloads.make_inputs(w)
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = exattn.forward(q, k, v, causal, w.scale)
    ref = exattn.backward(q, k, v, o, do, lse, causal, w.scale)
    torch.cuda.synchronize()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    code = exattn.ATTN_BF16 if dt == "bf16" else exattn.ATTN_FP16
    for call in range(2):
        dq, dk, dv = (torch.full_like(t, float("nan")) for t in (q, k, v))
        ptrs = [ctypes.c_void_p(t.data_ptr()) for t in (q, k, v, o, do, lse, dq, dk, dv)]
        st = lib.attn_bwd_noalloc(*ptrs, B, H, Nq, Nk, d, int(causal), w.scale, code, stream)
        assert st == 0, exattn.last_error()
        torch.cuda.synchronize()
        assert exattn.check_device_error() == 0
        for name, got, want in (("dq", dq, ref[0]), ("dk", dk, ref[1]), ("dv", dv, ref[2])):
            assert torch.isfinite(got).all(), (call, name)
        assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2]), call
        err = rel_l2(dq.float().cpu().numpy(), ref[0].double().cpu().numpy())
        assert err <= 1e-3, (call, "dq", err)
