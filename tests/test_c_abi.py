"""The C ABI used from C: include/exattn.h compiles as C99 and as C++, and a
plain C program (tests/c_abi/consumer.c) links libexattn.so and calls it.

CPU: the header compiles under strict warnings in both languages; the C
program's argument checks and host-side helpers (workspace size, status
strings, the dQ-mode and launch-group rules, the forward's packed lists) give
the documented results, with fake device pointers that are never
dereferenced.

GPU: the same program, built against the CUDA runtime for device memory, runs
attn_fwd and attn_bwd on a small ragged causal problem written by this test
from the seeded generator; its outputs are compared with the fp64 oracle at
the parity tolerances.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
SRC = os.path.join(ROOT, "tests", "c_abi", "consumer.c")
STRICT = ["-Wall", "-Wextra", "-Werror"]


def _lib_dir():
    from exact_head_attention_gb300 import build
    return os.path.dirname(build.build())


def _cuda_home():
    nvcc = shutil.which("nvcc")
    return os.path.dirname(os.path.dirname(nvcc)) if nvcc else "/usr/local/cuda"


def _compile(out, cflags, ldflags=()):
    """Compile and link the C program; libraries follow the source (the linker drops those named before)."""
    lib_dir = _lib_dir()
    cmd = ["gcc", "-std=c99", *STRICT, f"-I{INCLUDE}", *cflags, SRC, "-o", out,
           f"-L{lib_dir}", "-lexattn", f"-Wl,-rpath,{lib_dir}", *ldflags]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr


def test_header_compiles_as_c_and_cpp(tmp_path):
    src = tmp_path / "h.c"
    src.write_text('#include "exattn.h"\nint main(void) { return attn_bwd_workspace_size(1, 1, 1, 64) == 0; }\n')
    for cmd in (["gcc", "-std=c99", "-pedantic", *STRICT], ["gcc", "-std=c11", "-pedantic", *STRICT],
                ["g++", "-std=c++11", "-pedantic", *STRICT, "-x", "c++"]):
        r = subprocess.run([*cmd, f"-I{INCLUDE}", "-fsyntax-only", str(src)], capture_output=True, text=True)
        assert r.returncode == 0, (cmd, r.stderr)


def test_c_program_calls_the_library(tmp_path):
    exe = str(tmp_path / "consumer")
    _compile(exe, ["-pedantic"])
    r = subprocess.run([exe, "cpu"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(1, 2, 300, 300, 64, "bf16", True), (2, 1, 200, 333, 128, "fp16", False)])
def test_c_program_forward_backward_matches_oracle(tmp_path, shape):
    import torch

    import oracle
    from exact_head_attention_gb300 import workloads
    from parity import check_fwd, check_grads

    B, H, Nq, Nk, d, dt, causal = shape
    w = workloads.custom(B, H, Nq, Nk, d, dt, causal, index=40)
    x = workloads.make_inputs(w)
    cuda = _cuda_home()
    exe = str(tmp_path / "consumer_gpu")
    _compile(exe, ["-DWITH_CUDART", f"-I{cuda}/include"], [f"-L{cuda}/lib64", "-lcudart", f"-Wl,-rpath,{cuda}/lib64"])

    inp, out = tmp_path / "in.bin", tmp_path / "out.bin"
    hdr = np.array([B, H, Nq, Nk, d, 1 if causal else 0, 0 if dt == "bf16" else 1], dtype=np.int32)
    with open(inp, "wb") as f:
        f.write(hdr.tobytes())
        f.write(np.array([w.scale], dtype=np.float32).tobytes())
        for n in ("q", "k", "v", "do"):
            f.write(x[n].contiguous().view(torch.int16).numpy().tobytes())
    r = subprocess.run([exe, "gpu", str(inp), str(out)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr

    raw = out.read_bytes()
    tdt = torch.bfloat16 if dt == "bf16" else torch.float16
    sizes = [("o", B * H * Nq * d, 2), ("lse", B * H * Nq, 4), ("dq", B * H * Nq * d, 2), ("dk", B * H * Nk * d, 2),
             ("dv", B * H * Nk * d, 2)]
    got, pos = {}, 0
    for name, n, es in sizes:
        chunk = raw[pos:pos + n * es]
        pos += n * es
        if es == 4:
            got[name] = np.frombuffer(chunk, dtype=np.float32).reshape(B, H, Nq)
        else:
            a = torch.frombuffer(bytearray(chunk), dtype=torch.int16).view(tdt).float().numpy()
            got[name] = a.reshape(B, H, Nq if name in ("o", "dq") else Nk, d)
    assert pos == len(raw)

    o, lse = oracle.attn_fwd(x["q"], x["k"], x["v"], causal, w.scale)
    check_fwd(w, got["o"], got["lse"], o, lse, "C program")
    dq, dk, dv, _ = oracle.attn_bwd(x["q"], x["k"], x["v"], x["do"], causal, w.scale)
    check_grads(got, {"dq": dq, "dk": dk, "dv": dv}, "C program")
