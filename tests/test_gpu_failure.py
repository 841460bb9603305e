"""Failure detection on the GPU without a GPU fault: a bounded device wait that nothing satisfies must
give up, report ATTN_ERR_TIMEOUT through the error word and leave the context usable."""
import time

import numpy as np
import pytest
import torch

import oracle
from exact_head_attention_gb300 import exattn, workloads

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives():
    t = time.perf_counter()
    assert exattn.selftest_wait_timeout(30) == 5  # ATTN_ERR_TIMEOUT
    assert time.perf_counter() - t >= 0.025
    assert exattn.check_device_error() == 0  # the error word was read and cleared
    # the context still works: a small attention call is correct afterwards
    w = workloads.custom(1, 2, 130, 130, 64, "bf16", True)
    x = workloads.make_inputs(w, with_grad_out=False)
    o, lse = exattn.forward(*(x[n].cuda() for n in ("q", "k", "v")), w.causal, w.scale)
    torch.cuda.synchronize()
    assert exattn.check_device_error() == 0
    ref, _ = oracle.attn_fwd(x["q"], x["k"], x["v"], w.causal, w.scale)
    assert np.abs(o.float().cpu().numpy() - ref).max() <= 1e-2


def test_repeated_timeouts():
    for _ in range(3):
        assert exattn.selftest_wait_timeout(5) == 5
    assert exattn.check_device_error() == 0
