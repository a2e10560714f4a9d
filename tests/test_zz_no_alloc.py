"""ll_forward_noalloc: the forward for callers that cannot allocate device
memory (a framework that forbids allocation during a step, or plugin code
without access to the application's allocator).  Its scratch is a static
device array inside the library, so the caller passes only inputs and
outputs.  Called through the C ABI and checked against ll_forward (which
takes a caller workspace) on two calls in a row, plus the size limit.

This file is collected last so that a run stopping at its first failure has
already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from cross_entropy_rl_gb300 import synth
from gpu_util import TOL, check, dev

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 8 << 20


def _noalloc(L, lib, h, W, b, y, N, D, V, code):
    logp = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    st = L.ll_forward_noalloc(lib._ptr(h), lib._ptr(W), lib._ptr(b), lib._ptr(y), N, D, V, code,
                              lib._ptr(logp), lib._ptr(lse), lib._stream())
    return st, logp, lse


def test_noalloc_forward_matches_workspace_forward(lib):
    L = lib.load()
    atol, rtol = TOL["bf16"]["logp"]
    # two calls in a row on different problems: the second reuses the scratch
    # the first left behind
    for N, D, V, seed in ((1000, 256, 5000, 31), (333, 136, 1031, 32)):
        p = synth.linear_inputs(N, D, V, dtype="bf16", bias=True, seed=seed)
        h, W, b = dev(p["h"], "bf16"), dev(p["W"], "bf16"), dev(p["b"], "bf16")
        y = dev(p["y"])
        ref_logp, ref_lse = lib.forward(h, W, b, y)
        st, logp, lse = _noalloc(L, lib, h, W, b, y, N, D, V, lib.LL_BF16)
        assert st == 0, L.ll_status_string(st)
        torch.cuda.synchronize()
        assert lib.check_status() == 0
        check("logp", logp, ref_logp.double().cpu().numpy(), atol, rtol)
        check("lse", lse, ref_lse.double().cpu().numpy(), atol, rtol)


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    L = lib.load()
    D, V = 64, 151936
    W = torch.zeros(V, D, dtype=torch.bfloat16, device="cuda")
    n_segs = -(-(-(-V // 256)) // 4)
    N = SCRATCH_BYTES // ((2 * n_segs + 1) * 4) + 64  # just past the limit
    assert L.ll_workspace_size(N, D, V, lib.LL_BF16, 0, 0, 0) > SCRATCH_BYTES
    h = torch.zeros(N, D, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(N, dtype=torch.int64, device="cuda")
    st, logp, lse = _noalloc(L, lib, h, W, None, y, N, D, V, lib.LL_BF16)
    assert st == 5  # LL_ERR_WORKSPACE, nothing launched
    torch.cuda.synchronize()
    assert torch.isnan(logp).all()
