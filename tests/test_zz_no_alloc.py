"""ll_forward_noalloc: the forward for callers that cannot allocate device
memory (a framework that forbids allocation during a step, or plugin code
without access to the application's allocator).  Its scratch is a static
device array inside the library, so the caller passes only inputs and
outputs.

Called through the C ABI.  It runs the same kernels on the same scratch
layout as ll_forward with a caller workspace, so its logp and lse must be
the same bits; they are also checked against the FP64 oracle.  The calls
come in an order that would expose stale scratch: a small problem, then one
that needs more scratch, then the same shape with other data.  The size
limit is checked at its exact boundary.

This file is collected last so that a run stopping at its first failure has
already run every other test."""
import pytest
import torch

import oracle
from cross_entropy_rl_gb300 import synth
from gpu_util import TOL, bits_equal, check, dev

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 8 << 20
LL_ERR_WORKSPACE = 5


def _noalloc(L, lib, h, W, b, y, N, D, V, code):
    logp = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    st = L.ll_forward_noalloc(lib._ptr(h), lib._ptr(W), lib._ptr(b), lib._ptr(y), N, D, V, code,
                              lib._ptr(logp), lib._ptr(lse), lib._stream())
    return st, logp, lse


def test_noalloc_forward_matches_workspace_forward(lib):
    L = lib.load()
    atol, rtol = TOL["bf16"]["logp"]
    # a small problem, one needing more scratch (reads past what the first
    # call wrote would show), then the same shape with other data
    for N, D, V, seed in ((333, 136, 1031, 32), (1000, 256, 5000, 31), (1000, 256, 5000, 33)):
        p = synth.linear_inputs(N, D, V, dtype="bf16", bias=True, seed=seed)
        h, W, b = dev(p["h"], "bf16"), dev(p["W"], "bf16"), dev(p["b"], "bf16")
        y = dev(p["y"])
        ref_logp, ref_lse = lib.forward(h, W, b, y)
        st, logp, lse = _noalloc(L, lib, h, W, b, y, N, D, V, lib.LL_BF16)
        assert st == 0, L.ll_status_string(st)
        torch.cuda.synchronize()
        assert lib.check_status() == 0
        assert bits_equal(logp, ref_logp), (N, V, seed)
        assert bits_equal(lse, ref_lse), (N, V, seed)
        o_logp, o_lse = oracle.linear_forward(p["h"], p["W"], p["b"], p["y"], "bf16")
        check("logp", logp, o_logp, atol, rtol)
        check("lse", lse, o_lse, atol, rtol)


def test_noalloc_size_limit_boundary(lib):
    """At V = 151936 the scratch holds N = 7013 rows: that call runs and
    matches ll_forward bitwise, N = 7014 is rejected before anything runs."""
    L = lib.load()
    D, V = 64, 151936
    assert L.ll_workspace_size(7013, D, V, lib.LL_BF16, 0, 0, 0) <= SCRATCH_BYTES
    assert L.ll_workspace_size(7014, D, V, lib.LL_BF16, 0, 0, 0) > SCRATCH_BYTES
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    W = (torch.randn(V, D, generator=g, device="cuda") * D ** -0.5).to(torch.bfloat16)
    for N, ok in ((7013, True), (7014, False)):
        h = torch.randn(N, D, generator=g, device="cuda").to(torch.bfloat16)
        y = torch.randint(0, V, (N,), generator=g, device="cuda")
        st, logp, lse = _noalloc(L, lib, h, W, None, y, N, D, V, lib.LL_BF16)
        torch.cuda.synchronize()
        if ok:
            assert st == 0, L.ll_status_string(st)
            assert lib.check_status() == 0
            ref_logp, ref_lse = lib.forward(h, W, None, y)
            assert bits_equal(logp, ref_logp) and bits_equal(lse, ref_lse)
        else:
            assert st == LL_ERR_WORKSPACE
            assert torch.isnan(logp).all() and torch.isnan(lse).all()


def test_noalloc_empty_batch_like_ll_forward(lib):
    """N = 0 returns LL_OK without touching any pointer, as ll_forward does."""
    L = lib.load()
    W = torch.zeros(256, 64, dtype=torch.bfloat16, device="cuda")
    st = L.ll_forward_noalloc(None, lib._ptr(W), None, None, 0, 64, 256, lib.LL_BF16, None,
                              None, lib._stream())
    assert st == 0
