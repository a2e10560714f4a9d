"""The forward of small problems (fewer than 128 blocks of 128 rows x 1024
vocab columns, logits within 4 MiB): its GEMM runs one vocab tile per unit
and stores the FP32 logits, and fwd_fold_kernel forms the per-segment
(max, sum-exp) partials with the epilogue's own steps.  A row's logp and lse
are the same bits whichever path its batch takes (rows of a large batch,
fused epilogue, against the same rows alone), and the small path meets the
oracle at the plain tolerance, ragged vocab tails, invalid targets inside
the last tile's padding and temperature included."""
import numpy as np
import pytest
import torch

import oracle as O
from cross_entropy_rl_gb300 import synth
from gpu_util import TOL, bits_equal, check, dev

pytestmark = pytest.mark.gpu


def small_path(lib, N, V):
    """The small path keeps N x round_up(V, 8) FP32 logits in the forward
    workspace; the one-kernel path only the partials."""
    L = lib.load()
    n_segs = -(-V // 1024)
    partials = 2 * (-(-n_segs * N * 4 // 256) * 256) + (-(-N * 4 // 256) * 256)
    ws = L.ll_workspace_size(N, 64, V, lib.LL_BF16, 0, 0, 0)
    return ws >= partials + N * (-(-V // 8) * 8) * 4


@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("T", [1.0, 0.7])
def test_rows_bitwise_across_the_two_forward_paths(lib, dt, T):
    N, D, V = 6000, 64, 3001
    p = synth.linear_inputs(N, D, V, dtype=dt, bias=True, seed=71)
    p["y"][[7, 4000]] = [-100, V + 2]  # invalid, one inside the last tile's padding
    h, W, b, y = dev(p["h"], dt), dev(p["W"], dt), dev(p["b"], dt), dev(p["y"])
    assert not small_path(lib, N, V)
    logp, lse = lib.forward(h, W, b, y, temperature=T)
    for rows in ([0], [5999], [7, 4000, 3], list(range(100, 400)), list(range(1000, 1128))):
        assert small_path(lib, len(rows), V), len(rows)
        idx = torch.tensor(rows, device="cuda")
        lp, ls = lib.forward(h[idx].contiguous(), W, b, y[idx].contiguous(), temperature=T)
        torch.cuda.synchronize()
        assert lib.check_status() == 0
        assert bits_equal(lp, logp[idx]) and bits_equal(ls, lse[idx]), (rows[:3], dt, T)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("N,V", [(128, 4096), (1, 1), (37, 33), (130, 2081), (3, 40000)])
def test_small_path_meets_the_oracle(lib, dt, N, V):
    D = 64
    assert small_path(lib, N, V)
    p = synth.linear_inputs(N, D, V, dtype=dt, bias=True, seed=N + V)
    if N > 2:
        p["y"][[0, N - 1]] = [-100, V + (1 if V % 32 else 0)]
    h, W, b, y = dev(p["h"], dt), dev(p["W"], dt), dev(p["b"], dt), dev(p["y"])
    logp, lse = lib.forward(h, W, b, y)
    torch.cuda.synchronize()
    assert lib.check_status() == 0
    ref_logp, ref_lse = O.linear_forward(p["h"], p["W"], p["b"], p["y"], dt)
    la, lr = TOL[dt]["logp"]
    check("logp", logp, ref_logp, la, lr)
    check("lse", lse, ref_lse, la, lr)
    if N > 2:
        assert float(logp[0]) == 0.0 and float(logp[N - 1]) == 0.0
    assert np.isfinite(lse.cpu().numpy()).all()


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("N", [6000, 300])
def test_single_call_fold_bitwise_the_two_calls(lib, dt, N):
    """The single fwd+bwd call folds its stored logits in a second kernel
    whenever its forward has fewer than two units per SM (here at both
    sizes), while ll_forward fuses the fold at 6000 rows: the same bits."""
    V = 3001
    p = synth.linear_inputs(N, 64, V, dtype=dt, bias=True, seed=73)
    h, W, b, y = dev(p["h"], dt), dev(p["W"], dt), dev(p["b"], dt), dev(p["y"])
    g = dev(p["gl"])
    logp, lse = lib.forward(h, W, b, y)
    two = (logp, lse) + tuple(lib.backward(g, h, W, b, y, lse))
    one = lib.forward_backward(g, h, W, b, y)
    torch.cuda.synchronize()
    assert lib.check_status() == 0
    for k, (a, c) in enumerate(zip(two, one)):
        assert bits_equal(a, c), (k, dt, N)
