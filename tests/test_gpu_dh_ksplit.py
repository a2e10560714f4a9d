"""The FP32 gradient launch.  First, grad_hidden over a narrow hidden size
(D <= 512): the K = V
contraction is cut into parts of at least 16 K blocks (up to 16 parts), each
its own unit of the gradient launch, and a finishing pass adds the parts'
FP32 partial sums in ascending part order before the target column and the
zero rules.  The part count depends on (D, V) alone: a row's grad_hidden is
bitwise independent of the batch it is in, of the token chunks and of the
grad_weight tiles launched beside it, and it meets the FP32 tolerance against
the FP64 oracle (including vocab sizes that leave a short last part).
Second, the K-major operand copies of large problems give the bits of the
MN-major operands."""
import numpy as np
import pytest
import torch

import oracle as O
from cross_entropy_rl_gb300 import synth
from gpu_util import TOL, assert_pos_zero, bits_equal, check, dev

pytestmark = pytest.mark.gpu


def run(lib, p, token_chunks=0, need=(1, 1, None)):
    h, W, b = dev(p["h"], "f32"), dev(p["W"], "f32"), dev(p["b"], "f32")
    y, g = dev(p["y"]), dev(p["gl"])
    logp, lse = lib.forward(h, W, b, y)
    need_db = (b is not None) if need[2] is None else need[2]
    dh, dW, db = lib.backward(g, h, W, b, y, lse, need_dh=need[0], need_dw=need[1],
                              need_db=need_db, token_chunks=token_chunks)
    torch.cuda.synchronize()
    assert lib.check_status() == 0
    return dict(logp=logp, lse=lse, dh=dh, dW=dW, db=db)


@pytest.mark.parametrize("N,D,V", [(128, 256, 4096), (300, 64, 512), (257, 136, 513),
                                   (129, 512, 7001), (40, 8, 100000)])
def test_k_split_meets_the_fp32_tolerance(lib, N, D, V):
    p = synth.linear_inputs(N, D, V, dtype="f32", bias=True, seed=N + V)
    p["y"][[1, N // 2]] = [-100, V]  # dead rows: exact +0
    got = run(lib, p)
    ref = O.linear_forward_backward(p["gl"], p["h"], p["W"], p["b"], p["y"], "f32")
    ga, gr = TOL["f32"]["grad"]
    for k in ("dh", "dW", "db"):
        check(k, got[k], ref[k], ga, gr, out_dtype=got[k].dtype)
    for r in (1, N // 2):
        assert_pos_zero(f"dh[{r}]", got["dh"][r])


def test_k_split_rows_independent_of_the_batch(lib):
    p = synth.linear_inputs(700, 192, 3000, dtype="f32", bias=True, seed=9)
    p["gl"][[3, 400]] = 0.0
    full = run(lib, p)
    for rows in ([0], [699], [350, 5, 1], list(range(128, 300)), [3, 400, 2]):
        q = dict(p, h=p["h"][rows], y=p["y"][rows], gl=p["gl"][rows], N=len(rows))
        part = run(lib, q)
        idx = torch.tensor(rows, device="cuda")
        assert bits_equal(part["dh"], full["dh"][idx]), rows[:4]
    for r in (3, 400):
        assert_pos_zero(f"dh[{r}]", full["dh"][r])


def test_k_split_bitwise_across_chunks_and_launch_mixes(lib):
    p = synth.linear_inputs(1100, 256, 4096, dtype="f32", bias=False, seed=23)
    one = run(lib, p, token_chunks=1)
    for chunks in (2, 3, 9):
        got = run(lib, p, token_chunks=chunks)
        assert bits_equal(got["dh"], one["dh"]), chunks
    alone = run(lib, p, token_chunks=3, need=(1, 0, 0))
    assert bits_equal(alone["dh"], one["dh"])
    again = run(lib, p, token_chunks=1)
    for k in ("dh", "dW"):
        assert bits_equal(again[k], one[k]), k


def test_wide_hidden_keeps_one_part(lib):
    """D > 512 takes the whole-K units (no parts, no finishing pass): the
    same rows meet the same tolerance."""
    p = synth.linear_inputs(130, 520, 3000, dtype="f32", bias=True, seed=31)
    got = run(lib, p)
    ref = O.linear_forward_backward(p["gl"], p["h"], p["W"], p["b"], p["y"], "f32")
    ga, gr = TOL["f32"]["grad"]
    check("dh", got["dh"], ref["dh"], ga, gr, out_dtype=got["dh"].dtype)
    assert np.isfinite(ref["dh"]).all()


def test_kmajor_gradient_operands_bitwise_the_mn_major_ones(lib):
    """From 2^32 multiply-adds (N * D * V) on, the FP32 backward passes its
    gradient launch K-major copies (W^T, S^T, h^T) instead of W, S and h, so
    the converters need not transpose.  The products and their order are the
    same: rows of a 1024-row batch (copies) equal the same rows of a 1023-row
    batch (no copies) bitwise, grad_hidden included."""
    D, V = 1024, 4096
    L = lib.load()
    ws_t = L.ll_workspace_size(1024, D, V, lib.LL_F32, 0, 1, 0)
    ws_m = L.ll_workspace_size(1023, D, V, lib.LL_F32, 0, 1, 0)
    assert ws_t - ws_m >= D * V * 4  # W^T (and S^T, h^T) only for the larger batch
    p = synth.linear_inputs(1024, D, V, dtype="f32", bias=True, seed=83)
    big = run(lib, p)
    q = dict(p, h=p["h"][:1023], y=p["y"][:1023], gl=p["gl"][:1023], N=1023)
    small = run(lib, q)
    for k in ("logp", "lse", "dh"):
        assert bits_equal(small[k], big[k][:1023]), k
    ref = O.linear_forward_backward(p["gl"], p["h"], p["W"], p["b"], p["y"], "f32")
    ga, gr = TOL["f32"]["grad"]
    for k in ("dh", "dW", "db"):
        check(k, big[k], ref[k], ga, gr, out_dtype=big[k].dtype)


def test_kmajor_gradient_operands_ragged_shapes(lib):
    """K-major copies with ragged sizes (rows, hidden and vocab not multiples
    of the 32 x 32 transpose tile, vocab not a multiple of 4, two token
    chunks): every gradient meets the FP32 tolerance against the oracle."""
    N, D, V = 1031, 1032, 4099
    assert N * D * V >= 2 ** 32
    p = synth.linear_inputs(N, D, V, dtype="f32", bias=True, seed=89)
    p["y"][[4, 1030]] = [-100, V]
    got = run(lib, p, token_chunks=2)
    ref = O.linear_forward_backward(p["gl"], p["h"], p["W"], p["b"], p["y"], "f32")
    ga, gr = TOL["f32"]["grad"]
    for k in ("dh", "dW", "db"):
        check(k, got[k], ref[k], ga, gr, out_dtype=got[k].dtype)
    for r in (4, 1030):
        assert_pos_zero(f"dh[{r}]", got["dh"][r])
