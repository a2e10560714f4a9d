"""GPU parity of the vocab-parallel (tensor-parallel) pieces, the shards run
one after another on one GPU: the shards' segment partials, stacked in
shard order (padded as the multi-rank composition pads them) and merged,
give the whole-vocab forward's logp and lse bitwise; each shard's
grad_weight / grad_bias rows are bitwise the whole-vocab backward's; the
grad_hidden parts summed in shard order match the FP64 oracle."""
import numpy as np
import pytest
import torch

import oracle as O
from cross_entropy_rl_gb300 import synth, tp
from gpu_util import TOL, assert_pos_zero, bits_equal, check, dev

pytestmark = pytest.mark.gpu


def sharded(ll, h, W, b, y, g, V, world, token_chunks=0, need_db=None):
    """The multi-rank composition of tp.forward / tp.backward, ranks in turn."""
    N = h.shape[0]
    bounds = tp.shard_bounds(V, world)
    S_max = tp.max_segments(V, world)
    pm = torch.full((world * S_max, N), -float("inf"), device="cuda")
    ps = torch.zeros((world * S_max, N), device="cuda")
    zy = torch.full((N,), -float("inf"), device="cuda")
    for r, (v0, v1) in enumerate(bounds):
        if v1 == v0:
            continue
        S = ll.shard_segments(v1 - v0)
        m, s, z = ll.forward_shard(h, W[v0:v1].contiguous(),
                                   None if b is None else b[v0:v1].contiguous(), y, v0, V)
        pm[r * S_max:r * S_max + S] = m
        ps[r * S_max:r * S_max + S] = s
        zy = torch.maximum(zy, z)
    logp, lse = ll.lse_merge(pm, ps, zy, y, V)
    dh = torch.zeros(h.shape, dtype=torch.float32, device="cuda")
    dWs, dbs = [], []
    for v0, v1 in bounds:
        if v1 == v0:
            continue
        d, dW, db = ll.backward_shard(g, h, W[v0:v1].contiguous(),
                                      None if b is None else b[v0:v1].contiguous(), y, lse,
                                      v0, V, need_db=need_db, token_chunks=token_chunks)
        dh += d
        dWs.append(dW)
        dbs.append(db)
    torch.cuda.synchronize()
    assert ll.check_status() == 0
    dW = torch.cat(dWs)
    db = torch.cat(dbs) if dbs[0] is not None else None
    return logp, lse, dh, dW, db


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("V,world", [(5000, 2), (5000, 3), (5000, 7), (3072, 3), (1024, 2)])
def test_shards_reproduce_the_whole_vocab_run(lib, dt, V, world):
    N, D = 300, 128
    p = synth.linear_inputs(N, D, V, dtype=dt, bias=True, seed=V + world)
    y = p["y"].copy()
    y[[3, 77]] = [-100, V]            # invalid targets
    gl = p["gl"].copy()
    gl[[5, 150]] = [0.0, -0.0]        # zero upstream rows
    y[10:20] = np.arange(10) * (V // 10)  # targets spread over the shards
    h, W, b = dev(p["h"], dt), dev(p["W"], dt), dev(p["b"], dt)
    yd, gd = dev(y), dev(gl)
    logp, lse = lib.forward(h, W, b, yd)
    dh1, dW1, db1 = lib.backward(gd, h, W, b, yd, lse, dh_dtype=torch.float32)
    got = sharded(lib, h, W, b, yd, gd, V, world)
    # forward: bitwise the whole-vocab run
    assert bits_equal(got[0], logp) and bits_equal(got[1], lse)
    # grad_weight / grad_bias rows: bitwise
    assert bits_equal(got[3], dW1) and bits_equal(got[4], db1)
    # grad_hidden: the shards' parts summed, against the oracle
    ref = O.linear_forward_backward(gl, p["h"], p["W"], p["b"], y, dt)
    ga, gr = TOL[dt]["grad"]
    check("dh", got[2], ref["dh"], ga, gr)
    for r in (3, 77, 5, 150):
        assert_pos_zero(f"dh[{r}]", got[2][r])


def test_shard_token_chunks_and_16bit_tables(lib):
    """token_chunks > 1 and a 16-bit grad_weight: shard rows still bitwise."""
    N, D, V = 520, 64, 4100
    p = synth.linear_inputs(N, D, V, dtype="bf16", bias=True, seed=9)
    h, W, b = dev(p["h"], "bf16"), dev(p["W"], "bf16"), dev(p["b"], "bf16")
    y, g = dev(p["y"]), dev(p["gl"])
    logp, lse = lib.forward(h, W, b, y)
    _, dW1, db1 = lib.backward(g, h, W, b, y, lse, need_dh=False, token_chunks=3,
                               dw_dtype=torch.bfloat16)
    bounds = tp.shard_bounds(V, 2)
    for v0, v1 in bounds:
        _, dW, db = lib.backward_shard(g, h, W[v0:v1].contiguous(), b[v0:v1].contiguous(), y,
                                       lse, v0, V, need_dh=False, token_chunks=3,
                                       dw_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        assert bits_equal(dW, dW1[v0:v1]) and bits_equal(db, db1[v0:v1])


def test_shard_argument_checks(lib):
    N, D, V = 8, 16, 3000
    h = torch.zeros(N, D, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(1000, D, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(N, dtype=torch.int64, device="cuda")
    with pytest.raises(lib.LLError, match="status 3"):   # v0 off a segment boundary
        lib.forward_shard(h, W, None, y, 1000, V)
    with pytest.raises(lib.LLError, match="status 3"):   # inner shard not whole segments
        lib.forward_shard(h, W, None, y, 0, V)
    with pytest.raises(lib.LLError, match="status 3"):   # past the vocab
        lib.forward_shard(h, W, None, y, 2048, V)
    W2 = torch.zeros(3000 - 2048, D, dtype=torch.bfloat16, device="cuda")
    m, s, z = lib.forward_shard(h, W2, None, y, 2048, V)  # the last shard may be ragged
    torch.cuda.synchronize()
    assert m.shape == (1, N) and bool((z == -float("inf")).all())  # every target is 0
