"""GPU parity of temperature-scaled logp (softmax of z / T) against the FP64
oracle on the linear path, the single call, the logits path and the vocab
shards, plus exact identities: temperature 2 is bitwise the same as halving
the logits (or the weight and bias; halving is exact), with the gradients
halved as the chain rule says."""
import numpy as np
import pytest
import torch

import oracle as O
from cross_entropy_rl_gb300 import synth, tp
from gpu_util import TOL, bits_equal, check, dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("T", [0.7, 1.6])
def test_linear_temperature_parity(lib, dt, T):
    N, D, V = 200, 136, 4099
    p = synth.linear_inputs(N, D, V, dtype=dt, bias=True, seed=17)
    h, W, b = dev(p["h"], dt), dev(p["W"], dt), dev(p["b"], dt)
    y, g = dev(p["y"]), dev(p["gl"])
    logp, lse = lib.forward(h, W, b, y, temperature=T)
    dh, dW, db = lib.backward(g, h, W, b, y, lse, temperature=T)
    one = lib.forward_backward(g, h, W, b, y, temperature=T)
    torch.cuda.synchronize()
    ref = O.linear_forward_backward(p["gl"], p["h"], p["W"], p["b"], p["y"], dt, temperature=T)
    la, lr = TOL[dt]["logp"]
    ga, gr = TOL[dt]["grad"]
    check("logp", logp, ref["logp"], la, lr)
    check("lse", lse, ref["lse"], la, lr)
    for k, v in (("dh", dh), ("dW", dW), ("db", db)):
        check(k, v, ref[k], ga, gr, out_dtype=v.dtype)
    # the single call is bitwise the two calls at any temperature
    for a, c in zip(one, (logp, lse, dh, dW, db)):
        assert bits_equal(a, c)


def test_linear_temperature_two_is_halved_weights(lib):
    """z / 2 = h (W / 2)^T + b / 2 exactly: T = 2 gives the logp, lse and dh
    of the halved weights bitwise, and half their dW, db."""
    N, D, V = 256, 64, 3000
    p = synth.linear_inputs(N, D, V, dtype="bf16", bias=True, seed=23)
    h, W, b = dev(p["h"], "bf16"), dev(p["W"], "bf16"), dev(p["b"], "bf16")
    y, g = dev(p["y"]), dev(p["gl"])
    W2, b2 = W * 0.5, b * 0.5
    assert torch.equal(W2 * 2, W) and torch.equal(b2 * 2, b)  # exact halving
    a = lib.forward_backward(g, h, W, b, y, temperature=2.0)
    c = lib.forward_backward(g, h, W2, b2, y)
    torch.cuda.synchronize()
    assert bits_equal(a[0], c[0]) and bits_equal(a[1], c[1]) and bits_equal(a[2], c[2])
    assert bits_equal(a[3], c[3] * 0.5) and bits_equal(a[4], c[4] * 0.5)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_logits_temperature_parity_and_halving(lib, dt):
    N, V, T = 96, 151936 if dt == "bf16" else 5000, 0.7
    p = synth.logits_inputs(N, V, seed=29, dtype=dt)
    x, y, gl = dev(p["logits"], dt), dev(p["y"]), dev(p["gl"])
    logp, lse = lib.logits_fwd(x, y, temperature=T)
    gx = lib.logits_bwd(gl, x, y, lse, temperature=T)
    one = lib.logits_fwd_bwd(gl, x, y, temperature=T)
    torch.cuda.synchronize()
    la, lr = TOL[dt]["logp"]
    ga, gr = TOL[dt]["grad"]
    rl, rs = O.logits_forward(p["logits"], p["y"], dt, temperature=T)
    check("logp", logp, rl, la, lr)
    check("lse", lse, rs, la, lr)
    gref = O.logits_backward(p["gl"], p["logits"], p["y"], dt, temperature=T)
    check("dlogits", gx, gref, ga, gr, out_dtype=gx.dtype)
    for a, c in zip(one, (logp, lse, gx)):  # the one pass is bitwise the two calls
        assert bits_equal(a, c)
    # T = 2 is the halved logits with a halved upstream gradient, bitwise
    x2 = x * 0.5
    assert torch.equal(x2 * 2, x)
    a = lib.logits_fwd_bwd(gl, x, y, temperature=2.0)
    c = lib.logits_fwd_bwd(gl * 0.5, x2, y)
    torch.cuda.synchronize()
    for u, v in zip(a, c):
        assert bits_equal(u, v)


def test_shards_with_temperature(lib):
    """Vocab shards at T = 0.7: logp / lse bitwise the whole-vocab run."""
    N, D, V, T = 128, 64, 5000, 0.7
    p = synth.linear_inputs(N, D, V, dtype="bf16", bias=True, seed=31)
    h, W, b = dev(p["h"], "bf16"), dev(p["W"], "bf16"), dev(p["b"], "bf16")
    y, g = dev(p["y"]), dev(p["gl"])
    logp, lse = lib.forward(h, W, b, y, temperature=T)
    _, dW1, db1 = lib.backward(g, h, W, b, y, lse, need_dh=False, temperature=T)
    world = 3
    S_max = tp.max_segments(V, world)
    pm = torch.full((world * S_max, N), -float("inf"), device="cuda")
    ps = torch.zeros((world * S_max, N), device="cuda")
    zy = torch.full((N,), -float("inf"), device="cuda")
    dWs, dbs = [], []
    for r, (v0, v1) in enumerate(tp.shard_bounds(V, world)):
        S = lib.shard_segments(v1 - v0)
        m, s, z = lib.forward_shard(h, W[v0:v1].contiguous(), b[v0:v1].contiguous(), y, v0, V,
                                    temperature=T)
        pm[r * S_max:r * S_max + S] = m
        ps[r * S_max:r * S_max + S] = s
        zy = torch.maximum(zy, z)
    l2, s2 = lib.lse_merge(pm, ps, zy, y, V)
    for v0, v1 in tp.shard_bounds(V, world):
        _, dW, db = lib.backward_shard(g, h, W[v0:v1].contiguous(), b[v0:v1].contiguous(), y,
                                       s2, v0, V, need_dh=False, temperature=T)
        dWs.append(dW)
        dbs.append(db)
    torch.cuda.synchronize()
    assert bits_equal(l2, logp) and bits_equal(s2, lse)
    assert bits_equal(torch.cat(dWs), dW1) and bits_equal(torch.cat(dbs), db1)
