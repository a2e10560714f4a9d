"""GPU parity of the hi / lo split of the softmax part S (ll_options.split_s)
on a peaked distribution (weights scaled by 8, so off-target probabilities
are large): the split path meets the plain gradient tolerance against the
FP64 oracle, where storing S in one 16-bit part costs ~2^-9 of |grad_logp|
at the large entries; the single call stays bitwise the two calls; the
vocab shards stay bitwise the whole-vocab rows; FP32 operands ignore it."""
import numpy as np
import pytest
import torch

import oracle as O
from cross_entropy_rl_gb300 import synth, tp
from gpu_util import TOL, bits_equal, check, dev, host64

pytestmark = pytest.mark.gpu


def peaked(dt, N=256, D=128, V=4099, seed=37, scale=8.0):
    p = synth.linear_inputs(N, D, V, dtype=dt, bias=True, seed=seed)
    W = O.decode(p["W"], dt) * scale  # a power of two: exact in every dtype
    if dt == "bf16":
        p["W"] = synth.f32_to_bf16_bits(W.astype(np.float32))
    else:
        p["W"] = W.astype(np.float16 if dt == "f16" else np.float32)
    assert np.array_equal(O.decode(p["W"], dt), W)
    return p


def run(lib, p, split, single=False):
    """Forward + backward (or the single call); grad_hidden in FP32 so that
    its own output rounding does not hide the S storage error."""
    dt = p["dtype"]
    h, W, b = dev(p["h"], dt), dev(p["W"], dt), dev(p["b"], dt)
    y, g = dev(p["y"]), dev(p["gl"])
    if single:
        out = lib.forward_backward(g, h, W, b, y, split_s=split, dh_dtype=torch.float32)
    else:
        logp, lse = lib.forward(h, W, b, y)
        out = (logp, lse) + lib.backward(g, h, W, b, y, lse, split_s=split,
                                         dh_dtype=torch.float32)
    torch.cuda.synchronize()
    assert lib.check_status() == 0
    return dict(zip(("logp", "lse", "dh", "dW", "db"), out))


@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_split_meets_the_tolerance_on_a_peaked_distribution(lib, dt):
    p = peaked(dt)
    ref = O.linear_forward_backward(p["gl"], p["h"], p["W"], p["b"], p["y"], dt)
    pmax = np.exp(O.linear_logits(O.decode(p["h"], dt), O.decode(p["W"], dt),
                                  O.decode(p["b"], dt)).max(axis=1) - ref["lse"])
    assert np.median(pmax) > 0.5  # peaked indeed
    got = run(lib, p, split=True)
    ga, gr = TOL[dt]["grad"]
    errs = {}
    for k in ("dh", "dW", "db"):
        errs[k] = check(k, got[k], ref[k], ga, gr, out_dtype=got[k].dtype)
    plain = run(lib, p, split=False)
    for k in ("dh", "dW"):
        e_plain = np.abs(host64(plain[k]) - ref[k]).max()
        e_split = np.abs(host64(got[k]) - ref[k]).max()
        assert e_split * 4 < e_plain, (k, e_split, e_plain)
    # the forward is untouched by the option
    assert bits_equal(got["logp"], plain["logp"]) and bits_equal(got["lse"], plain["lse"])


def test_split_single_call_is_bitwise_the_two_calls(lib):
    p = peaked("bf16", N=300, V=5000, seed=41)
    a = run(lib, p, split=True)
    c = run(lib, p, split=True, single=True)
    for k in a:
        assert bits_equal(a[k], c[k]), k


def test_split_vocab_shards_bitwise(lib):
    p = peaked("bf16", N=200, V=5000, seed=43)
    h, W, b = dev(p["h"], "bf16"), dev(p["W"], "bf16"), dev(p["b"], "bf16")
    y, g = dev(p["y"]), dev(p["gl"])
    logp, lse = lib.forward(h, W, b, y)
    _, dW1, db1 = lib.backward(g, h, W, b, y, lse, need_dh=False, split_s=True)
    for v0, v1 in tp.shard_bounds(5000, 3):
        _, dW, db = lib.backward_shard(g, h, W[v0:v1].contiguous(), b[v0:v1].contiguous(), y,
                                       lse, v0, 5000, need_dh=False, split_s=True)
        torch.cuda.synchronize()
        assert bits_equal(dW, dW1[v0:v1]) and bits_equal(db, db1[v0:v1])


def test_split_is_ignored_for_fp32(lib):
    p = peaked("f32", N=128, V=2000, seed=47)
    a = run(lib, p, split=True)
    c = run(lib, p, split=False)
    for k in a:
        assert bits_equal(a[k], c[k]), k
