"""GPU parity of the fused linear logp path (C ABI through the binding)
against the FP64 oracle, plus the GPU-side invariants: determinism, batch
invariance, token-chunk independence of grad_hidden, zero rules."""
import numpy as np
import pytest
import torch

import oracle as O
from cross_entropy_rl_gb300 import synth
from gpu_util import TOL, TORCH, assert_pos_zero, bits_equal, check, dev

pytestmark = pytest.mark.gpu


def run(ll, p, *, token_chunks=0, dh_dtype=None, dw_dtype=None, gl=None, need=(1, 1, None)):
    dt = p["dtype"]
    h, W, b = dev(p["h"], dt), dev(p["W"], dt), dev(p["b"], dt)
    y = dev(p["y"])
    g = dev(p["gl"] if gl is None else gl)
    logp, lse = ll.forward(h, W, b, y)
    need_db = (b is not None) if need[2] is None else need[2]
    dh, dW, db = ll.backward(g, h, W, b, y, lse, need_dh=need[0], need_dw=need[1],
                             need_db=need_db, token_chunks=token_chunks,
                             dh_dtype=dh_dtype, dw_dtype=dw_dtype)
    torch.cuda.synchronize()
    assert ll.check_status() == 0
    return dict(logp=logp, lse=lse, dh=dh, dW=dW, db=db)


def compare(p, got, ref, report=None):
    """Full comparison at the plain tolerance."""
    dt = p["dtype"]
    la, lr = TOL[dt]["logp"]
    ga, gr = TOL[dt]["grad"]
    check("logp", got["logp"], ref["logp"], la, lr, report=report)
    check("lse", got["lse"], ref["lse"], la, lr, report=report)
    for k in ("dh", "dW", "db"):
        if got[k] is not None:
            check(k, got[k], ref[k], ga, gr, out_dtype=got[k].dtype, report=report)


def full_ref(p, gl=None):
    return O.linear_forward_backward(p["gl"] if gl is None else gl, p["h"], p["W"], p["b"],
                                     p["y"], p["dtype"])


# ------------------------------------------------------------ small, full --

def test_fp32_small_full_parity(lib):
    """The FP32 small problem (128 x 256 x 4096, bias), compared in full."""
    p = synth.linear_inputs(**synth.WORKLOADS["fp32_small"], seed=0)
    got = run(lib, p)
    compare(p, got, full_ref(p))


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("N,D,V,bias,chunks", [
    (300, 136, 1031, True, 0),     # ragged M, K (136 = 2*64 + 8) and vocab tiles
    (129, 64, 255, False, 0),      # one row past a tile, vocab below one tile
    (513, 264, 4099, True, 3),     # several tiles, three token chunks
    (1, 8, 1, True, 0),            # single row, single class
    (256, 512, 2304, False, 2),    # exact tiles, two chunks
])
def test_16bit_full_parity(lib, dt, N, D, V, bias, chunks):
    p = synth.linear_inputs(N, D, V, dtype=dt, bias=bias, seed=N + V)
    got = run(lib, p, token_chunks=chunks)
    compare(p, got, full_ref(p))


@pytest.mark.parametrize("N,D,V,bias", [(200, 72, 1031, True), (64, 8, 7, False)])
def test_fp32_ragged_full_parity(lib, N, D, V, bias):
    p = synth.linear_inputs(N, D, V, dtype="f32", bias=bias, seed=7)
    got = run(lib, p, token_chunks=2)
    compare(p, got, full_ref(p))


@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_16bit_grad_weight_output(lib, dt):
    """grad_weight / grad_bias in the operand dtype: FP32 accumulation, one
    rounding per token chunk; grad_hidden in FP32 on request."""
    p = synth.linear_inputs(384, 128, 1500, dtype=dt, bias=True, seed=3, grad="mean")
    got = run(lib, p, token_chunks=1, dw_dtype=TORCH[dt], dh_dtype=torch.float32)
    assert got["dW"].dtype == TORCH[dt] and got["dh"].dtype == torch.float32
    compare(p, got, full_ref(p))


def test_repeated_targets(lib):
    """Many tokens share a few targets: the one-hot part of grad_weight sums
    each target's tokens in a fixed order."""
    p = synth.linear_inputs(1000, 64, 300, dtype="bf16", bias=True, seed=11)
    p["y"] = (p["y"] % 5).astype(np.int64)
    got = run(lib, p, token_chunks=3)
    compare(p, got, full_ref(p))
    again = run(lib, p, token_chunks=3)
    assert bits_equal(got["dW"], again["dW"]) and bits_equal(got["db"], again["db"])


# ------------------------------------------------------------- invariants --

def test_bitwise_determinism(lib):
    p = synth.linear_inputs(700, 256, 5000, dtype="bf16", bias=True, seed=5)
    a, b = run(lib, p), run(lib, p)
    for k in ("logp", "lse", "dh", "dW", "db"):
        assert bits_equal(a[k], b[k]), k


def test_batch_invariance(lib):
    """logp, lse and grad_hidden of a row do not depend on the batch it is in."""
    p = synth.linear_inputs(700, 192, 3000, dtype="bf16", bias=True, seed=9)
    full = run(lib, p)
    for rows in ([0], [699], [350, 5, 1], list(range(128, 300))):
        q = dict(p)
        q["h"], q["y"], q["gl"] = p["h"][rows], p["y"][rows], p["gl"][rows]
        q["N"] = len(rows)
        part = run(lib, q)
        idx = torch.tensor(rows, device="cuda")
        for k in ("logp", "lse", "dh"):
            assert bits_equal(part[k], full[k][idx]), (k, rows[:4])


def test_token_chunks(lib):
    """grad_hidden is bitwise independent of the token chunking; grad_weight
    differs only by FP32 rounding."""
    p = synth.linear_inputs(1000, 128, 2048, dtype="bf16", bias=True, seed=13)
    ref = full_ref(p)
    outs = {k: run(lib, p, token_chunks=k) for k in (1, 2, 4, 7)}
    for k, o in outs.items():
        assert bits_equal(o["dh"], outs[1]["dh"]), k
        compare(p, o, ref)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_chunked_gradients_bitwise_whether_fused_or_alone(lib, dt):
    """Several token chunks, small enough that each gradient launch is mostly
    partial tiles: grad_hidden and grad_weight tiles launched together (one
    dynamically scheduled launch) or each alone give the same bits."""
    N, D, V = 1500, 136, 3001
    p = synth.linear_inputs(N, D, V, dtype=dt, bias=True, seed=29)
    p["y"][[3, 700]] = [-100, V]
    for chunks in (2, 3, 5):
        both = run(lib, p, token_chunks=chunks)
        dh_only = run(lib, p, token_chunks=chunks, need=(1, 0, 0))
        dw_only = run(lib, p, token_chunks=chunks, need=(0, 1, 1))
        assert bits_equal(both["dh"], dh_only["dh"]), chunks
        assert bits_equal(both["dW"], dw_only["dW"]), chunks
        assert bits_equal(both["db"], dw_only["db"]), chunks


def test_invalid_targets_and_zero_rows(lib):
    N, D, V = 260, 64, 700
    p = synth.linear_inputs(N, D, V, dtype="bf16", bias=True, seed=17)
    p["y"][[0, 5, 130, 259]] = [-100, V, V + 5, -1]
    p["gl"][[7, 140]] = [0.0, -0.0]
    got = run(lib, p, token_chunks=2)
    compare(p, got, full_ref(p))
    for r in (0, 5, 130, 259):
        assert float(got["logp"][r]) == 0.0
        assert_pos_zero(f"dh[{r}]", got["dh"][r])
    for r in (7, 140):
        assert_pos_zero(f"dh[{r}]", got["dh"][r])


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_zero_upstream_gives_positive_zeros(lib, dt):
    p = synth.linear_inputs(300, 64, 1000, dtype=dt, bias=True, seed=19)
    got = run(lib, p, gl=np.zeros(300, np.float32), token_chunks=2)
    for k in ("dh", "dW", "db"):
        assert_pos_zero(k, got[k])


def test_empty_batch(lib):
    D, V = 64, 300
    W = dev(synth.normal(0, "weight", (V, D), 0.1, "bf16"), "bf16")
    b = dev(synth.normal(0, "bias", (V,), 0.1, "bf16"), "bf16")
    h = torch.empty(0, D, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(0, dtype=torch.int64, device="cuda")
    g = torch.empty(0, dtype=torch.float32, device="cuda")
    logp, lse = lib.forward(h, W, b, y)
    assert logp.numel() == 0
    dW = torch.full((V, D), 7.0, device="cuda")
    db = torch.full((V,), 7.0, device="cuda")
    dh = torch.empty(0, D, dtype=torch.bfloat16, device="cuda")
    lib.backward(g, h, W, b, y, lse, out=(dh, dW, db), need_db=True)
    torch.cuda.synchronize()
    assert_pos_zero("dW", dW)
    assert_pos_zero("db", db)


def test_linearity_in_upstream(lib):
    """Scaling grad_logp by 2 scales every gradient by exactly 2."""
    p = synth.linear_inputs(300, 128, 1500, dtype="bf16", bias=True, seed=23)
    a = run(lib, p, dh_dtype=torch.float32)
    b = run(lib, p, gl=p["gl"] * np.float32(2.0), dh_dtype=torch.float32)
    for k in ("dh", "dW", "db"):
        assert torch.equal(b[k], 2 * a[k]), k


# --------------------------------------------------------- full-size cases --

def sampled(lib, p, rows, dw_rows=None, token_chunks=0, dw_dtype=None, report=None):
    """Compare sampled rows (logp, lse, dh) of the full run, then grad_weight /
    grad_bias of a run whose grad_logp is zero outside the sample."""
    got = run(lib, p, token_chunks=token_chunks, dw_dtype=dw_dtype, need=(1, 0, 0))
    ref = O.linear_rows(p["gl"], p["h"], p["W"], p["b"], p["y"], p["dtype"], rows,
                        dw_rows=dw_rows)
    idx = torch.tensor(rows, device="cuda")
    dt = p["dtype"]
    la, lr = TOL[dt]["logp"]
    ga, gr = TOL[dt]["grad"]
    check("logp", got["logp"][idx], ref["logp"], la, lr, report=report)
    check("lse", got["lse"][idx], ref["lse"], la, lr, report=report)
    check("dh", got["dh"][idx], ref["dh"], ga, gr, out_dtype=got["dh"].dtype, report=report)
    del got
    glm = np.zeros_like(p["gl"])
    glm[rows] = p["gl"][rows]
    got = run(lib, p, token_chunks=token_chunks, dw_dtype=dw_dtype, gl=glm, need=(0, 1, None))
    dW = got["dW"] if dw_rows is None else got["dW"][torch.tensor(dw_rows, device="cuda")]
    check("dW", dW, ref["dW"], ga, gr, out_dtype=got["dW"].dtype, report=report)
    if got["db"] is not None:
        check("db", got["db"], ref["db"], ga, gr, out_dtype=got["db"].dtype, report=report)


@pytest.mark.slow
def test_bf16_4k_2k_32k_sampled(lib):
    """The benchmark workload (4096 x 2048 x 32768, bf16, FP32 grad_weight) in
    the benchmark's launch configuration (automatic token chunks)."""
    p = synth.linear_inputs(**synth.WORKLOADS["bf16_4k_2k_32k"], seed=0)
    rows = synth.sample_rows(0, p["N"])
    sampled(lib, p, rows)


@pytest.mark.slow
@pytest.mark.parametrize("chunks", [2, 4, 8])
def test_bf16_4k_2k_32k_token_chunks(lib, chunks):
    p = synth.linear_inputs(**synth.WORKLOADS["bf16_4k_2k_32k"], seed=0)
    rows = synth.sample_rows(1, p["N"])
    sampled(lib, p, rows, token_chunks=chunks)


@pytest.mark.slow
@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("bias", [False, True])
def test_sweep_16k_4k_32000_sampled(lib, dt, bias):
    """Operands and grad_weight in one dtype, mean-loss upstream 1/N."""
    p = synth.linear_inputs(**synth.WORKLOADS["sweep_16k_4k_32000"], dtype=dt, bias=bias, seed=2)
    rows = synth.sample_rows(2, p["N"])
    sampled(lib, p, rows, dw_dtype=TORCH[dt])


@pytest.mark.slow
def test_bf16_32k_4k_151936_sampled(lib):
    """Large vocab, N*V > 2^31 (64-bit indexing), 10 % zero upstream rows."""
    p = synth.linear_inputs(**synth.WORKLOADS["bf16_32k_4k_151936"], seed=4)
    rows = synth.sample_rows(4, p["N"])
    zero = synth.zero_rows(4, p["N"], 0.1)
    assert (p["gl"][zero] == 0).all()
    dw_rows = np.unique(np.concatenate([p["y"][rows], np.arange(0, 151936, 593),
                                        [151935]])).astype(np.int64)
    sampled(lib, p, rows, dw_rows=dw_rows)


@pytest.mark.parametrize("need", [(1, 0, 0), (0, 1, 1), (0, 0, 1), (1, 1, 0)])
def test_requested_gradients_only(lib, need):
    """Each subset of (grad_hidden, grad_weight, grad_bias) matches the oracle;
    the others are not produced."""
    p = synth.linear_inputs(400, 128, 2100, dtype="bf16", bias=True, seed=29)
    got = run(lib, p, token_chunks=2, need=need)
    for k, want in zip(("dh", "dW", "db"), need):
        assert (got[k] is not None) == bool(want), k
    compare(p, got, full_ref(p))


@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("N,D,V,bias,chunks", [
    (300, 136, 1031, True, 0), (513, 264, 4099, True, 3), (1000, 128, 2048, False, 2)])
def test_single_call_forward_backward_is_bitwise_the_two_calls(lib, dt, N, D, V, bias, chunks):
    """ll_forward_backward (grad_logp known up front, no logits recompute)
    gives bitwise the outputs of ll_forward + ll_backward, and so the oracle's."""
    p = synth.linear_inputs(N, D, V, dtype=dt, bias=bias, seed=N + 7)
    two = run(lib, p, token_chunks=chunks)
    h, W, b = dev(p["h"], dt), dev(p["W"], dt), dev(p["b"], dt)
    logp, lse, dh, dW, db = lib.forward_backward(dev(p["gl"]), h, W, b, dev(p["y"]),
                                                 token_chunks=chunks)
    torch.cuda.synchronize()
    assert lib.check_status() == 0
    one = dict(logp=logp, lse=lse, dh=dh, dW=dW, db=db)
    for k in ("logp", "lse", "dh", "dW") + (("db",) if bias else ()):
        assert bits_equal(one[k], two[k]), k
    compare(p, one, full_ref(p))


@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
def test_single_call_bitwise_with_invalid_targets_zero_rows_and_temperature(lib, dt):
    """Rows with invalid targets or a zero upstream gradient, a ragged last
    32-row group, a ragged vocab tail and T != 1: the single call's softmax
    part (and its grad_bias partials) is still bitwise the recompute's."""
    N, D, V = 389, 72, 2053
    p = synth.linear_inputs(N, D, V, dtype=dt, bias=True, seed=41)
    p["y"][[0, 33, 200, 388]] = [-100, V, V + 9, -1]
    p["gl"][[5, 64, 387]] = [0.0, -0.0, 0.0]
    T = 0.8
    h, W, b, y, g = dev(p["h"], dt), dev(p["W"], dt), dev(p["b"], dt), dev(p["y"]), dev(p["gl"])
    logp2, lse2 = lib.forward(h, W, b, y, temperature=T)
    dh2, dW2, db2 = lib.backward(g, h, W, b, y, lse2, temperature=T, token_chunks=2)
    logp1, lse1, dh1, dW1, db1 = lib.forward_backward(g, h, W, b, y, temperature=T,
                                                      token_chunks=2)
    torch.cuda.synchronize()
    assert lib.check_status() == 0
    for k, a, c in (("logp", logp1, logp2), ("lse", lse1, lse2), ("dh", dh1, dh2),
                    ("dW", dW1, dW2), ("db", db1, db2)):
        assert bits_equal(a, c), k
    for r in (0, 33, 200, 388, 5, 64, 387):
        assert_pos_zero(f"dh[{r}]", dh1[r])


@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("N,V,chunks", [(1024, 1031, 0), (1500, 2053, 0), (2333, 777, 2)])
def test_single_call_larger_chunks_bitwise_the_two_calls(lib, dt, N, V, chunks):
    """Chunks of 1000+ rows with bias, invalid targets and zero upstream rows:
    the single call's outputs are bitwise the two calls'."""
    D = 136
    p = synth.linear_inputs(N, D, V, dtype=dt, bias=True, seed=N + 3)
    p["y"][[1, 700, N - 1]] = [-100, V, -1]
    p["gl"][[2, 900]] = [0.0, -0.0]
    two = run(lib, p, token_chunks=chunks)
    h, W, b = dev(p["h"], dt), dev(p["W"], dt), dev(p["b"], dt)
    logp, lse, dh, dW, db = lib.forward_backward(dev(p["gl"]), h, W, b, dev(p["y"]),
                                                 token_chunks=chunks)
    torch.cuda.synchronize()
    assert lib.check_status() == 0
    one = dict(logp=logp, lse=lse, dh=dh, dW=dW, db=db)
    for k in ("logp", "lse", "dh", "dW", "db"):
        assert bits_equal(one[k], two[k]), k


def test_single_call_split_s_temperature_and_dw_only(lib):
    """The single call with the hi / lo split of S, T != 1, and with
    grad_hidden not requested: bitwise the two calls."""
    N, D, V = 1300, 72, 1500
    p = synth.linear_inputs(N, D, V, dtype="bf16", bias=True, seed=5)
    h, W, b, y, g = (dev(p["h"], "bf16"), dev(p["W"], "bf16"), dev(p["b"], "bf16"),
                     dev(p["y"]), dev(p["gl"]))
    for need_dh in (True, False):
        logp2, lse2 = lib.forward(h, W, b, y, temperature=0.9)
        dh2, dW2, db2 = lib.backward(g, h, W, b, y, lse2, need_dh=need_dh, temperature=0.9,
                                     split_s=True)
        logp1, lse1, dh1, dW1, db1 = lib.forward_backward(g, h, W, b, y, need_dh=need_dh,
                                                          temperature=0.9, split_s=True)
        torch.cuda.synchronize()
        assert lib.check_status() == 0
        pairs = [("logp", logp1, logp2), ("lse", lse1, lse2), ("dW", dW1, dW2),
                 ("db", db1, db2)] + ([("dh", dh1, dh2)] if need_dh else [])
        for k, a, c in pairs:
            assert bits_equal(a, c), (k, need_dh)


def test_single_call_automatic_chunks_bitwise_the_two_calls(lib):
    """With token_chunks = 0 and a softmax part larger than the 2 GiB budget
    (8192 x 151936 bf16 = 2.5 GB, so two chunks), the single call picks the
    same chunks as the two calls: grad_weight too is bitwise theirs."""
    N, D, V = 8192, 64, 151936
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    h = torch.randn(N, D, generator=g, device="cuda").to(torch.bfloat16)
    W = (torch.randn(V, D, generator=g, device="cuda") * D ** -0.5).to(torch.bfloat16)
    y = torch.randint(0, V, (N,), generator=g, device="cuda")
    gl = torch.randn(N, generator=g, device="cuda")
    logp2, lse2 = lib.forward(h, W, None, y)
    dh2, dW2, _ = lib.backward(gl, h, W, None, y, lse2, token_chunks=0)
    logp1, lse1, dh1, dW1, _ = lib.forward_backward(gl, h, W, None, y, token_chunks=0)
    torch.cuda.synchronize()
    assert lib.check_status() == 0
    for k, a, c in (("logp", logp1, logp2), ("lse", lse1, lse2), ("dh", dh1, dh2),
                    ("dW", dW1, dW2)):
        assert bits_equal(a, c), k


@pytest.mark.slow
def test_single_call_bf16_4k_2k_32k_matches_two_calls(lib):
    p = synth.linear_inputs(**synth.WORKLOADS["bf16_4k_2k_32k"], seed=0)
    two = run(lib, p)
    h, W = dev(p["h"], "bf16"), dev(p["W"], "bf16")
    logp, lse, dh, dW, _ = lib.forward_backward(dev(p["gl"]), h, W, None, dev(p["y"]))
    torch.cuda.synchronize()
    for k, v in (("logp", logp), ("lse", lse), ("dh", dh), ("dW", dW)):
        assert bits_equal(v, two[k]), k


@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_gradients_into_given_16bit_buffers(lib, dt):
    """Caller-given grad buffers decide the output dtypes (grad_weight and
    grad_bias in the operand dtype here, as in the dtype sweep)."""
    p = synth.linear_inputs(640, 256, 3000, dtype=dt, bias=True, seed=37, grad="mean")
    h, W, b = dev(p["h"], dt), dev(p["W"], dt), dev(p["b"], dt)
    y, g = dev(p["y"]), dev(p["gl"])
    logp, lse = lib.forward(h, W, b, y)
    t = TORCH[dt]
    dh = torch.empty(640, 256, dtype=t, device="cuda")
    dW = torch.empty(3000, 256, dtype=t, device="cuda")
    db = torch.empty(3000, dtype=t, device="cuda")
    lib.backward(g, h, W, b, y, lse, out=(dh, dW, db))
    torch.cuda.synchronize()
    assert lib.check_status() == 0
    compare(p, dict(logp=logp, lse=lse, dh=dh, dW=dW, db=db), full_ref(p))


@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_16bit_grad_weight_several_chunks(lib, dt):
    """A 16-bit grad_weight over 3 token chunks: each later chunk reads the
    running table, adds its FP32 contribution and rounds once more."""
    p = synth.linear_inputs(700, 128, 1500, dtype=dt, bias=True, seed=43, grad="mean")
    got = run(lib, p, token_chunks=3, dw_dtype=TORCH[dt])
    ref = full_ref(p)
    # three roundings of a value of size |r|: allow three output ulps
    from gpu_util import ulp
    ga, gr = TOL[dt]["grad"]
    for k in ("dW", "db"):
        check(k, got[k], ref[k], ga, gr, extra=3 * ulp(ref[k], got[k].dtype))
    check("dh", got["dh"], ref["dh"], ga, gr, out_dtype=got["dh"].dtype)
