"""GPU parity of the logits-input logp forward/backward against the FP64
oracle; batch-size / row-position invariance sweep (bitwise); masked tails,
invalid targets, unaligned row strides."""
import numpy as np
import pytest
import torch

import oracle as O
from cross_entropy_rl_gb300 import synth
from gpu_util import TOL, accuracy, assert_pos_zero, bits_equal, check, dev

pytestmark = pytest.mark.gpu


def run(ll, x, y, gl, V=None):
    logp, lse = ll.logits_fwd(x, y, V)
    g = ll.logits_bwd(gl, x, y, lse, V)
    torch.cuda.synchronize()
    return logp, lse, g


def compare(p, got, rows=None, V=None):
    dt = p["dtype"]
    x = p["logits"] if rows is None else p["logits"][rows]
    y = p["y"] if rows is None else p["y"][rows]
    gl = p["gl"] if rows is None else p["gl"][rows]
    Vv = p["V"] if V is None else V
    lr_logp, lr_lse = O.logits_forward(x, y, dt, V=Vv)
    g_ref = O.logits_backward(gl, x, y, dt, V=Vv)
    logp, lse, g = got
    if rows is not None:
        idx = torch.tensor(rows, device="cuda")
        logp, lse, g = logp[idx], lse[idx], g[idx]
    la, lr = TOL[dt]["logp"]
    ga, gr = TOL[dt]["grad"]
    check("logp", logp, lr_logp, la, lr)
    check("lse", lse, lr_lse, la, lr)
    check("dlogits", g[:, :Vv], g_ref, ga, gr, out_dtype=g.dtype)


@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("V", [1, 255, 1031, 151936])
def test_full_parity(lib, dt, V):
    N = 64 if V > 10000 else 200
    p = synth.logits_inputs(N, V, seed=V, dtype=dt)
    x, y, gl = dev(p["logits"], dt), dev(p["y"]), dev(p["gl"])
    compare(p, run(lib, x, y, gl))


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_padded_and_unaligned_rows(lib, dt):
    """Row stride ld > V: aligned (vector path) and not 16-byte aligned."""
    for ld in (1040, 1033):
        p = synth.logits_inputs(96, 1031, seed=ld, dtype=dt, ld=ld)
        x, y, gl = dev(p["logits"], dt), dev(p["y"]), dev(p["gl"])
        got = run(lib, x, y, gl, V=1031)
        compare(p, got, V=1031)
        # columns [V, ld) of the gradient are not written
        out = torch.full_like(x, 3.0)
        lib.logits_bwd(gl, x, y, got[1], V=1031, out=out)
        torch.cuda.synchronize()
        assert bool((out[:, 1031:] == 3.0).all())


def test_invalid_targets_masked_tail(lib):
    """-inf tail (targets kept below it), invalid targets -100 / V / V+5,
    an all -inf row with an invalid target, zero upstream rows."""
    N, V = 40, 4096
    p = synth.logits_inputs(N, V, seed=3)
    x = dev(p["logits"], "bf16")
    x[:, 3000:] = -float("inf")
    x[11, :] = -float("inf")
    y = p["y"] % 1000
    y[[2, 9, 11, 30]] = [-100, V, -100, V + 5]
    gl = p["gl"].copy()
    gl[[4, 20]] = [0.0, -0.0]
    q = dict(p, y=y, gl=gl, logits=x.view(torch.int16).cpu().numpy().view(np.uint16))
    got = run(lib, x, dev(y), dev(gl))
    compare(q, got)
    logp, lse, g = got
    assert torch.isfinite(g.float()).all()
    for r in (2, 9, 11, 30, 4, 20):
        assert_pos_zero(f"g[{r}]", g[r])
    assert float(logp[11]) == 0.0 and float(lse[11]) == -float("inf")
    assert_pos_zero("tail", g[:, 3000:])


def test_empty(lib):
    x = torch.empty(0, 100, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(0, dtype=torch.int64, device="cuda")
    logp, lse = lib.logits_fwd(x, y)
    assert logp.numel() == 0


def _sweep_sizes(full):
    s = list(range(1, 10))
    k = 2
    while 2 ** k <= 2048:
        s += [2 ** k - 1, 2 ** k, 2 ** k + 1]
        k += 1
    s = sorted(set(s)) + [4096]
    if full:
        s += [32768]
    return s


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_batch_invariance_sweep(lib, seed):
    """Eight probe rows alone vs at the front, middle and back of batches of
    sizes 1-9, 2^k-1 / 2^k / 2^k+1 up to 2048, and 4096: logp, lse and
    dlogits bitwise identical (32768 in the full-size test)."""
    V = 151936
    probes = synth.logits_inputs(8, V, seed=100 + seed)
    px, py, pg = dev(probes["logits"], "bf16"), dev(probes["y"]), dev(probes["gl"])
    alone = [run(lib, px[i:i + 1], py[i:i + 1], pg[i:i + 1]) for i in range(8)]
    filler = synth.logits_inputs(4096 + 8, V, seed=200 + seed)
    fx, fy, fg = dev(filler["logits"], "bf16"), dev(filler["y"]), dev(filler["gl"])
    differ = 0
    total = 0
    for n in _sweep_sizes(False):
        for where in ("front", "middle", "back"):
            m = min(8, n)
            x, y, g = fx[:n].clone(), fy[:n].clone(), fg[:n].clone()
            pos = {"front": 0, "middle": (n - m) // 2, "back": n - m}[where]
            x[pos:pos + m], y[pos:pos + m], g[pos:pos + m] = px[:m], py[:m], pg[:m]
            logp, lse, dl = run(lib, x, y, g)
            for i in range(m):
                total += 1
                a = alone[i]
                same = (bits_equal(logp[pos + i:pos + i + 1], a[0]) and
                        bits_equal(lse[pos + i:pos + i + 1], a[1]) and
                        bits_equal(dl[pos + i:pos + i + 1], a[2]))
                differ += 0 if same else 1
    assert differ == 0, f"{differ} of {total} probe rows differ"


@pytest.mark.slow
def test_logits_32k_151936_sampled(lib):
    """The full logits workload (32768 x 151936 bf16; N*V > 2^31) on 256
    sampled rows, plus rows 0, N/2, N-1."""
    p = synth.logits_inputs(**synth.WORKLOADS["logits_32k_151936"], seed=0)
    x, y, gl = dev(p["logits"], "bf16"), dev(p["y"]), dev(p["gl"])
    got = run(lib, x, y, gl)
    rows = synth.sample_rows(0, p["N"])
    compare(p, got, rows=rows)
    # the probe rows of the sweep are position independent at full size too
    alone = run(lib, x[-1:], y[-1:], gl[-1:])
    assert bits_equal(alone[2], got[2][-1:]) and bits_equal(alone[1], got[1][-1:])


# ------------------------------------------------ one pass (known upstream) --

def run_fused(ll, x, y, gl, V=None):
    logp, lse, g = ll.logits_fwd_bwd(gl, x, y, V)
    torch.cuda.synchronize()
    assert ll.check_status() == 0
    return logp, lse, g


@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("V,ld", [(151936, 151936), (1024, 1024), (4096, 4104),
                                  (1031, 1031), (1031, 1040), (8, 8)])
def test_fused_full_parity(lib, dt, V, ld):
    """One-pass fwd+bwd vs the oracle (vector rows, V % 8 != 0, unaligned
    rows), and bitwise the two calls."""
    N = 48 if V > 10000 else 150
    p = synth.logits_inputs(N, V, seed=V + ld, dtype=dt, ld=ld)
    x, y, gl = dev(p["logits"], dt), dev(p["y"]), dev(p["gl"])
    got = run_fused(lib, x, y, gl, V=V)
    compare(p, got, V=V)
    two = run(lib, x, y, gl, V=V)
    for a, b in zip(got, two):
        assert bits_equal(a[:, :V] if a.dim() == 2 else a, b[:, :V] if b.dim() == 2 else b)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_fused_in_place(lib, dt):
    """grad_logits written over the logits buffer: the same bits as out of
    place; a partially overlapping output is refused."""
    N, V = 300, 151936 if dt == "bf16" else 4104
    p = synth.logits_inputs(N, V, seed=13, dtype=dt)
    x, y, gl = dev(p["logits"], dt), dev(p["y"]), dev(p["gl"])
    ref = run_fused(lib, x, y, gl)
    xi = x.clone()
    got = lib.logits_fwd_bwd(gl, xi, y, out=(torch.empty(N, device="cuda"),
                                             torch.empty(N, device="cuda"), xi))
    torch.cuda.synchronize()
    for a, b in zip(got, ref):
        assert bits_equal(a, b)
    assert got[2].data_ptr() == xi.data_ptr()
    big = torch.empty(N + 1, V, dtype=x.dtype, device="cuda")
    big[:N] = x
    with pytest.raises(lib.LLError, match="status 1"):
        lib.logits_fwd_bwd(gl, big[:N], y, out=(torch.empty(N, device="cuda"),
                                                torch.empty(N, device="cuda"), big[1:]))


def test_fused_invalid_targets_and_zero_rows(lib):
    N, V = 40, 4096
    p = synth.logits_inputs(N, V, seed=5)
    x = dev(p["logits"], "bf16")
    x[:, 3000:] = -float("inf")
    x[11, :] = -float("inf")
    y = p["y"] % 1000
    y[[2, 9, 11, 30]] = [-100, V, -100, V + 5]
    gl = p["gl"].copy()
    gl[[4, 20]] = [0.0, -0.0]
    q = dict(p, y=y, gl=gl, logits=x.view(torch.int16).cpu().numpy().view(np.uint16))
    got = run_fused(lib, x, dev(y), dev(gl))
    compare(q, got)
    logp, lse, g = got
    for r in (2, 9, 11, 30, 4, 20):
        assert_pos_zero(f"g[{r}]", g[r])
    assert float(logp[11]) == 0.0 and float(lse[11]) == -float("inf")


def test_fused_batch_invariance_and_determinism(lib):
    V = 151936
    p = synth.logits_inputs(300, V, seed=41)
    x, y, gl = dev(p["logits"], "bf16"), dev(p["y"]), dev(p["gl"])
    full = run_fused(lib, x, y, gl)
    again = run_fused(lib, x, y, gl)
    for a, b in zip(full, again):
        assert bits_equal(a, b)
    for rows in ([0], [299], [7, 150, 3], list(range(100, 257))):
        idx = torch.tensor(rows, device="cuda")
        part = run_fused(lib, x[idx].contiguous(), y[idx], gl[idx])
        for a, b in zip(part, full):
            assert bits_equal(a, b[idx])


@pytest.mark.slow
def test_fused_logits_32k_151936_sampled(lib):
    p = synth.logits_inputs(**synth.WORKLOADS["logits_32k_151936"], seed=0)
    x, y, gl = dev(p["logits"], "bf16"), dev(p["y"]), dev(p["gl"])
    got = run_fused(lib, x, y, gl)
    compare(p, got, rows=synth.sample_rows(0, p["N"]))


def test_accuracy_257x151936_against_fp64(lib):
    """Accuracy of the logits-input backward on the shape of PR #495's
    accuracy comparison ("Summary", the B200 table, and the author's rerun in
    the PR discussion): 257 rows x 151936, bf16 logits, the upstream gradient
    rounded to bf16 once and fed to both sides as the same FP32 values.
    Reported: max abs error, max error / max |ref|, and the share of gradient
    entries equal to the bf16 rounding of the FP64 value.  That PR lists
    99.9986% correctly rounded for its fused kernel, 99.99% for flash-attn's and
    74.3% for an unfused bf16 chain.

    Bound: p = 2^(z log2e - lse log2e) is formed in FP32.  The rounding of the
    ~17-magnitude argument (and of lse) leaves a relative error of ~1e-6 in p,
    plus ~2.4e-7 from ex2.approx.  A relative error d moves an entry across a
    bf16 rounding midpoint with probability ~d * 2^7.5.  At d <= 1.5e-6 that is
    <= 2.7e-4 of the entries, so at least 99.97% must round correctly."""
    p = synth.logits_inputs(257, 151936, seed=257)
    gl = torch.tensor(p["gl"]).to(torch.bfloat16).float().numpy()
    x, y, g_dev = dev(p["logits"], "bf16"), dev(p["y"]), dev(gl)
    _, _, g = run(lib, x, y, g_dev)
    g_ref = O.logits_backward(gl, p["logits"], p["y"], "bf16")
    acc = accuracy(g, g_ref)
    print(f"dlogits 257 x 151936: {acc}")
    assert acc["correctly_rounded"] >= 0.9997, acc
    fused = accuracy(run_fused(lib, x.clone(), y, g_dev)[2], g_ref)
    assert fused == acc
