"""Pins of the FP64 oracle against facts fixed by the mathematics.

None of these re-types the oracle's formula: they use closed forms (V = 1,
V = 2 softplus, uniform logits, shift invariance), central finite differences
of the oracle's own forward (which pin every gradient to the forward), an
unshifted brute-force log-sum-exp with exact summation, invariants of the
softmax (rows of onehot - p sum to zero) and the special cases of the
contract (invalid targets, zero upstream gradient, empty input, -inf tail).
"""
import math

import numpy as np
import pytest

import oracle as O
from cross_entropy_rl_gb300 import synth


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# --------------------------------------------------------------- decode ----

def test_decode_bf16_bit_patterns():
    bits = np.array([0x3F80, 0xC000, 0x0001, 0x7F80, 0x8000, 0x3F81], dtype=np.uint16)
    v = O.decode(bits, "bf16")
    assert v[0] == 1.0
    assert v[1] == -2.0
    assert v[2] == 2.0 ** -133          # smallest bf16 subnormal
    assert v[3] == np.inf
    assert v[4] == 0.0 and np.signbit(v[4])
    assert v[5] == 1.0 + 2.0 ** -7       # one ulp above 1 (7 stored mantissa bits)


def test_decode_fp16_and_fp32_exact():
    assert O.decode(np.array([65504.0], np.float16), "f16")[0] == 65504.0
    assert O.decode(np.array([2 ** -24], np.float16), "f16")[0] == 2.0 ** -24
    x = np.array([1.0 + 2 ** -23], np.float32)
    assert O.decode(x, "f32")[0] == 1.0 + 2.0 ** -23


def test_synth_bf16_rounding_is_nearest_even():
    x = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -8 + 2 ** -20], np.float32)
    b = O.decode(synth.f32_to_bf16_bits(x), "bf16")
    assert b[0] == 1.0                   # tie -> even
    assert b[1] == 1.0 + 2 ** -6         # tie -> even (upwards)
    assert b[2] == 1.0 + 2 ** -7         # above the tie -> up


# ----------------------------------------------------------- closed forms ----

def test_single_class_vocab():
    """V = 1: the only class has probability 1, so logp = 0 and every gradient is 0."""
    h, W, b = _rand((3, 4), 1), _rand((1, 4), 2), _rand((1,), 3)
    y = np.zeros(3, np.int64)
    gl = np.array([1.5, -2.0, 0.25])
    r = O.linear_forward_backward(gl, h, W, b, y, "f64")
    np.testing.assert_allclose(r["logp"], 0.0, atol=1e-15)
    np.testing.assert_allclose(r["lse"], (h @ W.T)[:, 0] + b[0], rtol=1e-15)
    for k in ("dh", "dW", "db"):
        assert np.abs(r[k]).max() < 1e-15


def test_two_class_softplus():
    """V = 2: logp_y = -softplus(z_other - z_y) and d logp / d z_y = sigmoid(z_o - z_y)."""
    h = np.array([[1.0, 2.0], [0.5, -1.0]])
    W = np.array([[1.0, 0.0], [0.0, 1.0]])
    b = np.array([0.25, -0.5])
    y = np.array([0, 1])
    gl = np.array([1.0, -3.0])
    r = O.linear_forward_backward(gl, h, W, b, y, "f64")
    z = [[1.25, 1.5], [0.75, -1.5]]     # h W^T + b, by hand
    for n in range(2):
        zy, zo = z[n][y[n]], z[n][1 - y[n]]
        sp = math.log1p(math.exp(zo - zy))
        assert r["logp"][n] == pytest.approx(-sp, abs=1e-15)
        sig = 1.0 / (1.0 + math.exp(-(zo - zy)))
        # dL/dz_y = gl*sig, dL/dz_o = -gl*sig; dh = sum_v dL/dz_v W_v
        dz = np.zeros(2)
        dz[y[n]] = gl[n] * sig
        dz[1 - y[n]] = -gl[n] * sig
        np.testing.assert_allclose(r["dh"][n], dz @ W, atol=1e-15)


def test_uniform_logits_give_minus_log_v():
    """Equal rows of W and no bias: p = 1/V, logp = -log V, dh = 0."""
    N, D, V = 5, 6, 4096
    h = _rand((N, D), 4)
    W = np.tile(_rand((1, D), 5), (V, 1))
    y = np.random.default_rng(6).integers(0, V, N)
    gl = _rand((N,), 7)
    r = O.linear_forward_backward(gl, h, W, None, y, "f64")
    np.testing.assert_allclose(r["logp"], -math.log(V), rtol=1e-14)
    assert np.abs(r["dh"]).max() < 1e-12


def test_shift_invariance():
    """Adding a constant to every logit of a row leaves logp unchanged."""
    N, D, V = 6, 8, 33
    h, W, b = _rand((N, D), 8), _rand((V, D), 9), _rand((V,), 10)
    y = np.random.default_rng(11).integers(0, V, N)
    base, _ = O.linear_forward(h, W, b, y, "f64")
    shifted_b, _ = O.linear_forward(h, W, b + 3.75, y, "f64")
    c = _rand((D,), 12)
    shifted_w, _ = O.linear_forward(h, W + c[None, :], b, y, "f64")
    np.testing.assert_allclose(shifted_b, base, atol=1e-13)
    np.testing.assert_allclose(shifted_w, base, atol=1e-12)


# -------------------------------------------------------------- bounds ----

def test_probability_bounds():
    N, D, V = 16, 12, 257
    h, W = _rand((N, D), 13), _rand((V, D), 14, 0.5)
    y = np.random.default_rng(15).integers(0, V, N)
    logp, lse = O.linear_forward(h, W, None, y, "f64")
    zmax = (h @ W.T).max(axis=1)
    assert (logp <= 0).all()
    assert (lse >= zmax).all()
    assert (lse <= zmax + math.log(V) + 1e-12).all()


def test_bruteforce_logsumexp_without_shift():
    """lse by exact summation of exp(z) (no max shift) on a tiny problem."""
    N, D, V = 4, 3, 9
    h, W, b = _rand((N, D), 16), _rand((V, D), 17), _rand((V,), 18)
    y = np.array([0, 8, 3, 5])
    logp, lse = O.linear_forward(h, W, b, y, "f64")
    for n in range(N):
        zs = [math.fsum(h[n, d] * W[v, d] for d in range(D)) + b[v] for v in range(V)]
        want = math.log(math.fsum(math.exp(t) for t in zs))
        assert lse[n] == pytest.approx(want, abs=1e-13)
        assert logp[n] == pytest.approx(zs[y[n]] - want, abs=1e-13)


# ---------------------------------------------------- finite differences ----

def _loss(gl, h, W, b, y):
    logp, _ = O.linear_forward(h, W, b, y, "f64")
    return float(np.dot(gl, logp))


@pytest.mark.parametrize("seed", [0, 1])
def test_finite_differences(seed):
    """Central differences of sum_n gl_n logp_n match dh, dW and db."""
    N, D, V = 3, 5, 7
    h, W, b = _rand((N, D), 20 + seed), _rand((V, D), 30 + seed, 0.7), _rand((V,), 40 + seed)
    y = np.random.default_rng(50 + seed).integers(0, V, N)
    gl = _rand((N,), 60 + seed)
    dh, dW, db = O.linear_backward(gl, h, W, b, y, "f64")
    eps = 1e-6

    def fd(arr, idx):
        a0 = arr[idx]
        arr[idx] = a0 + eps
        lp = _loss(gl, h, W, b, y)
        arr[idx] = a0 - eps
        lm = _loss(gl, h, W, b, y)
        arr[idx] = a0
        return (lp - lm) / (2 * eps)

    for arr, grad in ((h, dh), (W, dW), (b, db)):
        num = np.array([fd(arr, i) for i in np.ndindex(arr.shape)]).reshape(arr.shape)
        scale = max(1.0, np.abs(grad).max())
        assert np.abs(num - grad).max() / scale < 1e-6


def test_finite_differences_logits():
    N, V = 3, 6
    z = _rand((N, V), 70)
    y = np.array([2, 0, 5])
    gl = _rand((N,), 71)
    g = O.logits_backward(gl, z, y, "f64")
    eps = 1e-6
    for n in range(N):
        for v in range(V):
            zp, zm = z.copy(), z.copy()
            zp[n, v] += eps
            zm[n, v] -= eps
            lp = np.dot(gl, O.logits_forward(zp, y, "f64")[0])
            lm = np.dot(gl, O.logits_forward(zm, y, "f64")[0])
            assert (lp - lm) / (2 * eps) == pytest.approx(g[n, v], abs=1e-8)


# ----------------------------------------------------------- invariants ----

def test_gradient_rows_sum_to_zero():
    """Each row of onehot - p sums to 0, so sum_v db_v = 0 and sum_v dW_v = 0."""
    N, D, V = 9, 7, 31
    h, W, b = _rand((N, D), 80), _rand((V, D), 81), _rand((V,), 82)
    y = np.random.default_rng(83).integers(0, V, N)
    gl = _rand((N,), 84)
    dh, dW, db = O.linear_backward(gl, h, W, b, y, "f64")
    assert abs(db.sum()) < 1e-12
    assert np.abs(dW.sum(axis=0)).max() < 1e-12


def test_row_subset_matches_full_problem():
    """logp/lse/dh of selected rows equal the full run; dW/db equal a run with
    grad_logp zeroed outside the selection."""
    N, D, V = 12, 5, 19
    h, W, b = _rand((N, D), 90), _rand((V, D), 91), _rand((V,), 92)
    y = np.random.default_rng(93).integers(0, V, N)
    gl = _rand((N,), 94)
    rows = np.array([0, 4, 11])
    full = O.linear_forward_backward(gl, h, W, b, y, "f64")
    part = O.linear_rows(gl, h, W, b, y, "f64", rows)
    for k in ("logp", "lse", "dh"):
        np.testing.assert_array_equal(part[k], full[k][rows])
    glz = np.zeros_like(gl)
    glz[rows] = gl[rows]
    masked = O.linear_forward_backward(glz, h, W, b, y, "f64")
    np.testing.assert_allclose(part["dW"], masked["dW"], atol=1e-14)
    np.testing.assert_allclose(part["db"], masked["db"], atol=1e-14)
    sub = O.linear_rows(gl, h, W, b, y, "f64", rows, dw_rows=np.array([3, 7]))
    np.testing.assert_array_equal(sub["dW"], part["dW"][[3, 7]])


# --------------------------------------------------------- special cases ----

def test_invalid_targets_give_zero_rows():
    N, D, V = 6, 4, 10
    h, W, b = _rand((N, D), 100), _rand((V, D), 101), _rand((V,), 102)
    y = np.array([-100, 3, V, 7, V + 5, 0])
    gl = _rand((N,), 103)
    r = O.linear_forward_backward(gl, h, W, b, y, "f64")
    bad = np.array([0, 2, 4])
    assert (r["logp"][bad] == 0).all() and not np.signbit(r["logp"][bad]).any()
    assert (r["dh"][bad] == 0).all() and not np.signbit(r["dh"][bad]).any()
    good = np.array([1, 3, 5])
    glz = gl.copy()
    glz[bad] = 0
    ref = O.linear_forward_backward(glz, h, W, b, np.where(y < 0, 0, np.minimum(y, V - 1)), "f64")
    np.testing.assert_array_equal(r["dh"][good], ref["dh"][good])
    np.testing.assert_allclose(r["dW"], ref["dW"], atol=1e-15)


def test_zero_upstream_gives_positive_zeros():
    N, D, V = 5, 6, 11
    h, W, b = _rand((N, D), 110), _rand((V, D), 111), _rand((V,), 112)
    y = np.random.default_rng(113).integers(0, V, N)
    gl = np.zeros(N)
    gl[2] = -0.0
    dh, dW, db = O.linear_backward(gl, h, W, b, y, "f64")
    for a in (dh, dW, db):
        assert (a == 0).all() and not np.signbit(a).any()


def test_empty_input():
    D, V = 4, 7
    h = np.zeros((0, D))
    W, b = _rand((V, D), 120), _rand((V,), 121)
    r = O.linear_forward_backward(np.zeros(0), h, W, b, np.zeros(0, np.int64), "f64")
    assert r["logp"].shape == (0,) and r["dh"].shape == (0, D)
    assert r["dW"].shape == (V, D) and (r["dW"] == 0).all() and not np.signbit(r["dW"]).any()
    assert (r["db"] == 0).all() and not np.signbit(r["db"]).any()


def test_masked_tail_logits():
    """-inf entries contribute nothing; an all -inf row with an invalid target
    has logp 0, lse -inf and a zero gradient row."""
    N, V = 4, 12
    z = _rand((N, V), 130)
    zm = z.copy()
    zm[:, 8:] = -np.inf
    zm[3, :] = -np.inf
    y = np.array([1, 7, 0, -100])
    gl = _rand((N,), 131)
    logp, lse = O.logits_forward(zm, y, "f64")
    ref_logp, ref_lse = O.logits_forward(z[:, :8], y, "f64")
    np.testing.assert_allclose(logp[:3], ref_logp[:3], rtol=1e-15)
    assert lse[3] == -np.inf and logp[3] == 0.0
    g = O.logits_backward(gl, zm, y, "f64")
    assert np.isfinite(g).all()
    assert (g[:, 8:] == 0).all() and not np.signbit(g[:, 8:]).any()
    assert (g[3] == 0).all()
    np.testing.assert_allclose(g[:3, :8], O.logits_backward(gl[:3], z[:3, :8], y[:3], "f64"),
                               atol=1e-16)


# ---------------------------------------------------------- temperature ----

def test_temperature_two_class_softplus():
    """V = 2: logp_T of class 0 is -softplus((z1 - z0) / T) (closed form)."""
    z = np.array([[0.3, -1.1], [2.0, 2.5], [-4.0, 3.0]])
    y = np.array([0, 0, 1])
    for T in (0.7, 1.0, 2.5):
        logp, _ = O.logits_forward(z, y, "f64", temperature=T)
        d = np.array([z[0, 1] - z[0, 0], z[1, 1] - z[1, 0], z[2, 0] - z[2, 1]]) / T
        assert np.allclose(logp, -np.log1p(np.exp(d)), rtol=0, atol=1e-15)


def test_temperature_limits():
    """T -> inf: every class has probability 1/V; T -> 0: the argmax class
    has logp -> 0 and the others -> -inf."""
    z = _rand((4, 9), 120)
    y = np.array([0, 3, 8, 5])
    logp, _ = O.logits_forward(z, y, "f64", temperature=1e9)
    assert np.allclose(logp, -np.log(9.0), atol=1e-8)
    am = z.argmax(axis=1)
    logp, _ = O.logits_forward(z, am, "f64", temperature=1e-3)
    assert np.all(logp > -1e-10) and np.all(logp <= 0.0)
    other = (am + 1) % 9
    logp, _ = O.logits_forward(z, other, "f64", temperature=1e-3)
    assert np.all(logp < -10.0)


@pytest.mark.parametrize("T", [0.7, 1.6])
def test_temperature_finite_differences(T):
    """Central differences of sum_n gl_n logp_T,n (the oracle's forward) match
    its dh, dW, db and logits gradients: this pins the 1 / T factor."""
    N, D, V = 3, 4, 6
    h, W, b = _rand((N, D), 130), _rand((V, D), 131, 0.8), _rand((V,), 132)
    y = np.array([1, 5, 0])
    gl = _rand((N,), 133)
    dh, dW, db = O.linear_backward(gl, h, W, b, y, "f64", temperature=T)
    eps = 1e-6

    def loss():
        return float(np.dot(gl, O.linear_forward(h, W, b, y, "f64", temperature=T)[0]))

    for arr, grad in ((h, dh), (W, dW), (b, db)):
        num = np.zeros(arr.shape)
        for i in np.ndindex(arr.shape):
            a0 = arr[i]
            arr[i] = a0 + eps
            lp = loss()
            arr[i] = a0 - eps
            lm = loss()
            arr[i] = a0
            num[i] = (lp - lm) / (2 * eps)
        assert np.abs(num - grad).max() / max(1.0, np.abs(grad).max()) < 1e-6
    z = _rand((N, V), 134)
    g = O.logits_backward(gl, z, y, "f64", temperature=T)
    for n in range(N):
        for v in range(V):
            zp, zm = z.copy(), z.copy()
            zp[n, v] += eps
            zm[n, v] -= eps
            lp = np.dot(gl, O.logits_forward(zp, y, "f64", temperature=T)[0])
            lm = np.dot(gl, O.logits_forward(zm, y, "f64", temperature=T)[0])
            assert (lp - lm) / (2 * eps) == pytest.approx(g[n, v], abs=1e-8)
