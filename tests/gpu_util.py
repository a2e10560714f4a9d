"""Helpers for the GPU parity tests: moving the synthetic storage arrays to
the device and comparing against the FP64 oracle with the stated
tolerances.

Tolerances (|got - ref| <= atol + rtol * |ref| (+ one output ulp)):
  FP32 operands:            atol 1e-5, rtol 5e-4 on every output
  16-bit operands, logp/lse: atol 5e-3
  16-bit operands, grads:    atol 5e-4, plus one ulp of the output dtype at
                             |ref| when the output itself is 16-bit (its own
                             rounding is up to half an ulp)

For 16-bit operands the off-target entries S = -grad * p of g are stored in
the operand dtype before the two gradient contractions.  By default the
library also keeps the rounding rest S - S_hi of every entry with p >= 2^-8
(the automatic hi / lo split), and every parity test holds the plain bound
above.  With the split switched off (split_s = "never") the 16-bit rounding
of S alone can exceed 5e-4 outside the benchmark shapes; s_rounding_bounds
gives its worst case, u * (|S| . |W|) for grad_hidden, u * (|S|^T . |h|) for
grad_weight and u * sum_n |S| for grad_bias (u = 2^-8 for bf16, 2^-11 for
fp16), used only by the test of that mode.
"""
import math

import numpy as np
import torch

TOL = {
    "f32": dict(logp=(1e-5, 5e-4), grad=(1e-5, 5e-4)),
    "f16": dict(logp=(5e-3, 0.0), grad=(5e-4, 0.0)),
    "bf16": dict(logp=(5e-3, 0.0), grad=(5e-4, 0.0)),
}
TORCH = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
MANT = {torch.bfloat16: 7, torch.float16: 10}


def dev(a, dtype=None, device="cuda"):
    """numpy storage array -> device tensor (bf16 arrives as uint16 bits)."""
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if dtype == "bf16":
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(a).to(device)


def host64(t):
    return t.detach().float().cpu().numpy().astype(np.float64) if t.dtype != torch.float64 else \
        t.detach().cpu().numpy()


def ulp(ref, tdtype):
    """One ulp of the 16-bit output dtype at |ref| (0 for FP32 outputs)."""
    if tdtype not in MANT:
        return np.zeros_like(ref)
    m = MANT[tdtype]
    a = np.abs(ref)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    sub = -14 if tdtype == torch.float16 else -126
    e = np.maximum(e, sub)
    return np.exp2(e - m)


def s_rounding_bounds(p, temperature=1.0):
    """Worst-case effect of storing S = -grad * p / T (off-target) in 16 bits."""
    import oracle as O

    dt = p["dtype"]
    if dt == "f32":
        return {}
    u = 2.0 ** -8 if dt == "bf16" else 2.0 ** -11
    h, W, b = O.decode(p["h"], dt), O.decode(p["W"], dt), O.decode(p["b"], dt)
    z = O.linear_logits(h, W, b) / temperature
    lse = O.logsumexp_rows(z)
    S = np.abs(np.asarray(p["gl"], np.float64))[:, None] * np.exp(z - lse[:, None]) / temperature
    y = np.asarray(p["y"])
    V = W.shape[0]
    ok = (y >= 0) & (y < V) & (np.asarray(p["gl"]) != 0)
    S[~ok] = 0.0
    idx = np.nonzero(ok)[0]
    S[idx, y[idx]] = 0.0
    return {"dh": u * S @ np.abs(W), "dW": u * S.T @ np.abs(h), "db": u * S.sum(axis=0)}


def check(name, got, ref, atol, rtol, out_dtype=None, report=None, extra=None):
    g = host64(got) if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert g.shape == ref.shape, (name, g.shape, ref.shape)
    if g.size == 0:
        return 0.0
    with np.errstate(invalid="ignore"):
        err = np.abs(g - ref)
    err = np.where(g == ref, 0.0, err)  # equal infinities match
    bound = atol + rtol * np.abs(np.where(np.isfinite(ref), ref, 0.0))
    if out_dtype is not None:
        bound = bound + ulp(np.where(np.isfinite(ref), ref, 0.0), out_dtype)
    if extra is not None:
        bound = bound + extra
    bad = ~(err <= bound)
    worst = float(np.nanmax(err)) if np.isfinite(err).any() else math.inf
    if report is not None:
        report[name] = worst
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err - bound, -np.inf)), err.shape)
        raise AssertionError(
            f"{name}: {int(bad.sum())}/{bad.size} outside tolerance; worst at {i}: got "
            f"{g[i]!r} ref {ref[i]!r} (bound {bound[i]:.3g}); max err {worst:.3g}")
    return worst


def assert_pos_zero(name, t):
    x = t.detach().float().cpu()
    assert bool((x == 0).all()), f"{name}: not all zero"
    assert not bool(torch.signbit(x).any()), f"{name}: negative zero present"


def bits_equal(a, b):
    return torch.equal(a.view(torch.int8) if a.dtype != torch.int8 else a,
                       b.view(torch.int8) if b.dtype != torch.int8 else b)


def bf16_round(r):
    """float64 values rounded to the nearest bf16 (ties to even), as float64."""
    r = np.asarray(r, np.float64)
    b = r.astype(np.float32).view(np.uint32)
    lo_bits = b & np.uint32(0xFFFF0000)
    lo = lo_bits.view(np.float32).astype(np.float64)
    hi = (lo_bits + np.uint32(0x10000)).view(np.float32).astype(np.float64)
    dlo, dhi = np.abs(r - lo), np.abs(r - hi)
    even = ((lo_bits >> np.uint32(16)) & np.uint32(1)) == 0
    return np.where((dlo < dhi) | ((dlo == dhi) & even), lo, hi)


def accuracy(got, ref):
    """Max abs error, max error / max |ref|, and the fraction of entries equal
    to the bf16 rounding of the FP64 reference."""
    g = host64(got)
    ref = np.asarray(ref, np.float64)
    err = np.abs(g - ref)
    return dict(max_abs=float(err.max()), max_over_max=float(err.max() / np.abs(ref).max()),
                correctly_rounded=float(np.mean(g == bf16_round(ref))))

