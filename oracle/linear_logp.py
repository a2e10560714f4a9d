"""FP64 CPU oracle for the fused linear log-probability (``linear_logp``) path.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check and
the benchmark's CPU-baseline leg may import this module.  It shares no code
with the CUDA path and the CUDA path never calls it.

What it computes is the dense definition, written out in float64 with numpy
(a library matmul serves as the contraction step; nothing is blocked, fused or
reordered beyond that):

* forward  (RL-Kernel issue #261, "Current accumulation" and "Static traffic
  model"; RL-Kernel PR #495, "Summary" / "Behavior changes"):
      z      = h . W^T (+ b)                      logits, [N, V]
      lse_n  = log sum_v exp(z_nv)                (max-shifted)
      logp_n = z_{n, y_n} - lse_n  if 0 <= y_n < V, else 0
* backward (RL-Kernel PR #495, "Benchmark script": the original VJP builds the
  FP32 softmax, subtracts one at the target and scales by -grad):
      p      = exp(z - lse)
      g_nv   = gl_n * ([v == y_n] - p_nv); the whole row is 0 when y_n is
               outside [0, V)
      dh     = g . W,   dW = g^T . h,   db = sum_n g_nv
* the same two steps with the logits given directly (logits-input variant).
* temperature T > 0 (the sampling temperature of RL rollouts; RL-Kernel PR
  #495, the vLLM provider evidence runs temperatures 1.0 and 0.7): every
  function takes ``temperature``; the distribution is softmax(z / T), so
  logp_n = z_{n, y_n} / T - logsumexp_v(z_nv / T) and the gradient with
  respect to z is gl_n * ([v == y_n] - p_nv) / T, p = softmax(z / T).
  T = 1 is the plain definition above.

Signed zeros: the correctness boundary of issue #261 keeps a +0-initialised
gradient table, so an entry that receives no non-zero contribution is +0.  The
oracle states this by adding +0.0 to every gradient it returns (IEEE:
-0 + +0 = +0, x + +0 = x otherwise), and rows with an invalid target or a zero
upstream gradient are exactly +0.

Inputs are the stored bytes: float32 and float16 arrays, or bfloat16 given as
uint16 bit patterns with ``dtype="bf16"``.  Every one of them embeds exactly in
float64.  ``dtype="f64"`` passes float64 arrays through (used by the finite
difference pins).
"""
from __future__ import annotations

import numpy as np


def decode(x, dtype: str) -> np.ndarray:
    """Stored values -> float64, exactly.  bf16 arrives as uint16 bits."""
    if x is None:
        return None
    x = np.asarray(x)
    if dtype == "bf16":
        if x.dtype != np.uint16:
            raise TypeError("bf16 input must be given as uint16 bit patterns")
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if dtype == "f16":
        return x.astype(np.float16).astype(np.float64)
    if dtype == "f32":
        return x.astype(np.float32).astype(np.float64)
    if dtype == "f64":
        return x.astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


def _valid(y: np.ndarray, V: int) -> np.ndarray:
    y = np.asarray(y, dtype=np.int64)
    return (y >= 0) & (y < V)


# ----------------------------------------------------------------------------
# logits given: forward and backward of logp_n = z[n, y_n] - logsumexp_v z[n, v]
# ----------------------------------------------------------------------------

def logsumexp_rows(z: np.ndarray) -> np.ndarray:
    """lse_n = M_n + log sum_v exp(z_nv - M_n), M_n = max_v z_nv.

    A row whose entries are all -inf has lse = -inf (an empty sum).
    """
    M = z.max(axis=1)
    lse = np.full(z.shape[0], -np.inf)
    live = np.isfinite(M) | (M == np.inf)
    if live.any():
        with np.errstate(invalid="ignore", over="ignore"):
            s = np.exp(z[live] - M[live, None]).sum(axis=1)
        lse[live] = M[live] + np.log(s)
    return lse


def logp_from_logits(z: np.ndarray, y) -> tuple[np.ndarray, np.ndarray]:
    """(logp, lse) of each row; logp is 0 where the target is outside [0, V)."""
    N, V = z.shape
    lse = logsumexp_rows(z)
    ok = _valid(y, V)
    logp = np.zeros(N)
    idx = np.nonzero(ok)[0]
    with np.errstate(invalid="ignore"):
        logp[idx] = z[idx, np.asarray(y)[idx]] - lse[idx]
    return logp, lse


def grad_logits(z: np.ndarray, y, gl, lse=None) -> np.ndarray:
    """g = gl * (onehot(y) - softmax(z)); +0 rows for invalid targets."""
    N, V = z.shape
    if lse is None:
        lse = logsumexp_rows(z)
    gl = np.asarray(gl, dtype=np.float64)
    ok = _valid(y, V)
    with np.errstate(invalid="ignore", over="ignore"):
        p = np.exp(z - lse[:, None])
    onehot = np.zeros((N, V))
    idx = np.nonzero(ok)[0]
    onehot[idx, np.asarray(y)[idx]] = 1.0
    g = gl[:, None] * (onehot - p)
    g[~ok] = 0.0
    g[gl == 0.0] = 0.0
    return g + 0.0


# ----------------------------------------------------------------------------
# linear: z = h W^T (+ b)
# ----------------------------------------------------------------------------

def linear_logits(h, W, b=None) -> np.ndarray:
    """z = h . W^T (+ b) in float64 (h [N, D], W [V, D], b [V])."""
    z = h @ W.T
    if b is not None:
        z = z + b[None, :]
    return z


def _tempered(z: np.ndarray, temperature: float) -> np.ndarray:
    """z / T (the logits of the temperature-scaled distribution)."""
    if not temperature > 0:
        raise ValueError("temperature must be > 0")
    return z if temperature == 1.0 else z / temperature


def _tempered_grad(zT, y, gl, temperature: float, lse=None) -> np.ndarray:
    """d(sum gl logp_T)/dz = grad_logits(z / T) / T."""
    g = grad_logits(zT, y, gl, lse)
    return g if temperature == 1.0 else g / temperature + 0.0


def linear_forward(h, W, b, y, dtype: str, temperature: float = 1.0):
    """(logp, lse) for hidden h [N, D], weight W [V, D], optional bias b [V];
    lse is the one of the tempered logits z / T."""
    h64, W64, b64 = decode(h, dtype), decode(W, dtype), decode(b, dtype)
    return logp_from_logits(_tempered(linear_logits(h64, W64, b64), temperature), y)


def linear_backward(gl, h, W, b, y, dtype: str, dw_rows=None, temperature: float = 1.0):
    """(dh, dW, db) of sum_n gl_n * logp_n.

    dw_rows: optional index array; dW is then returned only for those vocab
    rows (each is a full sum over tokens, nothing is truncated).
    """
    h64, W64, b64 = decode(h, dtype), decode(W, dtype), decode(b, dtype)
    z = _tempered(linear_logits(h64, W64, b64), temperature)
    g = _tempered_grad(z, y, gl, temperature)
    dh = g @ W64 + 0.0
    gT = g.T if dw_rows is None else g.T[np.asarray(dw_rows)]
    dW = gT @ h64 + 0.0
    db = g.sum(axis=0) + 0.0
    return dh, dW, db


def linear_forward_backward(gl, h, W, b, y, dtype: str, dw_rows=None,
                            temperature: float = 1.0):
    """Forward and backward of one problem, sharing the float64 logits."""
    h64, W64, b64 = decode(h, dtype), decode(W, dtype), decode(b, dtype)
    z = _tempered(linear_logits(h64, W64, b64), temperature)
    logp, lse = logp_from_logits(z, y)
    g = _tempered_grad(z, y, gl, temperature, lse)
    dh = g @ W64 + 0.0
    gT = g.T if dw_rows is None else g.T[np.asarray(dw_rows)]
    dW = gT @ h64 + 0.0
    db = g.sum(axis=0) + 0.0
    return dict(logp=logp, lse=lse, dh=dh, dW=dW, db=db)


def linear_rows(gl, h, W, b, y, dtype: str, rows, dw_rows=None, temperature: float = 1.0):
    """Outputs restricted to the token rows ``rows``.

    logp, lse and dh of those rows are exactly the full problem's rows
    (each row is independent).  dW and db are the contribution of those rows
    only: the full gradient of sum over n in rows of gl_n * logp_n, i.e. the
    gradient of a run whose grad_logp is zero outside ``rows``.
    """
    rows = np.asarray(rows, dtype=np.int64)
    h_r = np.asarray(h)[rows]
    y_r = np.asarray(y)[rows]
    gl_r = np.asarray(gl)[rows]
    return linear_forward_backward(gl_r, h_r, W, b, y_r, dtype, dw_rows=dw_rows,
                                   temperature=temperature)


def logits_forward(x, y, dtype: str, V=None, temperature: float = 1.0):
    """(logp, lse) from stored logits x [N, ld]; columns >= V are ignored."""
    z = decode(x, dtype)
    if V is not None:
        z = z[:, :V]
    return logp_from_logits(_tempered(z, temperature), y)


def logits_backward(gl, x, y, dtype: str, V=None, temperature: float = 1.0):
    """Gradient w.r.t. the logits [N, V] (float64) of sum_n gl_n * logp_n."""
    z = decode(x, dtype)
    if V is not None:
        z = z[:, :V]
    return _tempered_grad(_tempered(z, temperature), y, gl, temperature)
