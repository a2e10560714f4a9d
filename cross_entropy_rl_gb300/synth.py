"""Seeded synthetic inputs for the fused linear log-probability path.

This module only draws random numbers and rounds them to the storage dtype.
It holds none of the method's arithmetic, so both the CUDA path and the FP64
oracle can be fed from it without sharing any of the computation.

Recipe (the workloads of the fused ``linear_logp`` scope request and of the
logits-input logp kernel; N(mu, s2) reads its second argument as a variance):

* hidden ~ N(0, 1), weight ~ N(0, 1/D), bias ~ N(0, 0.01)
* targets uniform in [0, V), int64
* grad_logp ~ N(0, 1), or the mean-loss constant 1/N, optionally with a seeded
  10 % of rows set to exactly +0
* logits ~ N(0, 2)

Values are drawn in float32 from numpy's PCG64 generator keyed by
``(seed, stream)``, scaled in float32 and rounded to the storage dtype with
round-to-nearest-even.  16-bit storage is returned as raw ``uint16`` bit
patterns for bf16 and as ``float16`` for fp16, so the exact bytes handed to the
GPU are also what the oracle decodes.
"""
from __future__ import annotations

import numpy as np

DTYPES = ("f32", "f16", "bf16")

# independent streams per tensor, so changing one size does not shift another
_STREAM = {"hidden": 1, "weight": 2, "bias": 3, "targets": 4, "grad": 5,
           "zero_rows": 6, "logits": 7, "sample": 8}

_CHUNK = 1 << 24  # elements drawn per block, bounds the float32 temporaries


def _rng(seed: int, stream: str) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([int(seed), _STREAM[stream]]))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return the bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    if nan.any():
        r[nan] = ((u[nan] >> 16) | 0x40).astype(np.uint16)
    return r


def to_storage(x32: np.ndarray, dtype: str) -> np.ndarray:
    """Round a float32 array to the storage dtype (bf16 as uint16 bits)."""
    if dtype == "f32":
        return np.ascontiguousarray(x32, dtype=np.float32)
    if dtype == "f16":
        return x32.astype(np.float16)
    if dtype == "bf16":
        return f32_to_bf16_bits(x32)
    raise ValueError(f"unknown dtype {dtype!r}")


def normal(seed: int, stream: str, shape, std: float, dtype: str = "f32") -> np.ndarray:
    """N(0, std^2) drawn in float32 blocks, scaled, rounded to ``dtype``."""
    shape = tuple(int(s) for s in shape)
    total = int(np.prod(shape)) if shape else 1
    g = _rng(seed, stream)
    out_dtype = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}[dtype]
    out = np.empty(total, dtype=out_dtype)
    std32 = np.float32(std)
    for s in range(0, total, _CHUNK):
        e = min(total, s + _CHUNK)
        x = g.standard_normal(e - s, dtype=np.float32)
        x *= std32
        out[s:e] = to_storage(x, dtype)
    return out.reshape(shape)


def uniform_targets(seed: int, N: int, V: int) -> np.ndarray:
    return _rng(seed, "targets").integers(0, V, size=int(N), dtype=np.int64)


def zero_rows(seed: int, N: int, frac: float) -> np.ndarray:
    """Indices of exactly round(frac*N) rows picked by a seeded permutation."""
    k = int(round(frac * N))
    return np.sort(_rng(seed, "zero_rows").permutation(int(N))[:k])


def sample_rows(seed: int, N: int, k: int = 256) -> np.ndarray:
    """k distinct rows, always including 0, N//2 and N-1 (sorted)."""
    N = int(N)
    if N <= k:
        return np.arange(N, dtype=np.int64)
    must = {0, N // 2, N - 1}
    perm = _rng(seed, "sample").permutation(N)
    rest = [int(i) for i in perm if int(i) not in must][: k - len(must)]
    return np.array(sorted(must.union(rest)), dtype=np.int64)


def linear_inputs(N, D, V, dtype="bf16", bias=False, seed=0, grad="normal",
                  zero_frac=0.0):
    """Inputs of one linear_logp problem.

    grad: "normal" (N(0,1)) or "mean" (the constant 1/N, a mean loss).
    zero_frac: fraction of grad_logp rows set to exactly +0.
    """
    h = normal(seed, "hidden", (N, D), 1.0, dtype)
    W = normal(seed, "weight", (V, D), float(np.sqrt(1.0 / D)), dtype)
    b = normal(seed, "bias", (V,), 0.1, dtype) if bias else None
    y = uniform_targets(seed, N, V)
    if grad == "normal":
        gl = normal(seed, "grad", (N,), 1.0, "f32")
    elif grad == "mean":
        gl = np.full((N,), np.float32(1.0 / max(N, 1)), dtype=np.float32)
    else:
        raise ValueError(grad)
    if zero_frac:
        gl[zero_rows(seed, N, zero_frac)] = np.float32(0.0)
    return dict(h=h, W=W, b=b, y=y, gl=gl, dtype=dtype, N=N, D=D, V=V)


def logits_inputs(N, V, seed=0, dtype="bf16", ld=None, var=2.0):
    """Logits [N, ld] (columns >= V are padding), targets, grad_logp."""
    ld = V if ld is None else ld
    x = normal(seed, "logits", (N, ld), float(np.sqrt(var)), dtype)
    y = uniform_targets(seed, N, V)
    gl = normal(seed, "grad", (N,), 1.0, "f32")
    return dict(logits=x, y=y, gl=gl, dtype=dtype, N=N, V=V, ld=ld)


# The five workloads, by what they are.
WORKLOADS = {
    "fp32_small": dict(N=128, D=256, V=4096, dtype="f32", bias=True, grad="normal"),
    "bf16_4k_2k_32k": dict(N=4096, D=2048, V=32768, dtype="bf16", bias=False, grad="normal"),
    "sweep_16k_4k_32000": dict(N=16384, D=4096, V=32000, grad="mean"),
    "logits_32k_151936": dict(N=32768, V=151936, dtype="bf16"),
    "bf16_32k_4k_151936": dict(N=32768, D=4096, V=151936, dtype="bf16", bias=False,
                               grad="normal", zero_frac=0.1),
}
