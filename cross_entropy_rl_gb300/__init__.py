"""GB300-native fused linear log-probability: thin Python binding.

The computation runs in the CUDA library ``_lib/libll_gb300.so`` built from
``csrc/`` (C ABI in ``include/ll_linear_logp.h``).  This module only
marshals arguments: it takes torch tensors, allocates outputs and the scratch
workspace with torch (the library itself never allocates), and passes raw
pointers plus the current CUDA stream.  There is no fallback: every call
raises when the library is missing or a call returns an error status.

    import cross_entropy_rl_gb300 as ll
    logp, lse = ll.forward(hidden, weight, bias, targets)
    dh, dW, db = ll.backward(grad_logp, hidden, weight, bias, targets, lse)
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "LLError", "load", "lib", "forward", "backward", "forward_backward", "logits_fwd",
    "logits_bwd", "logits_fwd_bwd", "shard_segments", "forward_shard", "lse_merge",
    "backward_shard", "SEGMENT_COLS",
    "workspace_size", "check_status", "DTYPE_CODES", "EXPORTS",
]

_LIB = None
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libll_gb300.so")

# ll_dtype codes of the C ABI
LL_F32, LL_F16, LL_BF16 = 0, 1, 2
# vocab entries per LSE segment; vocab shards start on a multiple of it
SEGMENT_COLS = 1024

_c_i64 = ctypes.c_int64
_c_p = ctypes.c_void_p
_c_int = ctypes.c_int
_c_size = ctypes.c_size_t

# name -> (restype, argtypes): every symbol the header declares
EXPORTS = {
    "ll_status_string": (ctypes.c_char_p, [_c_int]),
    "ll_version": (_c_int, []),
    "ll_workspace_size": (_c_size, [_c_i64, _c_i64, _c_i64, _c_int, _c_int, _c_int, _c_int]),
    "ll_forward": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_i64, _c_i64, _c_i64, _c_int,
                            _c_p, _c_p, _c_p, _c_size, _c_p]),
    "ll_backward": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i64, _c_i64, _c_i64,
                             _c_int, _c_int, _c_int, _c_int, _c_p, _c_int, _c_p, _c_int,
                             _c_p, _c_int, _c_p, _c_size, _c_p]),
    "ll_forward_backward": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_i64, _c_i64, _c_i64,
                                     _c_int, _c_p, _c_p, _c_int, _c_int, _c_int, _c_p, _c_int,
                                     _c_p, _c_int, _c_p, _c_int, _c_p, _c_size, _c_p]),
    "logits_logp_fwd": (_c_int, [_c_p, _c_i64, _c_int, _c_p, _c_i64, _c_i64, _c_p, _c_p, _c_p]),
    "logits_logp_bwd": (_c_int, [_c_p, _c_p, _c_i64, _c_int, _c_p, _c_p, _c_i64, _c_i64,
                                 _c_p, _c_p]),
    "logits_logp_fwd_bwd": (_c_int, [_c_p, _c_p, _c_i64, _c_int, _c_p, _c_i64, _c_i64, _c_p,
                                     _c_p, _c_p, _c_p]),
    "ll_shard_segments": (_c_i64, [_c_i64]),
    "ll_workspace_size_shard": (_c_size, [_c_i64, _c_i64, _c_i64, _c_int, _c_int, _c_int,
                                          _c_int]),
    "ll_forward_shard": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_i64, _c_i64, _c_i64, _c_i64,
                                  _c_i64, _c_int, _c_p, _c_p, _c_p, _c_p, _c_size, _c_p, _c_p]),
    "ll_lse_merge": (_c_int, [_c_p, _c_p, _c_i64, _c_i64, _c_p, _c_p, _c_i64, _c_i64, _c_p,
                              _c_p, _c_p]),
    "ll_backward_shard": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i64, _c_i64, _c_i64,
                                   _c_i64, _c_i64, _c_int, _c_int, _c_int, _c_int, _c_p,
                                   _c_int, _c_p, _c_int, _c_p, _c_int, _c_p, _c_size, _c_p,
                                   _c_p]),
    "ll_forward_ex": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_i64, _c_i64, _c_i64, _c_int,
                               _c_p, _c_p, _c_p, _c_size, _c_p, _c_p]),
    "ll_backward_ex": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i64, _c_i64, _c_i64,
                                _c_int, _c_int, _c_int, _c_int, _c_p, _c_int, _c_p, _c_int,
                                _c_p, _c_int, _c_p, _c_size, _c_p, _c_p]),
    "ll_forward_backward_ex": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_i64, _c_i64, _c_i64,
                                        _c_int, _c_p, _c_p, _c_int, _c_int, _c_int, _c_p,
                                        _c_int, _c_p, _c_int, _c_p, _c_int, _c_p, _c_size,
                                        _c_p, _c_p]),
    "logits_logp_fwd_ex": (_c_int, [_c_p, _c_i64, _c_int, _c_p, _c_i64, _c_i64, _c_p, _c_p,
                                    _c_p, _c_p]),
    "logits_logp_bwd_ex": (_c_int, [_c_p, _c_p, _c_i64, _c_int, _c_p, _c_p, _c_i64, _c_i64,
                                    _c_p, _c_p, _c_p]),
    "logits_logp_fwd_bwd_ex": (_c_int, [_c_p, _c_p, _c_i64, _c_int, _c_p, _c_i64, _c_i64,
                                        _c_p, _c_p, _c_p, _c_p, _c_p]),
    "ll_check_status": (_c_int, [_c_p]),
    "ll_set_wait_limit_ns": (None, [_c_i64]),
    "ll_debug_unsatisfied_wait": (_c_int, [_c_p, _c_p]),
    "ll_forward_noalloc": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_i64, _c_i64, _c_i64, _c_int,
                                    _c_p, _c_p, _c_p]),
    "ll_launch_count": (ctypes.c_longlong, []),
    "ll_profile_enable": (None, [_c_int]),
    "ll_profile_summary": (_c_int, [ctypes.c_char_p, _c_size]),
    "ll_sum_ordered": (_c_int, [_c_p, _c_i64, _c_i64, _c_i64, _c_int, _c_p, _c_p]),
}


class Options(ctypes.Structure):
    """ll_options of the C ABI."""
    _fields_ = [("temperature", ctypes.c_float), ("split_s", ctypes.c_int),
                ("reserved", ctypes.c_int * 6)]


SPLIT_MODES = {"auto": 0, "always": 1, "never": 2}


def _split_code(split_s) -> int:
    """ll_options.split_s of a binding argument: "auto" (or None, the
    default), "always" (or True) or "never" (or False)."""
    if split_s is None:
        return 0
    if isinstance(split_s, bool):
        return 1 if split_s else 2
    if split_s not in SPLIT_MODES:
        raise ValueError(f"split_s must be one of {sorted(SPLIT_MODES)}, True, False or None")
    return SPLIT_MODES[split_s]


def _opts(temperature=1.0, split_s="auto"):
    """ll_options pointer for a call (None when every option is default)."""
    t = 1.0 if temperature is None else float(temperature)
    if not t > 0:
        raise ValueError("temperature must be > 0")
    code = _split_code(split_s)
    if t == 1.0 and code == 0:
        return None
    return ctypes.byref(Options(temperature=t, split_s=code))


class LLError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = "?"
        if _LIB is not None:
            msg = _LIB.ll_status_string(status).decode()
        super().__init__(f"{fn} failed: status {status} ({msg})")
        self.status = status


def load(path: str | None = None):
    """Load the shared library (raises if it has not been built)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(
            f"CUDA library not built: {path} is missing "
            "(run `python -m cross_entropy_rl_gb300.build`)")
    lib_ = ctypes.CDLL(path)
    for name, (res, args) in EXPORTS.items():
        f = getattr(lib_, name)
        f.restype = res
        f.argtypes = args
    _LIB = lib_
    return _LIB


def lib():
    return load()


def _torch():
    import torch
    return torch


def _code(dtype) -> int:
    torch = _torch()
    m = {torch.float32: LL_F32, torch.float16: LL_F16, torch.bfloat16: LL_BF16}
    if dtype not in m:
        raise TypeError(f"unsupported dtype {dtype}")
    return m[dtype]


def DTYPE_CODES():
    torch = _torch()
    return {torch.float32: LL_F32, torch.float16: LL_F16, torch.bfloat16: LL_BF16}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    torch = _torch()
    if stream is None and not torch.cuda.is_available():
        return ctypes.c_void_p(None)  # the call itself then fails: no device memory
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn: str, st: int):
    if st != 0:
        raise LLError(fn, st)


def workspace_size(N, D, V, dtype, token_chunks=0, backward=False, need_db=False) -> int:
    code = dtype if isinstance(dtype, int) else _code(dtype)
    return int(load().ll_workspace_size(N, D, V, code, token_chunks, int(backward),
                                        int(bool(need_db))))


def _need(t, name, shape, dtype=None, device=None, dtypes=None):
    """Raise unless tensor t is contiguous, on `device`, of `shape` and dtype.

    The C ABI receives bare pointers, so every buffer it reads or writes is
    checked here, where the sizes are still known."""
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if dtypes is not None and t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype}, expected one of {dtypes}")
    if device is not None and t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")
    if t.numel() and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _check_linear(hidden, weight, bias, targets):
    torch = _torch()
    if hidden.dim() != 2 or weight.dim() != 2:
        raise ValueError("hidden and weight must be 2-D")
    N, D = hidden.shape
    V = weight.shape[0]
    dev = hidden.device
    _need(hidden, "hidden", (N, D), device=dev,
          dtypes=(torch.float32, torch.float16, torch.bfloat16))
    _need(weight, "weight", (V, D), hidden.dtype, dev)
    if bias is not None:
        _need(bias, "bias", (V,), hidden.dtype, dev)
    _need(targets, "targets", (N,), torch.int64, dev)
    return N, D, V, dev


def _workspace(nbytes, device):
    torch = _torch()
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def _grad_outputs(out, need_dh, need_dw, need_db, N, D, V, op_dtype, dh_dtype, dw_dtype, dev):
    """Gradient buffers (given or allocated) and their dtypes.  A given
    buffer's dtype decides; an explicit dtype that disagrees with it raises."""
    torch = _torch()
    if out is not None:
        dh, dW, db = out
        if dh is not None:
            if dh_dtype is not None and dh_dtype != dh.dtype:
                raise TypeError("dh_dtype disagrees with the given grad_hidden")
            dh_dtype = dh.dtype
        if dW is not None or db is not None:
            given = (dW if dW is not None else db).dtype
            if dw_dtype is not None and dw_dtype != given:
                raise TypeError("dw_dtype disagrees with the given grad_weight / grad_bias")
            dw_dtype = given
    dh_dtype = op_dtype if dh_dtype is None else dh_dtype
    dw_dtype = torch.float32 if dw_dtype is None else dw_dtype
    if out is None:
        dh = torch.empty(N, D, dtype=dh_dtype, device=dev) if need_dh else None
        dW = torch.empty(V, D, dtype=dw_dtype, device=dev) if need_dw else None
        db = torch.empty(V, dtype=dw_dtype, device=dev) if need_db else None
    if need_dh:
        _need(dh, "grad_hidden", (N, D), dh_dtype, dev)
    if need_dw:
        _need(dW, "grad_weight", (V, D), dw_dtype, dev)
    if need_db:
        _need(db, "grad_bias", (V,), dw_dtype, dev)
    return dh, dW, db, dh_dtype, dw_dtype


def forward(hidden, weight, bias, targets, *, temperature=1.0, workspace=None, out=None,
            stream=None):
    """(logp [N] fp32, lse [N] fp32) of z = hidden . weight^T (+ bias); with a
    temperature T the distribution is softmax(z / T)."""
    torch = _torch()
    L = load()
    N, D, V, dev = _check_linear(hidden, weight, bias, targets)
    code = _code(hidden.dtype)
    if out is None:
        logp = torch.empty(N, dtype=torch.float32, device=dev)
        lse = torch.empty(N, dtype=torch.float32, device=dev)
    else:
        logp, lse = out
    _need(logp, "logp", (N,), torch.float32, dev)
    _need(lse, "lse", (N,), torch.float32, dev)
    ws_need = L.ll_workspace_size(N, D, V, code, 0, 0, 0)
    if workspace is None:
        workspace = _workspace(ws_need, dev)
    _need(workspace, "workspace", (workspace.numel(),), torch.uint8, dev)
    st = L.ll_forward_ex(_ptr(hidden), _ptr(weight), _ptr(bias), _ptr(targets), N, D, V, code,
                         _ptr(logp), _ptr(lse), _ptr(workspace), workspace.numel(),
                         _opts(temperature), _stream(stream))
    _check("ll_forward", st)
    return logp, lse


def backward(grad_logp, hidden, weight, bias, targets, lse, *, need_dh=True, need_dw=True,
             need_db=None, dh_dtype=None, dw_dtype=None, token_chunks=0, temperature=1.0,
             split_s="auto", workspace=None, out=None, stream=None):
    """(grad_hidden, grad_weight, grad_bias); entries not requested are None.

    dw_dtype defaults to float32; grad_bias uses dw_dtype.
    """
    torch = _torch()
    L = load()
    N, D, V, dev = _check_linear(hidden, weight, bias, targets)
    code = _code(hidden.dtype)
    if need_db is None:
        need_db = bias is not None
    _need(grad_logp, "grad_logp", (N,), torch.float32, dev)
    _need(lse, "lse", (N,), torch.float32, dev)
    dh, dW, db, dh_dtype, dw_dtype = _grad_outputs(out, need_dh, need_dw, need_db, N, D, V,
                                                   hidden.dtype, dh_dtype, dw_dtype, dev)
    ws_need = L.ll_workspace_size(N, D, V, code, token_chunks, 1,
                                  int(bool(need_db)) | (_split_code(split_s) << 1))
    if workspace is None:
        workspace = _workspace(ws_need, dev)
    _need(workspace, "workspace", (workspace.numel(),), torch.uint8, dev)
    st = L.ll_backward_ex(_ptr(grad_logp), _ptr(hidden), _ptr(weight), _ptr(bias),
                          _ptr(targets), _ptr(lse), N, D, V, code, int(bool(need_dh)),
                          int(bool(need_dw)), int(bool(need_db)), _ptr(dh), _code(dh_dtype),
                          _ptr(dW), _code(dw_dtype), _ptr(db), int(token_chunks),
                          _ptr(workspace), workspace.numel(), _opts(temperature, split_s),
                          _stream(stream))
    _check("ll_backward", st)
    return dh, dW, db


def forward_backward(grad_logp, hidden, weight, bias, targets, *, need_dh=True, need_dw=True,
                     need_db=None, dh_dtype=None, dw_dtype=None, token_chunks=0,
                     temperature=1.0, split_s="auto", workspace=None, out=None, stream=None):
    """(logp, lse, grad_hidden, grad_weight, grad_bias) in one call, for a
    grad_logp known before the forward; bitwise equal to forward + backward."""
    torch = _torch()
    L = load()
    N, D, V, dev = _check_linear(hidden, weight, bias, targets)
    code = _code(hidden.dtype)
    if need_db is None:
        need_db = bias is not None
    _need(grad_logp, "grad_logp", (N,), torch.float32, dev)
    if out is not None:
        logp, lse, dh, dW, db = out
        grads = (dh, dW, db)
    else:
        logp = torch.empty(N, dtype=torch.float32, device=dev)
        lse = torch.empty(N, dtype=torch.float32, device=dev)
        grads = None
    _need(logp, "logp", (N,), torch.float32, dev)
    _need(lse, "lse", (N,), torch.float32, dev)
    dh, dW, db, dh_dtype, dw_dtype = _grad_outputs(grads, need_dh, need_dw, need_db, N, D, V,
                                                   hidden.dtype, dh_dtype, dw_dtype, dev)
    ws_need = L.ll_workspace_size(N, D, V, code, token_chunks, 2,
                                  int(bool(need_db)) | (_split_code(split_s) << 1))
    if workspace is None:
        workspace = _workspace(ws_need, dev)
    _need(workspace, "workspace", (workspace.numel(),), torch.uint8, dev)
    st = L.ll_forward_backward_ex(_ptr(grad_logp), _ptr(hidden), _ptr(weight), _ptr(bias),
                                  _ptr(targets), N, D, V, code, _ptr(logp), _ptr(lse),
                                  int(bool(need_dh)), int(bool(need_dw)), int(bool(need_db)),
                                  _ptr(dh), _code(dh_dtype), _ptr(dW), _code(dw_dtype),
                                  _ptr(db), int(token_chunks), _ptr(workspace),
                                  workspace.numel(), _opts(temperature, split_s),
                                  _stream(stream))
    _check("ll_forward_backward", st)
    return logp, lse, dh, dW, db


def logits_fwd(logits, targets, V=None, *, temperature=1.0, out=None, stream=None):
    """(logp, lse) from logits [N, ld]; columns >= V (default ld) ignored."""
    torch = _torch()
    L = load()
    N, ld = logits.shape
    V = ld if V is None else V
    dev = logits.device
    _need(logits, "logits", (N, ld), device=dev,
          dtypes=(torch.float32, torch.float16, torch.bfloat16))
    _need(targets, "targets", (N,), torch.int64, dev)
    if out is None:
        logp = torch.empty(N, dtype=torch.float32, device=dev)
        lse = torch.empty(N, dtype=torch.float32, device=dev)
    else:
        logp, lse = out
    _need(logp, "logp", (N,), torch.float32, dev)
    _need(lse, "lse", (N,), torch.float32, dev)
    st = L.logits_logp_fwd_ex(_ptr(logits), ld, _code(logits.dtype), _ptr(targets), N, V,
                              _ptr(logp), _ptr(lse), _opts(temperature), _stream(stream))
    _check("logits_logp_fwd", st)
    return logp, lse


def logits_bwd(grad_logp, logits, targets, lse, V=None, *, temperature=1.0, out=None,
               stream=None):
    """grad_logits [N, ld] in the logits dtype (columns [0, V) written)."""
    torch = _torch()
    L = load()
    N, ld = logits.shape
    V = ld if V is None else V
    dev = logits.device
    _need(logits, "logits", (N, ld), device=dev,
          dtypes=(torch.float32, torch.float16, torch.bfloat16))
    _need(targets, "targets", (N,), torch.int64, dev)
    _need(grad_logp, "grad_logp", (N,), torch.float32, dev)
    _need(lse, "lse", (N,), torch.float32, dev)
    if out is None:
        out = torch.empty_like(logits)
    _need(out, "grad_logits", (N, ld), logits.dtype, dev)
    st = L.logits_logp_bwd_ex(_ptr(grad_logp), _ptr(logits), ld, _code(logits.dtype),
                              _ptr(targets), _ptr(lse), N, V, _ptr(out), _opts(temperature),
                              _stream(stream))
    _check("logits_logp_bwd", st)
    return out


def launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return int(load().ll_launch_count())


def profile(enable: bool):
    """Start (clearing earlier records) or stop per-phase CUDA-event tracing."""
    load().ll_profile_enable(int(bool(enable)))


def profile_summary() -> dict:
    """{phase: (count, total_ms)} of the recorded phases (synchronises)."""
    buf = ctypes.create_string_buffer(8192)
    n = load().ll_profile_summary(buf, len(buf))
    if n < 0:
        raise LLError("ll_profile_summary", -n)
    out = {}
    for line in buf.value.decode().splitlines():
        name, cnt, ms = line.split()
        out[name] = (int(cnt), float(ms))
    return out


def logits_fwd_bwd(grad_logp, logits, targets, V=None, *, temperature=1.0, out=None,
                   stream=None):
    """(logp, lse, grad_logits) in one pass over the logits (grad_logp known
    before the forward)."""
    torch = _torch()
    L = load()
    N, ld = logits.shape
    V = ld if V is None else V
    dev = logits.device
    _need(logits, "logits", (N, ld), device=dev,
          dtypes=(torch.float32, torch.float16, torch.bfloat16))
    _need(targets, "targets", (N,), torch.int64, dev)
    _need(grad_logp, "grad_logp", (N,), torch.float32, dev)
    if out is None:
        logp = torch.empty(N, dtype=torch.float32, device=dev)
        lse = torch.empty(N, dtype=torch.float32, device=dev)
        g = torch.empty_like(logits)
    else:
        logp, lse, g = out
    _need(logp, "logp", (N,), torch.float32, dev)
    _need(lse, "lse", (N,), torch.float32, dev)
    _need(g, "grad_logits", (N, ld), logits.dtype, dev)
    st = L.logits_logp_fwd_bwd_ex(_ptr(grad_logp), _ptr(logits), ld, _code(logits.dtype),
                                  _ptr(targets), N, V, _ptr(logp), _ptr(lse), _ptr(g),
                                  _opts(temperature), _stream(stream))
    _check("logits_logp_fwd_bwd", st)
    return logp, lse, g


def sum_ordered(parts, out=None, stream=None):
    """out[i] = parts[0, i] + parts[1, i] + ... in ascending order (FP32
    accumulation, one rounding to the dtype): parts is a device tensor
    [nparts, n] (contiguous rows), out [n]."""
    torch = _torch()
    L = load()
    if parts.dim() != 2 or not parts.is_cuda or parts.stride(1) != 1:
        raise ValueError("parts must be a CUDA tensor [nparts, n] with contiguous rows")
    k, n = parts.shape
    if out is None:
        out = torch.empty(n, dtype=parts.dtype, device=parts.device)
    _need(out, "out", (n,), parts.dtype, parts.device)
    st = L.ll_sum_ordered(_ptr(parts), k, n, parts.stride(0), _code(parts.dtype), _ptr(out),
                          _stream(stream))
    _check("ll_sum_ordered", st)
    return out


def check_status(stream=None) -> int:
    """Synchronise and return (and clear) the device-side status word."""
    return int(load().ll_check_status(_stream(stream)))


# ---------------------------------------------------------- vocab shards

def shard_segments(Vs: int) -> int:
    """LSE segments of a vocab shard of Vs entries."""
    return int(load().ll_shard_segments(int(Vs)))


def forward_shard(hidden, weight, bias, targets, v0, V, *, temperature=1.0, workspace=None,
                  out=None, stream=None):
    """Segment partials of the vocab shard [v0, v0 + weight.shape[0]) of a
    vocab of V entries: (part_m, part_s) [shard_segments(Vs), N] and zy [N]
    (z of the target where it lies in the shard, -inf elsewhere).  targets
    are global ids."""
    torch = _torch()
    L = load()
    N, D, Vs, dev = _check_linear(hidden, weight, bias, targets)
    code = _code(hidden.dtype)
    S = shard_segments(Vs)
    if out is None:
        part_m = torch.empty(S, N, dtype=torch.float32, device=dev)
        part_s = torch.empty(S, N, dtype=torch.float32, device=dev)
        zy = torch.empty(N, dtype=torch.float32, device=dev)
    else:
        part_m, part_s, zy = out
    _need(part_m, "part_m", (S, N), torch.float32, dev)
    _need(part_s, "part_s", (S, N), torch.float32, dev)
    _need(zy, "zy", (N,), torch.float32, dev)
    if workspace is None:
        workspace = _workspace(L.ll_workspace_size_shard(N, D, Vs, code, 0, 0, 0), dev)
    _need(workspace, "workspace", (workspace.numel(),), torch.uint8, dev)
    st = L.ll_forward_shard(_ptr(hidden), _ptr(weight), _ptr(bias), _ptr(targets), N, D, Vs,
                            int(v0), int(V), code, _ptr(part_m), _ptr(part_s), _ptr(zy),
                            _ptr(workspace), workspace.numel(), _opts(temperature),
                            _stream(stream))
    _check("ll_forward_shard", st)
    return part_m, part_s, zy


def lse_merge(part_m, part_s, zy, targets, V, *, out=None, stream=None):
    """(logp, lse) from whole-vocab segment partials [n_segs, N] in ascending
    segment order (rows of m = -inf, s = 0 change nothing)."""
    torch = _torch()
    L = load()
    if part_m.dim() != 2:
        raise ValueError("part_m must be 2-D [n_segs, N]")
    n_segs, N = part_m.shape
    dev = part_m.device
    _need(part_m, "part_m", (n_segs, N), torch.float32, dev)
    _need(part_s, "part_s", (n_segs, N), torch.float32, dev)
    _need(zy, "zy", (N,), torch.float32, dev)
    _need(targets, "targets", (N,), torch.int64, dev)
    if out is None:
        logp = torch.empty(N, dtype=torch.float32, device=dev)
        lse = torch.empty(N, dtype=torch.float32, device=dev)
    else:
        logp, lse = out
    _need(logp, "logp", (N,), torch.float32, dev)
    _need(lse, "lse", (N,), torch.float32, dev)
    st = L.ll_lse_merge(_ptr(part_m), _ptr(part_s), n_segs, N, _ptr(zy), _ptr(targets), N,
                        int(V), _ptr(logp), _ptr(lse), _stream(stream))
    _check("ll_lse_merge", st)
    return logp, lse


def backward_shard(grad_logp, hidden, weight, bias, targets, lse, v0, V, *, need_dh=True,
                   need_dw=True, need_db=None, dh_dtype=None, dw_dtype=None, token_chunks=0,
                   temperature=1.0, split_s="auto", workspace=None, out=None, stream=None):
    """(grad_hidden part, grad_weight rows, grad_bias rows) of the vocab shard
    [v0, v0 + weight.shape[0]); lse is the merged whole-vocab lse.  The
    grad_hidden part defaults to float32 (the shards' parts are summed)."""
    torch = _torch()
    L = load()
    N, D, Vs, dev = _check_linear(hidden, weight, bias, targets)
    code = _code(hidden.dtype)
    if need_db is None:
        need_db = bias is not None
    if dh_dtype is None and (out is None or out[0] is None):
        dh_dtype = torch.float32
    _need(grad_logp, "grad_logp", (N,), torch.float32, dev)
    _need(lse, "lse", (N,), torch.float32, dev)
    dh, dW, db, dh_dtype, dw_dtype = _grad_outputs(out, need_dh, need_dw, need_db, N, D, Vs,
                                                   hidden.dtype, dh_dtype, dw_dtype, dev)
    if workspace is None:
        workspace = _workspace(L.ll_workspace_size_shard(
            N, D, Vs, code, token_chunks, 1, int(bool(need_db)) | (_split_code(split_s) << 1)), dev)
    _need(workspace, "workspace", (workspace.numel(),), torch.uint8, dev)
    st = L.ll_backward_shard(_ptr(grad_logp), _ptr(hidden), _ptr(weight), _ptr(bias),
                             _ptr(targets), _ptr(lse), N, D, Vs, int(v0), int(V), code,
                             int(bool(need_dh)), int(bool(need_dw)), int(bool(need_db)),
                             _ptr(dh), _code(dh_dtype), _ptr(dW), _code(dw_dtype), _ptr(db),
                             int(token_chunks), _ptr(workspace), workspace.numel(),
                             _opts(temperature, split_s), _stream(stream))
    _check("ll_backward_shard", st)
    return dh, dW, db
