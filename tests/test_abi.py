"""The C-ABI library loads, exports every declared symbol, and validates its
arguments on the host (no GPU needed: every case here returns before the
first CUDA call)."""
import ctypes
import os
import re

import pytest

import cross_entropy_rl_gb300 as ll
from cross_entropy_rl_gb300 import build as B

HEADER = os.path.join(B.ROOT, "include", "ll_linear_logp.h")


@pytest.fixture(scope="module")
def L():
    B.build()
    return ll.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_abi():
    names = declared_functions()
    for must in ("ll_forward", "ll_backward", "logits_logp_fwd", "logits_logp_bwd",
                 "ll_workspace_size", "ll_check_status", "ll_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
        assert name in ll.EXPORTS, f"binding does not marshal {name}"


def test_version_and_status_strings(L):
    assert L.ll_version() >= 100
    assert L.ll_status_string(0) == b"ok"
    assert L.ll_status_string(4).startswith(b"misaligned")
    assert L.ll_status_string(999) == b"unknown status"


def test_workspace_size_rules(L):
    # forward: two FP32 partials per (segment, row) + target logit per row
    N, V = 4096, 32768
    n_segs = -(-(-(-V // 256)) // 4)
    fwd = L.ll_workspace_size(N, 2048, V, ll.LL_BF16, 0, 0, 0)
    assert fwd >= (2 * n_segs + 1) * N * 4
    assert L.ll_workspace_size(0, 2048, V, ll.LL_BF16, 0, 0, 0) == 0
    assert fwd < N * V  # partials only: not the logits
    # a small forward (few 128-row x 1024-column blocks) also keeps its FP32
    # logits, N x round_up(V, 8), for the second kernel that folds them
    small = L.ll_workspace_size(128, 256, 4096, ll.LL_F32, 0, 0, 0)
    assert 128 * 4096 * 4 <= small <= 128 * 4096 * 4 + 64 * 1024
    assert L.ll_workspace_size(2, 64, 3001, ll.LL_BF16, 0, 0, 0) >= 2 * 3008 * 4
    big_v = L.ll_workspace_size(128, 256, 300000, ll.LL_F32, 0, 0, 0)  # logits > 4 MiB
    assert big_v < 128 * 300000 * 4
    # backward, one chunk: [N, round_up(V, 8)] 16-bit softmax part
    bwd1 = L.ll_workspace_size(N, 2048, V, ll.LL_BF16, 1, 1, 0)
    assert bwd1 >= N * V * 2
    bwd8 = L.ll_workspace_size(N, 2048, V, ll.LL_BF16, 8, 1, 0)
    assert bwd8 < bwd1 and bwd8 >= (N // 8) * V * 2
    # automatic chunking keeps the softmax part within 2 GiB (split_s =
    # never: S alone, plus the transposed hidden states h^T of 16-bit
    # operands); the default automatic split adds one S-sized buffer and its
    # small piece flags and plan
    hT = 4096 * 6656 * 2  # one chunk's h^T (5 chunks of 6656 rows)
    big = L.ll_workspace_size(32768, 4096, 151936, ll.LL_BF16, 0, 1, 2 << 1)
    assert hT <= big <= (2 << 30) + hT + (64 << 20)
    auto = L.ll_workspace_size(32768, 4096, 151936, ll.LL_BF16, 0, 1, 0)
    always = L.ll_workspace_size(32768, 4096, 151936, ll.LL_BF16, 0, 1, 1 << 1)
    s_only = big - hT
    assert 2 * s_only - (64 << 20) <= always - hT <= auto - hT <= 2 * s_only + (64 << 20)
    assert L.ll_workspace_size(32768, 4096, 151936, ll.LL_BF16, 0, 1, 3 << 1) == 0
    # FP32 keeps S in FP32: the split mode changes nothing
    f = [L.ll_workspace_size(4096, 2048, 32768, ll.LL_F32, 1, 1, m << 1) for m in range(3)]
    assert f[0] == f[1] == f[2]
    assert L.ll_workspace_size(N, 2048, V, ll.LL_F32, 1, 1, 0) >= N * V * 4
    # FP32 grad_hidden over D <= 512 is cut along K = V into min(16, ceil(V / 16) / 16)
    # parts whose FP32 partial sums take [parts, round_up(N, 128), D] of the workspace
    # (FP32 also keeps K-major copies W^T [D, round_up(V, 4)], h^T and S^T of
    # the chunk, so the wider D and the larger V add a little of those)
    narrow = L.ll_workspace_size(128, 512, 4096, ll.LL_F32, 1, 1, 0)
    wide = L.ll_workspace_size(128, 520, 4096, ll.LL_F32, 1, 1, 0)
    parts = 16 * 128 * 512 * 4
    assert parts - 256 * 1024 <= narrow - wide <= parts
    two = L.ll_workspace_size(100, 512, 520, ll.LL_F32, 1, 1, 0)  # ceil(520/16)/16 = 2 parts
    one = L.ll_workspace_size(100, 512, 496, ll.LL_F32, 1, 1, 0)  # ceil(496/16) = 31: one part
    assert 2 * 128 * 512 * 4 <= two - one <= 2 * 128 * 512 * 4 + 128 * 1024
    # FP32: W^T, S^T and h^T of one chunk on top of S
    N1, D1, V1 = 4096, 1024, 32768
    f32 = L.ll_workspace_size(N1, D1, V1, ll.LL_F32, 1, 1, 0)
    assert f32 >= (2 * N1 * V1 + D1 * V1 + D1 * N1) * 4
    # grad_bias partials only when requested
    assert L.ll_workspace_size(N, 2048, V, ll.LL_BF16, 1, 1, 1) > bwd1


NULL = None


def fwd(L, **kw):
    a = dict(hidden=16, weight=32, bias=NULL, targets=48, N=4, D=8, V=10, dtype=ll.LL_BF16,
             logp=64, lse=80, ws=256, ws_bytes=1 << 20)
    a.update(kw)
    p = lambda x: None if x is None else ctypes.c_void_p(x)
    return L.ll_forward(p(a["hidden"]), p(a["weight"]), p(a["bias"]), p(a["targets"]), a["N"],
                        a["D"], a["V"], a["dtype"], p(a["logp"]), p(a["lse"]), p(a["ws"]),
                        a["ws_bytes"], None)


def test_forward_validation_before_launch(L):
    assert fwd(L, N=-1) == 3
    assert fwd(L, V=0) == 3
    assert fwd(L, D=0) == 3
    assert fwd(L, V=(1 << 31)) == 3
    assert fwd(L, dtype=7) == 2
    assert fwd(L, weight=None) == 1
    assert fwd(L, N=0) == 0              # empty batch: nothing to do
    assert fwd(L, hidden=None) == 1
    assert fwd(L, D=12) == 4             # rows not 16-byte multiples
    assert fwd(L, hidden=24) == 4        # misaligned pointer
    assert fwd(L, ws=None) == 5
    assert fwd(L, ws_bytes=8) == 5
    assert fwd(L, ws=264) == 5           # workspace not 256-byte aligned


def bwd(L, **kw):
    a = dict(grad=8, hidden=16, weight=32, bias=NULL, targets=48, lse=64, N=4, D=8, V=10,
             dtype=ll.LL_BF16, dh=1, dw=1, db=0, dh_ptr=256, dh_dt=ll.LL_BF16, dw_ptr=512,
             dw_dt=ll.LL_F32, db_ptr=None, chunks=0, ws=1024, ws_bytes=1 << 20)
    a.update(kw)
    p = lambda x: None if x is None else ctypes.c_void_p(x)
    return L.ll_backward(p(a["grad"]), p(a["hidden"]), p(a["weight"]), p(a["bias"]),
                         p(a["targets"]), p(a["lse"]), a["N"], a["D"], a["V"], a["dtype"],
                         a["dh"], a["dw"], a["db"], p(a["dh_ptr"]), a["dh_dt"], p(a["dw_ptr"]),
                         a["dw_dt"], p(a["db_ptr"]), a["chunks"], p(a["ws"]), a["ws_bytes"], None)


def test_backward_validation_before_launch(L):
    assert bwd(L, N=-3) == 3
    assert bwd(L, dtype=5) == 2
    assert bwd(L, dh=2) == 1
    assert bwd(L, chunks=-1) == 1
    assert bwd(L, dh_dt=ll.LL_F16) == 2           # dh must be the operand dtype or FP32
    assert bwd(L, dw_dt=ll.LL_F16) == 2           # dW must be FP32 or the operand dtype
    assert bwd(L, dw_ptr=None) == 1
    assert bwd(L, db=1, db_ptr=None) == 1
    assert bwd(L, D=20) == 4
    assert bwd(L, dw_ptr=520) == 4
    assert bwd(L, dh=0, dw=0, db=0) == 0          # nothing requested: nothing to do


def logits(L, fn, **kw):
    a = dict(grad=8, logits=16, ld=10, dtype=ll.LL_BF16, targets=32, lse=48, N=4, V=10,
             logp=64, out=4096)
    a.update(kw)
    p = lambda x: None if x is None else ctypes.c_void_p(x)
    if fn == "fwd":
        return L.logits_logp_fwd(p(a["logits"]), a["ld"], a["dtype"], p(a["targets"]), a["N"],
                                 a["V"], p(a["logp"]), p(a["lse"]), None)
    return L.logits_logp_bwd(p(a["grad"]), p(a["logits"]), a["ld"], a["dtype"], p(a["targets"]),
                             p(a["lse"]), a["N"], a["V"], p(a["out"]), None)


def test_logits_validation_before_launch(L):
    assert logits(L, "fwd", ld=5) == 3            # ld < V
    assert logits(L, "fwd", dtype=9) == 2
    assert logits(L, "fwd", N=0) == 0
    assert logits(L, "fwd", targets=None) == 1
    assert logits(L, "fwd", logits=17) == 4       # not element aligned
    assert logits(L, "bwd", out=20) == 1          # output overlaps the logits
    assert logits(L, "bwd", grad=None) == 1


def test_binding_fails_loudly_without_library(tmp_path):
    import importlib

    mod = importlib.reload(ll)
    try:
        mod._LIB = None
        with pytest.raises(RuntimeError, match="not built"):
            mod.load(str(tmp_path / "missing.so"))
    finally:
        importlib.reload(ll)


def test_options_are_validated_before_any_device_work(L):
    """A bad temperature or a non-zero reserved field is LL_ERR_INVALID_ARG,
    returned before any pointer is touched (all pointers here are NULL)."""
    for T in (0.0, -1.0, float("inf"), float("nan")):
        o = ll.Options(temperature=T)
        assert L.ll_forward_ex(None, None, None, None, 4, 8, 16, ll.LL_BF16, None, None, None,
                               0, ctypes.byref(o), None) == 1
        assert L.logits_logp_fwd_ex(None, 16, ll.LL_BF16, None, 4, 16, None, None,
                                    ctypes.byref(o), None) == 1
    o = ll.Options(temperature=1.0)
    o.reserved[3] = 7
    assert L.ll_backward_ex(None, None, None, None, None, None, 4, 8, 16, ll.LL_BF16, 1, 1, 0,
                            None, ll.LL_BF16, None, ll.LL_F32, None, 0, None, 0,
                            ctypes.byref(o), None) == 1
    for bad in (-1, 3):  # split_s is 0 (automatic), 1 (always) or 2 (never)
        o = ll.Options(temperature=1.0, split_s=bad)
        assert L.ll_backward_ex(None, None, None, None, None, None, 4, 8, 16, ll.LL_BF16, 1, 1,
                                0, None, ll.LL_BF16, None, ll.LL_F32, None, 0, None, 0,
                                ctypes.byref(o), None) == 1
    with pytest.raises(ValueError, match="temperature"):
        ll._opts(-2.0)
    # binding: the default is the automatic split (no options struct at all)
    assert ll._opts(1.0) is None and ll._opts(1.0, "auto") is None
    assert ll._split_code(True) == 1 and ll._split_code("always") == 1
    assert ll._split_code(False) == 2 and ll._split_code("never") == 2
    with pytest.raises(ValueError, match="split_s"):
        ll._split_code("sometimes")


C_PROGRAM = r"""
#include <stdio.h>
#include "ll_linear_logp.h"
int main(void) {
    /* host-only entry points: no device needed */
    size_t ws = ll_workspace_size(4096, 2048, 32768, LL_BF16, 0, 1, 0);
    ll_options opt = {1.0f, 0, {0, 0, 0, 0, 0, 0}};
    (void)opt;
    printf("%d %zu %s\n", ll_version(), ws, ll_status_string(LL_ERR_ALIGN));
    return ws == 0;
}
"""


def test_header_is_plain_c_and_links(L, tmp_path):
    """The header compiles as C99 (no C++ or torch types) and a C program
    links against the shared library and calls its host-only entry points."""
    import shutil
    import subprocess

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "use_abi"
    lib_dir = os.path.dirname(B.LIB_PATH)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER),
                        str(src), "-o", str(exe), "-L", lib_dir,
                        "-l:" + os.path.basename(B.LIB_PATH), "-Wl,-rpath," + lib_dir],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    version, ws, name = r.stdout.split(maxsplit=2)
    assert int(version) == L.ll_version()
    assert int(ws) == L.ll_workspace_size(4096, 2048, 32768, ll.LL_BF16, 0, 1, 0)
    assert name.strip() != ""
