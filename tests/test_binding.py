"""The binding checks every buffer before the C ABI sees a pointer: the ABI
takes bare pointers, so a wrong dtype, shape or layout would make a kernel
write or read past a buffer.  These run on the CPU (host tensors): the checks
fire before any CUDA call, and host memory itself is refused by the ABI."""
import pytest
import torch

import cross_entropy_rl_gb300 as ll
from cross_entropy_rl_gb300 import build as B


@pytest.fixture(scope="module", autouse=True)
def _built():
    B.build()
    ll.load()


def _inputs(N=8, D=16, V=40, dtype=torch.bfloat16):
    h = torch.zeros(N, D, dtype=dtype)
    W = torch.zeros(V, D, dtype=dtype)
    b = torch.zeros(V, dtype=dtype)
    y = torch.zeros(N, dtype=torch.int64)
    g = torch.zeros(N, dtype=torch.float32)
    lse = torch.zeros(N, dtype=torch.float32)
    return h, W, b, y, g, lse


def test_forward_rejects_bad_buffers():
    h, W, b, y, g, lse = _inputs()
    with pytest.raises(ValueError, match="targets"):
        ll.forward(h, W, b, y[:-1])
    with pytest.raises(TypeError, match="targets"):
        ll.forward(h, W, b, y.to(torch.int32))
    with pytest.raises(TypeError, match="weight"):
        ll.forward(h, W.float(), b, y)
    with pytest.raises(ValueError, match="bias"):
        ll.forward(h, W, b[:-1], y)
    with pytest.raises(ValueError, match="contiguous"):
        ll.forward(torch.zeros(16, 8, dtype=torch.bfloat16).t(), W, b, y)
    with pytest.raises(ValueError, match="logp"):
        ll.forward(h, W, b, y, out=(torch.zeros(7), torch.zeros(8)))


def test_backward_takes_output_dtypes_from_given_buffers():
    h, W, b, y, g, lse = _inputs()
    dh = torch.zeros(8, 16, dtype=torch.bfloat16)
    dW16 = torch.zeros(40, 16, dtype=torch.bfloat16)
    db16 = torch.zeros(40, dtype=torch.bfloat16)
    # an explicit dtype that disagrees with the given grad_weight is refused
    with pytest.raises(TypeError, match="dw_dtype"):
        ll.backward(g, h, W, b, y, lse, out=(dh, dW16, db16), dw_dtype=torch.float32)
    with pytest.raises(ValueError, match="grad_weight"):
        ll.backward(g, h, W, b, y, lse, out=(dh, dW16[:-1], db16))
    with pytest.raises(TypeError, match="grad_bias"):
        ll.backward(g, h, W, b, y, lse, out=(dh, dW16, db16.float()))
    with pytest.raises(ValueError, match="grad_logp"):
        ll.backward(g[:-1], h, W, b, y, lse)
    # consistent buffers on host memory reach the ABI, which refuses host pointers
    with pytest.raises(ll.LLError, match="status 1"):
        ll.backward(g, h, W, b, y, lse, out=(dh, dW16, db16))


def test_forward_backward_and_logits_checks():
    h, W, b, y, g, lse = _inputs()
    with pytest.raises(ValueError, match="grad_logp"):
        ll.forward_backward(g[:3], h, W, b, y)
    x = torch.zeros(8, 40, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="targets"):
        ll.logits_fwd(x, y[:4])
    with pytest.raises(TypeError, match="grad_logits"):
        ll.logits_bwd(g, x, y, lse, out=torch.zeros(8, 40))
    with pytest.raises(ll.LLError, match="status 1"):
        ll.logits_fwd(x, y)
