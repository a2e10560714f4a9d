"""The C ABI on user streams and inside CUDA graphs: calls in flight on two
streams at once, and fwd + bwd (and the single call) captured once and
replayed on new inputs, give bitwise the results of plain calls."""
import pytest
import torch

from cross_entropy_rl_gb300 import synth
from gpu_util import bits_equal, dev

pytestmark = pytest.mark.gpu


def _inputs(N, D, V, dt, seed, bias=True):
    p = synth.linear_inputs(N, D, V, dtype=dt, bias=bias, seed=seed)
    return [dev(p["h"], dt), dev(p["W"], dt), dev(p["b"], dt), dev(p["y"]), dev(p["gl"])]


def _plain(lib, h, W, b, y, g, chunks=0):
    logp, lse = lib.forward(h, W, b, y)
    dh, dW, db = lib.backward(g, h, W, b, y, lse, token_chunks=chunks)
    torch.cuda.synchronize()
    assert lib.check_status() == 0
    return [logp, lse, dh, dW, db]


def test_two_streams_in_flight(lib):
    A = _inputs(700, 136, 3000, "bf16", 1)
    B = _inputs(1100, 72, 2053, "f16", 2)
    ref_a = _plain(lib, *A)
    ref_b = _plain(lib, *B, chunks=2)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s1):
        la, lsa = lib.forward(*A[:4])
    with torch.cuda.stream(s2):
        lb, lsb = lib.forward(*B[:4])
    with torch.cuda.stream(s1):
        ga = lib.backward(A[4], *A[:4], lsa)
    with torch.cuda.stream(s2):
        gb = lib.backward(B[4], *B[:4], lsb, token_chunks=2)
    torch.cuda.synchronize()
    assert lib.check_status() == 0
    for got, ref in (([la, lsa, *ga], ref_a), ([lb, lsb, *gb], ref_b)):
        for i, (x, r) in enumerate(zip(got, ref)):
            assert bits_equal(x, r), i


@pytest.mark.parametrize("single", [False, True])
def test_cuda_graph_capture_and_replay(lib, single):
    N, D, V = 1000, 128, 4099
    h, W, b, y, g = _inputs(N, D, V, "bf16", 3)
    logp = torch.empty(N, device="cuda")
    lse = torch.empty_like(logp)
    dh = torch.empty_like(h)
    dW = torch.empty(V, D, device="cuda")
    db = torch.empty(V, device="cuda")
    mode = 2 if single else 1
    L = lib.load()
    ws_f = torch.empty(max(256, lib.workspace_size(N, D, V, torch.bfloat16)), dtype=torch.uint8,
                       device="cuda")
    ws_b = torch.empty(max(256, L.ll_workspace_size(N, D, V, 2, 0, mode, 1)), dtype=torch.uint8,
                       device="cuda")

    def step():
        if single:
            lib.forward_backward(g, h, W, b, y, workspace=ws_b, out=(logp, lse, dh, dW, db))
        else:
            lib.forward(h, W, b, y, workspace=ws_f, out=(logp, lse))
            lib.backward(g, h, W, b, y, lse, workspace=ws_b, out=(dh, dW, db))

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # first use outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    new = _inputs(N, D, V, "bf16", 4)
    for dst, src in zip((h, W, b, y, g), new):
        dst.copy_(src)
    graph.replay()
    torch.cuda.synchronize()
    assert lib.check_status() == 0
    ref = _plain(lib, *new)
    for i, (x, r) in enumerate(zip([logp, lse, dh, dW, db], ref)):
        assert bits_equal(x, r), i
