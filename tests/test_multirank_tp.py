"""Vocab-parallel composition with CPU ranks (gloo): the host logic of
cross_entropy_rl_gb300.tp (shard bounds on segment boundaries, the padded
all-gather of the segment partials, the MAX all-reduce of the target logit,
the ordered merge, the fixed-order grad_hidden sum) with an FP64 oracle
stand-in for the three per-shard calls.  The composed logp / lse are
bitwise those of merging every segment in one process, for 1-4 ranks,
including a rank with an empty shard; the gradients match the oracle."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from cross_entropy_rl_gb300 import synth, tp

LOG2E = 1.0 / np.log(2.0)


class OracleShards:
    """The per-shard calls of the C ABI, in FP64 from the oracle's logits,
    with the ABI's semantics (partials per 1024-column segment, -inf zy
    outside the shard, ascending-order merge)."""

    def forward_shard(self, hidden, weight, bias, targets, v0, V, out, temperature=1.0):
        import oracle

        part_m, part_s, zy = out
        h = hidden.double().numpy()
        W = weight.double().numpy()
        b = None if bias is None else bias.double().numpy()
        z = oracle.linear_logits(h, W, b) / temperature * LOG2E
        Vs = W.shape[0]
        for j in range(-(-Vs // tp.SEGMENT_COLS)):
            seg = z[:, j * tp.SEGMENT_COLS:(j + 1) * tp.SEGMENT_COLS]
            m = seg.max(axis=1)
            part_m[j] = torch.from_numpy(m)
            part_s[j] = torch.from_numpy(np.exp2(seg - m[:, None]).sum(axis=1))
        y = targets.numpy()
        mine = (y >= v0) & (y < v0 + Vs)
        zl = np.full(len(y), -np.inf)
        zl[mine] = z[np.nonzero(mine)[0], y[mine] - v0] / LOG2E
        zy.copy_(torch.from_numpy(zl))

    def lse_merge(self, part_m, part_s, zy, targets, V):
        m = part_m.double().numpy()
        s = part_s.double().numpy()
        M = m.max(axis=0)
        S = np.zeros(m.shape[1])
        for j in range(m.shape[0]):  # ascending segment order
            S = S + s[j] * np.exp2(m[j] - M)
        lse = (M + np.log2(S)) / LOG2E
        y = targets.numpy()
        ok = (y >= 0) & (y < V)
        logp = np.where(ok, zy.double().numpy() - lse, 0.0)
        return torch.from_numpy(logp), torch.from_numpy(lse)

    def backward_shard(self, grad_logp, hidden, weight, bias, targets, lse, v0, V, need_db,
                       token_chunks, temperature=1.0):
        import oracle

        h = hidden.double().numpy()
        W = weight.double().numpy()
        b = None if bias is None else bias.double().numpy()
        z = oracle.linear_logits(h, W, b) / temperature
        p = np.exp(z - lse.double().numpy()[:, None])
        y = targets.numpy()
        gl = grad_logp.double().numpy()
        Vs = W.shape[0]
        onehot = np.zeros_like(p)
        mine = np.nonzero((y >= v0) & (y < v0 + Vs))[0]
        onehot[mine, y[mine] - v0] = 1.0
        g = gl[:, None] * (onehot - p) / temperature
        g[(y < 0) | (y >= V)] = 0.0
        db = torch.from_numpy(g.sum(axis=0)) if need_db else None
        return torch.from_numpy(g @ W), torch.from_numpy(g.T @ h), db


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


N, D, V = 23, 8, 2500


def _inputs():
    p = synth.linear_inputs(N, D, V, dtype="f32", bias=True, seed=11)
    y = p["y"].copy()
    y[[1, 2, 3]] = [5, 2100, 2499]  # a target in every segment
    y[4] = -100
    return p, y


def _worker(rank, world, port, out_dir, T=1.0):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=__import__("datetime").timedelta(seconds=30))
    try:
        p, y = _inputs()
        h = torch.from_numpy(p["h"])
        W = torch.from_numpy(p["W"])
        b = torch.from_numpy(p["b"])
        yt = torch.from_numpy(y)
        gl = torch.from_numpy(p["gl"])
        v0, v1 = tp.shard_bounds(V, world)[rank]
        impl = OracleShards()
        logp, lse = tp.forward(h, W[v0:v1], b[v0:v1], yt, v0, V, impl=impl, temperature=T)
        dh, dW, db = tp.backward(gl, h, W[v0:v1], b[v0:v1], yt, lse.float(), v0, V, impl=impl,
                                 temperature=T)
        np.save(os.path.join(out_dir, f"logp{rank}.npy"), logp.numpy())
        np.save(os.path.join(out_dir, f"lse{rank}.npy"), lse.numpy())
        np.save(os.path.join(out_dir, f"dh{rank}.npy"), dh.numpy())
        np.save(os.path.join(out_dir, f"dW{rank}.npy"), dW.numpy())
        np.save(os.path.join(out_dir, f"db{rank}.npy"), db.numpy())
    finally:
        dist.destroy_process_group()


def test_shard_bounds_are_whole_segments():
    for V_ in (1, 1023, 1024, 1025, 5000, 151936):
        for world in (1, 2, 3, 4, 8, 200):
            b = tp.shard_bounds(V_, world)
            assert len(b) == world and b[0][0] == 0 and b[-1][1] == V_
            for (a0, a1), (c0, c1) in zip(b, b[1:]):
                assert a1 == c0
            for v0, v1 in b:
                assert v0 % tp.SEGMENT_COLS == 0 or v0 == v1 == V_  # empty shards at the end
                assert v1 == V_ or v1 % tp.SEGMENT_COLS == 0
            sizes = [-(-(v1 - v0) // tp.SEGMENT_COLS) for v0, v1 in b]
            assert max(sizes) - min(sizes) <= 1 and max(sizes) == tp.max_segments(V_, world)


def _single_process_merge(T=1.0):
    """Every segment's partial in one process, merged: the reference bits."""
    p, y = _inputs()
    impl = OracleShards()
    S = -(-V // tp.SEGMENT_COLS)
    m = torch.empty(S, N, dtype=torch.float32)
    s = torch.empty(S, N, dtype=torch.float32)
    zy = torch.empty(N, dtype=torch.float32)
    impl.forward_shard(torch.from_numpy(p["h"]), torch.from_numpy(p["W"]),
                       torch.from_numpy(p["b"]), torch.from_numpy(y), 0, V, out=(m, s, zy),
                       temperature=T)
    return impl.lse_merge(m, s, zy, torch.from_numpy(y), V)


@pytest.mark.parametrize("world,T", [(2, 1.0), (3, 1.0), (4, 1.0), (3, 0.7)])
def test_vocab_parallel_composition(tmp_path, world, T):
    import oracle

    port = _free_port()
    mp.start_processes(_worker, args=(world, port, str(tmp_path), T), nprocs=world, join=True,
                       start_method="spawn")
    p, y = _inputs()
    logp1, lse1 = _single_process_merge(T)
    full = oracle.linear_forward_backward(p["gl"], p["h"], p["W"], p["b"], y, "f32",
                                          temperature=T)
    ld = lambda k, r: np.load(tmp_path / f"{k}{r}.npy")
    for r in range(world):
        # bitwise the one-process merge of all segments, on every rank
        assert np.array_equal(ld("logp", r), logp1.numpy())
        assert np.array_equal(ld("lse", r), lse1.numpy())
        assert np.array_equal(ld("dh", r), ld("dh", 0))
    np.testing.assert_allclose(ld("lse", 0), full["lse"], rtol=0, atol=1e-5)
    np.testing.assert_allclose(ld("logp", 0), full["logp"], rtol=0, atol=1e-5)
    np.testing.assert_allclose(ld("dh", 0), full["dh"], rtol=1e-5, atol=1e-6)
    dW = np.concatenate([ld("dW", r) for r in range(world)])
    db = np.concatenate([ld("db", r) for r in range(world)])
    np.testing.assert_allclose(dW, full["dW"], rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(db, full["db"], rtol=1e-5, atol=1e-6)
