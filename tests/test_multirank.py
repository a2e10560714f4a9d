"""Token-sharded data parallelism with CPU ranks (gloo, world_size 2 and 3):
per-rank shards through the FP64 oracle, the fixed-order grad_weight /
grad_bias reduction (a reduce-scatter by all-to-all, each slice summed in
ascending rank order by its owner, then an all-gather) reproduces the
single-process gradients and is bitwise identical on every rank; a rank that
fails is seen by the others as an error, not a hang."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from cross_entropy_rl_gb300 import dp, synth


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_dir, fail_rank):
    import oracle

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=__import__("datetime").timedelta(seconds=20))
    try:
        p = synth.linear_inputs(37, 16, 50, dtype="f32", bias=True, seed=3)
        b, e = dp.shard_rows(p["N"], world, rank)
        if rank == fail_rank:
            raise RuntimeError("injected rank failure")
        rows = np.arange(b, e)
        r = oracle.linear_rows(p["gl"], p["h"], p["W"], p["b"], p["y"], "f32", rows)
        dW = dp.reduce_sum_fixed_order(torch.from_numpy(r["dW"]))
        db = dp.reduce_sum_fixed_order(torch.from_numpy(r["db"]))
        np.save(os.path.join(out_dir, f"dW{rank}.npy"), dW.numpy())
        np.save(os.path.join(out_dir, f"db{rank}.npy"), db.numpy())
        np.save(os.path.join(out_dir, f"logp{rank}.npy"), r["logp"])
    finally:
        dist.destroy_process_group()


def _rs_worker(rank, world, port, out_dir, numel):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=__import__("datetime").timedelta(seconds=20))
    try:
        g = torch.Generator().manual_seed(100 + rank)
        t = torch.randn(numel, generator=g, dtype=torch.float32)
        mine = dp.reduce_scatter_fixed_order(t)
        full = dp.reduce_sum_fixed_order(t.view(-1, 1))
        np.save(os.path.join(out_dir, f"slice{rank}.npy"), mine.numpy())
        np.save(os.path.join(out_dir, f"full{rank}.npy"), full.view(-1).numpy())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,numel", [(2, 1000), (3, 1001), (3, 2)])
def test_reduce_scatter_fixed_order(tmp_path, world, numel):
    """Each rank's slice is the ascending-rank FP32 sum of that slice of
    every rank's table (bitwise); the all-gathered sum is the same bits on
    every rank, shape kept."""
    port = _free_port()
    mp.start_processes(_rs_worker, args=(world, port, str(tmp_path), numel), nprocs=world,
                       join=True, start_method="spawn")
    ts = [torch.randn(numel, generator=torch.Generator().manual_seed(100 + r),
                      dtype=torch.float32) for r in range(world)]
    want = ts[0].clone()
    for t in ts[1:]:
        want += t
    for r in range(world):
        b, e = dp.shard_rows(numel, world, r)
        got = np.load(tmp_path / f"slice{r}.npy")
        assert np.array_equal(got, want[b:e].numpy()), r
        assert np.array_equal(np.load(tmp_path / f"full{r}.npy"), want.numpy()), r


def test_exchange_bytes_per_rank():
    """(world - 1) / world of the table leaves and enters each rank."""
    d = dp.slice_bytes(151936 * 4096, 4, 8)
    table = 151936 * 4096 * 4
    assert d["reduce_scatter_send"] == table - table // 8
    assert d["reduce_scatter_recv"] == table - table // 8
    assert dp.slice_bytes(100, 4, 1)["reduce_scatter_send"] == 0


def test_shard_rows_cover_exactly_once():
    for N in (0, 1, 7, 37, 4096):
        for world in (1, 2, 3, 8):
            spans = [dp.shard_rows(N, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == N
            for (b0, e0), (b1, e1) in zip(spans, spans[1:]):
                assert e0 == b1
            sizes = [e - b for b, e in spans]
            assert max(sizes) - min(sizes) <= 1


def test_two_rank_reduction_matches_single_process(tmp_path):
    import oracle

    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path), -1), nprocs=2, join=True,
                       start_method="spawn")
    p = synth.linear_inputs(37, 16, 50, dtype="f32", bias=True, seed=3)
    full = oracle.linear_forward_backward(p["gl"], p["h"], p["W"], p["b"], p["y"], "f32")
    dW0, dW1 = np.load(tmp_path / "dW0.npy"), np.load(tmp_path / "dW1.npy")
    assert np.array_equal(dW0, dW1)  # identical bits on every rank
    np.testing.assert_allclose(dW0, full["dW"], atol=1e-13)
    np.testing.assert_allclose(np.load(tmp_path / "db0.npy"), full["db"], atol=1e-13)
    logp = np.concatenate([np.load(tmp_path / "logp0.npy"), np.load(tmp_path / "logp1.npy")])
    np.testing.assert_array_equal(logp, full["logp"])


def test_failed_rank_is_reported_not_hung(tmp_path):
    port = _free_port()
    with pytest.raises(Exception):
        mp.start_processes(_worker, args=(2, port, str(tmp_path), 1), nprocs=2, join=True,
                           start_method="spawn")
    assert not (tmp_path / "dW0.npy").exists()
