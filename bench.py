#!/usr/bin/env python
"""Throughput of the fused linear logp forward + backward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = ll_forward + ll_backward (grad_hidden and an FP32 grad_weight;
no bias) over one batch of the large-vocabulary workload: 32768 tokens,
hidden 4096, vocab 151936 (N * V > 2^31), bf16 operands, grad_logp ~ N(0, 1)
with exactly 10 % of the rows +0, synthetic seeded inputs.  Rank 0 prints one
JSON line.  Inputs are resident in HBM for `value`; `e2e` adds, every step,
the host->device copy of the step's hidden states / targets / upstream
gradient from pinned memory and the device->host read of logp.  L2 is
flushed between steps (a 512 MiB write outside the timed events).  The same
line carries the 4096 x 2048 x 32768 bf16 step and the logits-input path
(bf16 logits [32768, 151936]) as extra keys.

--impl reference times the FP64 CPU oracle on a bounded sample of the same
workload (rank 0 only; other ranks exit at once).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tokens/sec fwd+bwd fused linear_logp (1 GB300) and % of BF16 tensor peak"
WORKLOAD = "bf16_32k_4k_151936"
SMALL_WORKLOAD = "bf16_4k_2k_32k"
# a step longer than this runs the GPU at its power cap: its kernels are rated
# against the sustained tensor peak, shorter ones against the burst peak
LONG_STEP_MS = 5.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--token-chunks", type=int, default=0)
    ap.add_argument("--split-s", default="auto", choices=["auto", "always", "never"],
                    help="hi / lo split of the softmax part S (16-bit operands)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-logits", action="store_true",
                    help="skip the logits-input path measurement")
    ap.add_argument("--no-small", action="store_true",
                    help="skip the 4096 x 2048 x 32768 step measured beside the default one")
    ap.add_argument("--no-single", action="store_true",
                    help="skip the single-call (ll_forward_backward) measurement")
    ap.add_argument("--rows", type=int, default=0,
                    help="override the workload's token count (a smaller case of the same "
                         "shape, for profiling)")
    ap.add_argument("--workload", default=WORKLOAD,
                    choices=["fp32_small", "bf16_4k_2k_32k", "sweep_16k_4k_32000",
                             "bf16_32k_4k_151936"],
                    help="linear workload to time (default: the benchmark workload)")
    ap.add_argument("--dtype", default=None, choices=["bf16", "f16", "f32"],
                    help="operand dtype of the dtype sweep workload")
    ap.add_argument("--bias", action="store_true", help="dtype sweep workload with a bias")
    ap.add_argument("--shards", type=int, default=0,
                    help="also time the vocab-parallel composition with this many shards, "
                         "run one after another on this GPU (the collectives replaced by "
                         "their single-process equivalents)")
    ap.add_argument("--logits-rows", type=int, default=32768,
                    help="rows of the logits-input measurement (vocab 151936)")
    ap.add_argument("--logits-only", action="store_true",
                    help="time only the logits-input path (for profiling; prints its object)")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def fp32_sgemm_tflops(device) -> float:
    """The FP32 GEMM rate of this GPU through cuBLAS with TF32 off: the
    denominator an FP32 user compares against."""
    import torch
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        n = 8192
        a = torch.randn(n, n, device=device)
        b = torch.randn(n, n, device=device)
        c = torch.empty(n, n, device=device)
        torch.matmul(a, b, out=c)
        best = float("inf")
        for _ in range(5):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            torch.matmul(a, b, out=c)
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        del a, b, c
        torch.cuda.empty_cache()
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


def tf32_tflops(device, sustained: bool) -> dict:
    """cuBLAS FP32 GEMM with TF32 tensor cores allowed (8192^3): best of 10
    (burst) and, when asked, the rate of a 2 s back-to-back loop (sustained)."""
    import torch
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        n = 8192
        a = torch.randn(n, n, device=device)
        b = torch.randn(n, n, device=device)
        c = torch.empty(n, n, device=device)
        for _ in range(3):
            torch.matmul(a, b, out=c)
        best = float("inf")
        for _ in range(10):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            torch.matmul(a, b, out=c)
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        out = {"burst": 2.0 * n ** 3 / (best * 1e-3) / 1e12, "sustained": None,
               "how": "torch.matmul FP32 8192^3, allow_tf32, CUDA events"}
        if sustained:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            k, t0 = 0, time.time()
            e0.record()
            while time.time() - t0 < 2.0:
                torch.matmul(a, b, out=c)
                k += 1
                if k % 16 == 0:
                    torch.cuda.synchronize()
            e1.record()
            torch.cuda.synchronize()
            out["sustained"] = 2.0 * n ** 3 * k / (e0.elapsed_time(e1) * 1e-3) / 1e12
        del a, b, c
        torch.cuda.empty_cache()
        return out
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(k):
            return int(os.environ[k])
    return os.cpu_count() or 1


class Clocks:
    """nvidia-smi samples during the timed region (SM clock, throttle reasons)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", delete=False, suffix=".csv")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.strip().split(",") for r in self.file.read().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[0]))
                mx = float(r[1])
                for nm, v in zip(names, r[3:7]):
                    if v.strip().lower() == "active":
                        reasons.add(nm)
            except (ValueError, IndexError):
                continue
        if not sm:
            return None
        busy = [s for s in sm if s > 0.5 * (mx or max(sm))] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": mx, "samples": len(sm),
                "reasons": sorted(reasons)}


# source files each timed kernel is built from (a change to any of them
# invalidates a stored ncu traffic figure for that kernel)
KERNEL_SOURCES = {
    "gemm": ["gemm_tc.cu", "gemm_common.cuh", "epilogue.cuh", "ll_device.cuh", "ll_internal.h",
             "capi.cu"],
    "gemm_f32": ["gemm_tf32.cu", "gemm_tc.cu", "gemm_common.cuh", "epilogue.cuh", "ll_device.cuh",
                 "ll_internal.h", "capi.cu"],
    "logits": ["logits_kernels.cu", "ll_device.cuh", "ll_internal.h"],
}
PHASE_SOURCES = {"fwd_gemm": "gemm", "recompute_gemm": "gemm", "grad_gemm": "gemm",
                 "fwd_gemm_f32": "gemm_f32", "recompute_gemm_f32": "gemm_f32",
                 "grad_gemm_f32": "gemm_f32", "logits_fwd": "logits", "logits_bwd": "logits",
                 "logits_fused": "logits"}


def kernel_source_hash(phase: str) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "cross_entropy_rl_gb300", "csrc")
    for f in KERNEL_SOURCES[PHASE_SOURCES[phase]]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(phase: str, workload: str = WORKLOAD):
    """DRAM bytes per launch of `phase` from the committed ncu summary, if it
    was taken on the current sources of that kernel; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p) or phase not in PHASE_SOURCES:
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get(workload, {}).get(phase)
    if not ent or ent.get("source_hash") != kernel_source_hash(phase):
        return None
    return ent.get("dram_bytes_per_launch")


def decoded(p):
    """The workload's stored operands as float64 arrays, decoded once (every
    storage dtype embeds exactly in float64), as the GPU side's inputs are
    resident before its timed region."""
    import oracle

    dt = p["dtype"]
    return dict(p, h=oracle.decode(p["h"], dt), W=oracle.decode(p["W"], dt),
                b=oracle.decode(p["b"], dt), dtype="f64")


def cpu_baseline(p, rows_target_s=12.0):
    """The FP64 oracle on a bounded sample of the workload's rows: the seeded
    256-row sample, doubled while a call stays well under the target time."""
    import oracle
    from cross_entropy_rl_gb300 import synth

    q = decoded(p)
    rows = min(256, p["N"])
    while True:
        sel = synth.sample_rows(0, p["N"], rows)
        t0 = time.perf_counter()
        oracle.linear_rows(q["gl"], q["h"], q["W"], q["b"], q["y"], "f64", sel)
        dt = time.perf_counter() - t0
        if dt * 2.5 > rows_target_s or rows >= p["N"]:
            break
        rows = min(p["N"], rows * 2)
    extra = "" if rows >= p["N"] else "; tokens/s extrapolated linearly in N"
    return {"value": rows / dt, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"{rows} of {p['N']} tokens (seeded sample; full vocab {p['V']}, hidden "
                      f"{p['D']}): forward, grad_hidden and those tokens' grad_weight/grad_bias "
                      f"contribution, {dt:.2f} s{extra}"}


def run_reference(args, rank):
    """The oracle as the reference arm: each step is a bounded sample of the
    same workload as the other arm."""
    if rank != 0:
        return
    import numpy as np

    import oracle
    from cross_entropy_rl_gb300 import synth

    wl = dict(synth.WORKLOADS[args.workload])
    if args.workload == "sweep_16k_4k_32000":
        wl.update(dtype=args.dtype or "bf16", bias=args.bias)
    p = synth.linear_inputs(**wl, seed=0)
    q = decoded(p)
    # tokens per step: a step also pays a fixed cost (the sample's grad_weight
    # contribution touches all of [V, D]), so too small a sample understates the
    # oracle's rate; 128 tokens keep a step near 2 s at the large workload
    rows = 128
    for i in range(args.warmup):
        oracle.linear_rows(q["gl"], q["h"], q["W"], q["b"], q["y"], "f64",
                           np.arange(rows) % p["N"])
    t0 = time.perf_counter()
    for i in range(args.steps):
        s = (np.arange(rows) + i * rows) % p["N"]
        oracle.linear_rows(q["gl"], q["h"], q["W"], q["b"], q["y"], "f64", s)
    t = time.perf_counter() - t0
    v = rows * args.steps / t
    out = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
           "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": 1e3 * t / args.steps, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": args.workload, "N": p["N"], "D": p["D"], "V": p["V"],
                      "bias": p["b"] is not None, "grad_weight": "fp64",
                      "step": f"{rows} tokens per step (bounded sample)"},
           "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": blas_threads(),
                            "kind": "oracle",
                            "sample": f"{rows} tokens per step, {args.steps} steps"},
           "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch

    import cross_entropy_rl_gb300 as ll
    from cross_entropy_rl_gb300 import dp, synth

    dist = None
    if world > 1:
        import torch.distributed as dist
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    ll.load()
    if args.logits_only:
        if rank == 0:
            print(json.dumps(logits_path(args, device, peaks()[0])), flush=True)
        return
    wl = dict(synth.WORKLOADS[args.workload])
    if args.workload == "sweep_16k_4k_32000":
        wl.update(dtype=args.dtype or "bf16", bias=args.bias)
    if args.rows > 0:
        wl.update(N=args.rows)
    p = synth.linear_inputs(**wl, seed=rank)
    N, D, V, dt = p["N"], p["D"], p["V"], p["dtype"]
    tdt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[dt]
    # grad_weight: FP32, except the dtype sweep (operands and grad_weight in one dtype)
    dw_dt = tdt if args.workload == "sweep_16k_4k_32000" else torch.float32
    has_bias = p["b"] is not None

    def to_dev(a, bf16=False):
        a = np.ascontiguousarray(a)
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if bf16 else torch.from_numpy(a)
        return t.to(device)

    isbf = dt == "bf16"
    h, W = to_dev(p["h"], isbf), to_dev(p["W"], isbf)
    b = to_dev(p["b"], isbf) if has_bias else None
    y, gl = to_dev(p["y"]), to_dev(p["gl"])
    logp = torch.empty(N, dtype=torch.float32, device=device)
    lse = torch.empty_like(logp)
    dh = torch.empty(N, D, dtype=tdt, device=device)
    dW = torch.empty(V, D, dtype=dw_dt, device=device)
    db = torch.empty(V, dtype=dw_dt, device=device) if has_bias else None
    ws_f = torch.empty(max(256, ll.workspace_size(N, D, V, tdt)), dtype=torch.uint8,
                       device=device)
    split_code = ll.SPLIT_MODES[args.split_s]
    ws_b = torch.empty(max(256, ll.load().ll_workspace_size(
        N, D, V, ll._code(tdt), args.token_chunks, 1, int(has_bias) | (split_code << 1))),
        dtype=torch.uint8, device=device)
    flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()

    def step(hh, yy, gg):
        ll.forward(hh, W, b, yy, workspace=ws_f, out=(logp, lse))
        ll.backward(gg, hh, W, b, yy, lse, need_dh=True, need_dw=True, need_db=has_bias,
                    dh_dtype=tdt, dw_dtype=dw_dt, token_chunks=args.token_chunks,
                    split_s=args.split_s, workspace=ws_b, out=(dh, dW, db))
        if world > 1:
            # the gradient exchange of token-sharded data parallelism: the
            # ranks' grad_weight (and grad_bias) tables summed in ascending
            # rank order, slice by slice, then gathered (dp.py)
            dp.reduce_sum_fixed_order(dW)
            if db is not None:
                dp.reduce_sum_fixed_order(db)

    def barrier():
        if dist is not None:
            dist.barrier()

    def timed_loop(fn, k):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(k)]
        barrier()
        torch.cuda.synchronize()
        for i in range(k):
            flush_buf.zero_()
            evs[i][0].record(stream)
            fn()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        barrier()
        times = [a.elapsed_time(b) for a, b in evs]
        step_times.clear()
        step_times.extend(times)
        return sum(times) / k

    step_times = []
    for _ in range(args.warmup):
        step(h, y, gl)
    torch.cuda.synchronize()
    assert ll.check_status() == 0

    # device memory of one fwd + bwd through the binding (outputs and workspaces
    # allocated by the calls), above what is resident before it
    torch.cuda.synchronize()
    mem_base = torch.cuda.memory_allocated(device)
    torch.cuda.reset_peak_memory_stats(device)
    m_logp, m_lse = ll.forward(h, W, b, y)
    m_out = ll.backward(gl, h, W, b, y, m_lse, need_db=has_bias, dh_dtype=tdt, dw_dtype=dw_dt,
                        token_chunks=args.token_chunks, split_s=args.split_s)
    torch.cuda.synchronize()
    mem_peak = torch.cuda.max_memory_allocated(device) - mem_base
    del m_logp, m_lse, m_out
    torch.cuda.empty_cache()

    clocks = Clocks(local_rank)
    clocks.start()
    n0 = ll.launch_count()
    ms = timed_loop(lambda: step(h, y, gl), args.steps)
    st_sorted = sorted(step_times)
    pct = {q: st_sorted[min(len(st_sorted) - 1, int(round(q / 100 * (len(st_sorted) - 1))))]
           for q in (20, 50, 80)}
    launches = ll.launch_count() - n0
    clk = clocks.stop()
    assert ll.check_status() == 0
    if dist is not None:
        t = torch.tensor([ms], device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    value = world * N / (ms * 1e-3)

    # per-kernel durations: a second pass of the same steps with per-phase events
    ll.profile(True)
    timed_loop(lambda: step(h, y, gl), args.steps)
    prof = ll.profile_summary()
    ll.profile(False)

    # end to end: every step's inputs copied from pinned host memory and its
    # logp read back.  A copy stream and two device input sets let step i + 1's
    # host-to-device copy overlap step i; each step's timed region covers the
    # wait for its own copy, its compute and the read-back (step 0's copy is
    # issued inside its region).
    h_host = torch.empty(N, D, dtype=tdt).pin_memory()
    h_host.copy_(h.cpu())
    y_host = y.cpu().pin_memory()
    g_host = gl.cpu().pin_memory()
    logp_host = torch.empty(N, dtype=torch.float32).pin_memory()
    sets = [(torch.empty_like(h), torch.empty_like(y), torch.empty_like(gl)) for _ in range(2)]
    ready = [torch.cuda.Event() for _ in range(2)]
    used = [torch.cuda.Event() for _ in range(2)]
    cstream = torch.cuda.Stream(device=device)

    def copy_in(i):
        with torch.cuda.stream(cstream):
            cstream.wait_event(used[i % 2])  # the set's previous step is done with it
            hb, yb, gb = sets[i % 2]
            hb.copy_(h_host, non_blocking=True)
            yb.copy_(y_host, non_blocking=True)
            gb.copy_(g_host, non_blocking=True)
            ready[i % 2].record(cstream)

    def e2e_loop(k):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(k)]
        barrier()
        torch.cuda.synchronize()
        for i in range(k):
            flush_buf.zero_()
            evs[i][0].record(stream)
            if i == 0:
                copy_in(0)
            stream.wait_event(ready[i % 2])
            if i + 1 < k:
                copy_in(i + 1)
            step(*sets[i % 2])
            used[i % 2].record(stream)
            logp_host.copy_(logp, non_blocking=True)
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        barrier()
        return sum(a.elapsed_time(b) for a, b in evs) / k

    if args.warmup > 0:
        e2e_loop(args.warmup)
    ms_e2e = e2e_loop(args.steps)
    if dist is not None:
        t = torch.tensor([ms_e2e], device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_e2e = float(t.item())

    # single call (upstream gradient known before the forward): no logits recompute
    ms_fb, prof_fb = None, {}
    if not args.no_single:
        ws_fb = torch.empty(max(256, ll.load().ll_workspace_size(
            N, D, V, ll._code(tdt), args.token_chunks, 2, int(has_bias) | (split_code << 1))),
            dtype=torch.uint8, device=device)

        def fb_step():
            ll.forward_backward(gl, h, W, b, y, need_dh=True, need_dw=True, need_db=has_bias,
                                dh_dtype=tdt, dw_dtype=dw_dt, token_chunks=args.token_chunks,
                                split_s=args.split_s, workspace=ws_fb, out=(logp, lse, dh, dW, db))

        for _ in range(args.warmup):
            fb_step()
        ms_fb = timed_loop(fb_step, args.steps)
        assert ll.check_status() == 0
        ll.profile(True)
        timed_loop(fb_step, args.steps)
        prof_fb = ll.profile_summary()
        ll.profile(False)
        if dist is not None:
            t = torch.tensor([ms_fb], device=device)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            ms_fb = float(t.item())
        del ws_fb

    if rank != 0:
        return
    pk, pk_kind = peaks()
    sfx = "_f32" if dt == "f32" else ""
    flops = {"fwd_gemm" + sfx: 2.0 * N * D * V, "recompute_gemm" + sfx: 2.0 * N * D * V,
             "grad_gemm" + sfx: 4.0 * N * D * V}  # grad_hidden + grad_weight tiles
    gemms = {k: v for k, v in prof.items() if k in flops}
    dom = max(gemms, key=lambda k: gemms[k][1])
    cnt, tot = gemms[dom]
    avg_ms = tot / cnt
    # flops[] are per step; a step launches the kernel once per token chunk
    launch_flops = flops[dom] * args.steps / cnt
    achieved = launch_flops / (avg_ms * 1e-3) / 1e12
    simt_peak = 152 * 128 * 2 * pk.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
    # a long step keeps the GPU at its power cap: its kernels are rated
    # against the sustained peak, a short step's against the burst peak
    sustained = ms > LONG_STEP_MS
    bf16_sus = pk.get("bf16_tflops_sustained", pk["bf16_tflops"])
    tf32 = None
    if dt == "f32":
        # FP32 operands run as three TF32 MMAs per product (hi*hi + hi*lo +
        # lo*hi): the tensor peak for FP32 work is the TF32 rate / 3, the
        # TF32 rate measured here through cuBLAS (FP32 inputs, TF32 allowed)
        tf32 = tf32_tflops(device, sustained)
        burst_pk = tf32["burst"] / 3.0
        sus_pk = tf32["sustained"] / 3.0 if tf32["sustained"] else None
        pk_kind = (f"measured in this run: cuBLAS TF32 8192^3 "
                   f"{'sustained (2 s loop)' if sustained else 'burst (best of 10)'} / 3 "
                   "(3 x TF32 per FP32 product)")
    else:
        # fp16 has the same dense tensor rate as bf16
        burst_pk, sus_pk = pk["bf16_tflops"], bf16_sus
        pk_kind = f"{pk_kind} bf16 {'sustained' if sustained else 'burst'}"
    peak = sus_pk if sustained else burst_pk
    bound = "tensor"
    useful = 6.0 * N * D * V / (ms * 1e-3) / 1e12
    executed = 8.0 * N * D * V / (ms * 1e-3) / 1e12
    sgemm = fp32_sgemm_tflops(device) if dt == "f32" else None
    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dt,
        "data": "synthetic",
        "config": {"workload": args.workload, "N": N, "D": D, "V": V, "bias": has_bias,
                   "grad_weight": str(dw_dt).replace("torch.", ""),
                   "grad_hidden": str(tdt).replace("torch.", ""),
                   "token_chunks": args.token_chunks or "auto",
                   "split_s": args.split_s if dt != "f32" else None,
                   "l2": "flushed between steps (512 MiB write outside the timed events)",
                   "parallelism": f"dp{world}",
                   "dp_sync": None if world == 1 else {
                       "what": "grad_weight (+ grad_bias) summed over ranks in ascending rank "
                               "order: all-to-all reduce-scatter + ll_sum_ordered + all-gather, "
                               "inside the timed step",
                       "bytes_per_rank": dp.slice_bytes(dW.numel(), dW.element_size(), world)}},
        "useful_tflops": useful, "useful_frac_of_bf16_peak": useful / pk["bf16_tflops"],
        "useful_frac_of_sustained_bf16_peak": useful / bf16_sus,
        "useful_frac_of_peak": useful / peak, "peak_tflops": peak,
        "target": None if dt == "f32" else {
            "useful_frac": 0.60, "against": "peak_tflops", "peak_kind":
                "sustained (the step runs at the power cap)" if sustained else "burst",
            "met": bool(useful / peak >= 0.60)},
        "tf32_tflops": tf32,
        "useful_frac_of_fp32_cuda_core_peak": useful / simt_peak if dt == "f32" else None,
        "fp32_sgemm": None if sgemm is None else {
            "tflops": sgemm, "useful_frac": useful / sgemm,
            "how": "torch.matmul FP32 8192^3 with TF32 off, best of 5, CUDA events, "
                   "measured in this run before the timed steps"},
        "executed_tflops_incl_recompute": executed,
        "peak_source": pk_kind,
        "roofline": {"bound": bound, "kernel": dom, "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak,
                     "peak_kind": "sustained" if sustained else "burst",
                     "frac_of_burst": achieved / burst_pk,
                     "frac_of_sustained": achieved / sus_pk if sus_pk else None,
                     "traffic": ncu_traffic(dom, args.workload), "avg_launch_ms": avg_ms,
                     "flops_per_launch": launch_flops, "launches_per_step": cnt / args.steps},
        "kernels_ms_per_step": {k: v[1] / args.steps for k, v in prof.items()},
        "gpu_launches": launches,
        "single_call": None if ms_fb is None else {
            "value": world * N / (ms_fb * 1e-3), "unit": "tokens/s", "ms_per_step": ms_fb,
            "useful_frac_of_bf16_peak": 6.0 * N * D * V / (ms_fb * 1e-3) / 1e12
            / pk["bf16_tflops"],
            "kernels_ms_per_step": {k: v[1] / args.steps for k, v in prof_fb.items()},
            "call": "ll_forward_backward (grad_logp known before the forward; "
                    "bitwise the outputs of ll_forward + ll_backward)"},
        "e2e": {"value": world * N / (ms_e2e * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": h.numel() * h.element_size() + y.numel() * 8 + gl.numel() * 4,
                "d2h_bytes_per_step": logp.numel() * 4, "ms_per_step": ms_e2e,
                "pipeline": "a copy stream and two device input sets: step i + 1's host-to-"
                            "device copy overlaps step i; each step waits for its own copy"},
        "clocks": clk,
        "step_ms_percentiles": {"p20": pct[20], "p50": pct[50], "p80": pct[80]},
        "memory": {"peak_bytes_above_resident": mem_peak,
                   "workspace_bytes": {"forward": ws_f.numel(), "backward": ws_b.numel()},
                   "note": "one ll_forward + ll_backward allocating its outputs and "
                           "workspaces, max_memory_allocated above the resident inputs"},
    }
    if args.shards > 1 and world == 1:
        out["vocab_shards"] = shard_path(args, h, W, b, y, gl, ms, timed_loop, tdt, dw_dt)
    if args.workload == WORKLOAD and not args.no_small:
        out[SMALL_WORKLOAD] = small_workload(args, device, pk, flush_buf)
    if not args.no_logits and args.workload == WORKLOAD:
        del ws_b, flush_buf
        torch.cuda.empty_cache()
        out["logits_path"] = logits_path(args, device, pk)
    if world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(p)
    print(json.dumps(out), flush=True)


def small_workload(args, device, pk, flush_buf):
    """The 4096 x 2048 x 32768 bf16 step (FP32 grad_weight, no bias): two
    calls and the single call, L2 flushed between steps, with the gradient
    launch's rate against the burst peak (a short step)."""
    import numpy as np
    import torch

    import cross_entropy_rl_gb300 as ll
    from cross_entropy_rl_gb300 import synth

    p = synth.linear_inputs(**synth.WORKLOADS[SMALL_WORKLOAD], seed=0)
    N, D, V = p["N"], p["D"], p["V"]

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(
            torch.bfloat16).to(device)

    h, W = bf(p["h"]), bf(p["W"])
    y, gl = torch.from_numpy(p["y"]).to(device), torch.from_numpy(p["gl"]).to(device)
    logp = torch.empty(N, dtype=torch.float32, device=device)
    lse = torch.empty_like(logp)
    dh = torch.empty(N, D, dtype=torch.bfloat16, device=device)
    dW = torch.empty(V, D, dtype=torch.float32, device=device)
    ws_f = torch.empty(max(256, ll.workspace_size(N, D, V, torch.bfloat16)), dtype=torch.uint8,
                       device=device)
    ws_b = torch.empty(max(256, ll.workspace_size(N, D, V, torch.bfloat16, 0, backward=True)),
                       dtype=torch.uint8, device=device)
    ws_fb = torch.empty(max(256, ll.workspace_size(N, D, V, torch.bfloat16, 0, backward=2)),
                        dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()

    def two():
        ll.forward(h, W, None, y, workspace=ws_f, out=(logp, lse))
        ll.backward(gl, h, W, None, y, lse, need_dh=True, need_dw=True, need_db=False,
                    workspace=ws_b, out=(dh, dW, None))

    def one():
        ll.forward_backward(gl, h, W, None, y, need_dh=True, need_dw=True, need_db=False,
                            workspace=ws_fb, out=(logp, lse, dh, dW, None))

    k = max(args.steps, 100)

    def timed(fn):
        for _ in range(max(args.warmup, 3)):
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(k)]
        torch.cuda.synchronize()
        for i in range(k):
            flush_buf.zero_()
            evs[i][0].record(stream)
            fn()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in evs) / k

    ms2 = timed(two)
    ll.profile(True)
    for _ in range(k):
        flush_buf.zero_()
        two()
    prof = ll.profile_summary()
    ll.profile(False)
    ms1 = timed(one)
    assert ll.check_status() == 0
    useful = 6.0 * N * D * V
    cnt, tot = prof["grad_gemm"]
    grad = 4.0 * N * D * V * k / cnt / (tot / cnt * 1e-3) / 1e12
    return {"N": N, "D": D, "V": V, "steps": k, "ms_per_step": ms2, "value": N / (ms2 * 1e-3),
            "unit": "tokens/s",
            "useful_frac_of_bf16_peak": useful / (ms2 * 1e-3) / 1e12 / pk["bf16_tflops"],
            "single_call_ms_per_step": ms1,
            "single_call_useful_frac_of_bf16_peak":
                useful / (ms1 * 1e-3) / 1e12 / pk["bf16_tflops"],
            "grad_gemm_tflops": grad, "grad_gemm_frac_of_burst": grad / pk["bf16_tflops"],
            "grad_gemm_traffic": ncu_traffic("grad_gemm", SMALL_WORKLOAD),
            "kernels_ms_per_step": {kk: v[1] / k for kk, v in prof.items()},
            "l2": "flushed between steps (512 MiB write outside the timed events)"}


def shard_path(args, h, W, b, y, gl, ms_whole, timed_loop, tdt, dw_dt):
    """The vocab-parallel composition on one GPU: per step, each shard's
    forward (segment partials), the ordered merge of all partials, each
    shard's backward; the rank exchanges become a copy into the gathered
    partials, a max over the shards' zy and a fixed-order sum of the
    grad_hidden parts.  Compared with the whole-vocab step it shows what
    sharding costs apart from the communication."""
    import torch

    import cross_entropy_rl_gb300 as ll
    from cross_entropy_rl_gb300 import tp

    K = args.shards
    N, D = h.shape
    V = W.shape[0]
    dev = h.device
    bounds = [(v0, v1) for v0, v1 in tp.shard_bounds(V, K) if v1 > v0]
    segs = [ll.shard_segments(v1 - v0) for v0, v1 in bounds]
    pm = torch.empty(sum(segs), N, dtype=torch.float32, device=dev)
    ps = torch.empty_like(pm)
    zys = [torch.empty(N, dtype=torch.float32, device=dev) for _ in bounds]
    logp = torch.empty(N, dtype=torch.float32, device=dev)
    lse = torch.empty_like(logp)
    dh_parts = [torch.empty(N, D, dtype=torch.float32, device=dev) for _ in bounds]
    dh = torch.empty(N, D, dtype=torch.float32, device=dev)
    dW = torch.empty(V, D, dtype=dw_dt, device=dev)
    db = torch.empty(V, dtype=dw_dt, device=dev) if b is not None else None
    code = {torch.bfloat16: 2, torch.float16: 1, torch.float32: 0}[tdt]
    L = ll.load()
    ws_f = [torch.empty(max(256, L.ll_workspace_size_shard(N, D, v1 - v0, code, 0, 0, 0)),
                        dtype=torch.uint8, device=dev) for v0, v1 in bounds]
    ws_b = [torch.empty(max(256, L.ll_workspace_size_shard(N, D, v1 - v0, code, 0, 1,
                                                           int(b is not None))),
                        dtype=torch.uint8, device=dev) for v0, v1 in bounds]

    def step():
        s0 = 0
        for i, (v0, v1) in enumerate(bounds):
            bb = None if b is None else b[v0:v1]
            ll.forward_shard(h, W[v0:v1], bb, y, v0, V, workspace=ws_f[i],
                             out=(pm[s0:s0 + segs[i]], ps[s0:s0 + segs[i]], zys[i]))
            s0 += segs[i]
        zy = zys[0]
        for z in zys[1:]:
            zy = torch.maximum(zy, z)
        ll.lse_merge(pm, ps, zy, y, V, out=(logp, lse))
        for i, (v0, v1) in enumerate(bounds):
            bb = None if b is None else b[v0:v1]
            ll.backward_shard(gl, h, W[v0:v1], bb, y, lse, v0, V, workspace=ws_b[i],
                              out=(dh_parts[i], dW[v0:v1], None if db is None else db[v0:v1]))
        dh.copy_(dh_parts[0])
        for part in dh_parts[1:]:
            dh.add_(part)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    assert ll.check_status() == 0
    ms = timed_loop(step, args.steps)
    return {"shards": len(bounds), "ms_per_step": ms, "value": N / (ms * 1e-3),
            "unit": "tokens/s", "ratio_to_whole_vocab": ms / ms_whole,
            "note": "shards run one after another on one GPU; the rank exchanges "
                    "(partials gather, zy max, grad_hidden sum) are single-process "
                    "copies, max and adds; grad_hidden accumulated in FP32"}


def logits_path(args, device, pk):
    """logits_logp_fwd + logits_logp_bwd on bf16 logits [32768, 151936]
    (9.27 GiB, larger than L2): tokens/s and HBM roofline of each kernel."""
    import torch

    import cross_entropy_rl_gb300 as ll

    N, V = args.logits_rows, 151936
    g = torch.Generator(device=device)
    g.manual_seed(0)
    x = (torch.randn(N, V, generator=g, device=device) * (2.0 ** 0.5)).to(torch.bfloat16)
    y = torch.randint(0, V, (N,), generator=g, device=device)
    gl = torch.randn(N, generator=g, device=device)
    logp = torch.empty(N, device=device)
    lse = torch.empty(N, device=device)
    dx = torch.empty_like(x)
    stream = torch.cuda.current_stream()
    steps = max(3, min(args.steps, 20))

    def step():
        ll.logits_fwd(x, y, out=(logp, lse))
        ll.logits_bwd(gl, x, y, lse, out=dx)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    ll.profile(True)
    for _ in range(steps):
        step()
    prof = ll.profile_summary()
    ll.profile(False)
    assert ll.check_status() == 0

    # one pass over the logits when grad_logp is known before the forward
    def fused_step():
        ll.logits_fwd_bwd(gl, x, y, out=(logp, lse, dx))

    for _ in range(3):
        fused_step()
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(steps):
        fused_step()
    b.record(stream)
    torch.cuda.synchronize()
    ms_fused = a.elapsed_time(b) / steps
    assert ll.check_status() == 0
    fwd_ms = prof["logits_fwd"][1] / prof["logits_fwd"][0]
    bwd_ms = prof["logits_bwd"][1] / prof["logits_bwd"][0]
    fwd_b, bwd_b = 2.0 * N * V, 4.0 * N * V
    peak = pk["hbm_gbs"]
    # the stored figure is per launch of 32768 rows (scaled from a smaller capture)
    t_full = ncu_traffic("logits_bwd", "logits_32k_151936")
    logits_traffic = None if t_full is None else t_full * N / 32768
    return {"workload": "logits_32k_151936" if N == 32768 else f"logits_{N}_151936",
            "N": N, "V": V, "dtype": "bf16",
            "value": N / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms,
            "steps": steps, "l2": "inputs (9.27 GiB) larger than L2, no flush",
            "bytes_per_token": 6 * V, "step_gbs": 6.0 * N * V / (ms * 1e-3) / 1e9,
            "step_frac_of_hbm": 6.0 * N * V / (ms * 1e-3) / 1e9 / peak,
            "roofline": {"bound": "hbm", "kernel": "logits_bwd",
                         "achieved": bwd_b / (bwd_ms * 1e-3) / 1e9, "peak": peak, "unit": "GB/s",
                         "frac": bwd_b / (bwd_ms * 1e-3) / 1e9 / peak,
                         "traffic": logits_traffic, "avg_launch_ms": bwd_ms},
            "logits_fwd": {"ms": fwd_ms, "gbs": fwd_b / (fwd_ms * 1e-3) / 1e9,
                           "frac": fwd_b / (fwd_ms * 1e-3) / 1e9 / peak},
            "single_pass": {"call": "logits_logp_fwd_bwd (grad_logp known before the forward)",
                            "traffic": None if ncu_traffic("logits_fused", "logits_32k_151936")
                            is None else ncu_traffic("logits_fused", "logits_32k_151936")
                            * N / 32768,
                            "ms_per_step": ms_fused, "value": N / (ms_fused * 1e-3),
                            "unit": "tokens/s", "bytes_per_token": 4 * V,
                            "gbs": 4.0 * N * V / (ms_fused * 1e-3) / 1e9,
                            "frac": 4.0 * N * V / (ms_fused * 1e-3) / 1e9 / peak}}


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
