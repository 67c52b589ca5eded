#!/usr/bin/env python
"""Benchmark of the quantized attention hot path (prep + fused attention).

One step = sage_prep_qkv + sage_attn_fwd over the long-sequence DiT-like
workload: B=1, H=24, Nq=Nkv=16384, D=128, BF16, strided NHD views into one
fused [B, N, 3, H, D] projection buffer, non-causal.  The metric is
4*B*H*Nq*Nkv*D / step time in TOPS.  Inputs (302 MB) and output (101 MB) are
larger than the 129 MB L2, so no L2 flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --forms     # one JSON line per form of the path (not the
                              # contract line): causal, fused entry, BKV = 64, D = 64
  python bench.py --latency   # p50 latency on the single-tile workload (Q128 x KV192 x
                              # D128, the pages' prototype shape); not the contract line
  python bench.py --configs [i ...]   # one JSON line per named workload (1-5), with
                              # the CPU oracle timed beside it; not the contract line

--impl reference times the CPU oracle (the only other implementation of the
contract; no other implementation exists to install) on a bounded sample of
the same workload.  Under torchrun (N > 1) the ranks split the heads of the
one problem (each head is independent: K mean, scales and attention are per
(b, h); no exchange step), or with --replicas each rank runs the whole
problem; rank 0 prints one JSON line with the whole-job throughput.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "quantized attention TOPS (4·B·H·N²·D/t) at N=16K,D=128; % of FP8/INT8 peak"
UNIT = "TOPS"
CONFIG_ID = 4
DTYPE = "int8 QK (FP16 integer codes) + e4m3 PV, FP32 accumulate, bf16 in/out"
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
E2E_HEAD_GROUPS = 6     # head ranges of the overlapped host entry (4..8 measured best on this workload)
E2E_WINDOWS = 3         # end-to-end timing windows (the median is reported)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--replicas", action="store_true",
                    help="with several ranks, run one whole problem per rank instead of splitting its heads")
    ap.add_argument("--forms", action="store_true",
                    help="time every form of the path on the bench workload shape instead")
    ap.add_argument("--latency", action="store_true",
                    help="p50 latency of prep + attention on the single-tile workload instead")
    ap.add_argument("--configs", type=int, nargs="*", default=None,
                    help="one JSON line per named workload (default all five) with the oracle timed beside it")
    return ap.parse_args()


def sources_sha256(paths):
    """SHA-256 over the given repository files, concatenated in order."""
    import hashlib
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def kernel_traffic():
    """DRAM bytes per launch of the attention kernel from the committed ncu
    capture (profiles/sage_attn_kernel_counters.json), or None when any source
    the kernel is compiled from has changed since the counters were taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "sage_attn_kernel_counters.json")) as f:
            rec = json.load(f)
        sha = sources_sha256(rec["sources"])
    except (OSError, KeyError, ValueError, TypeError):
        return None
    if sha != rec.get("sources_sha256"):
        return None
    return int(rec["dram_bytes_read"]) + int(rec["dram_bytes_write"])


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def peaks():
    """bf16 dense peak (TFLOP/s) from the measured file, else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"sage_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        self.proc.wait()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        loaded = [s for s in sm if s > 0.5 * max(sm)] if sm else []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------
# The CPU oracle on the host cores.  Work is split by (b, h) head over spawned
# worker processes (spawned, never forked, so no CUDA state is inherited), one
# BLAS thread each, so the worker count is the number of cores used.
# ----------------------------------------------------------------------------
_BLAS_ENV = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


class _OneBlasThread:
    """Spawned children inherit os.environ at start: hold the one-thread BLAS
    settings while workers start (they unpickle numpy inputs before any code
    of theirs runs)."""

    def __enter__(self):
        self.old = {k: os.environ.get(k) for k in _BLAS_ENV}
        for k in _BLAS_ENV:
            os.environ[k] = "1"

    def __exit__(self, *exc):
        for k, v in self.old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def _oracle_worker_init():
    for name in _BLAS_ENV:
        os.environ[name] = "1"
    import numpy  # noqa: F401
    from oracle import sage_oracle  # noqa: F401


def _oracle_head_task(task):
    """Prepare one head and attend the given query rows of it (None: every
    valid row).  Returns (t_prep, t_attention, ops)."""
    import numpy as np

    from oracle import sage_oracle as O
    q, k, v, lq, lk, rows = task
    t0 = time.perf_counter()
    prep = O.prepare(q, k, v, [lq], [lk])
    t1 = time.perf_counter()
    rows = np.arange(lq) if rows is None else np.asarray(rows)
    O.attention_rows(prep, 0, 0, rows)
    t2 = time.perf_counter()
    return t1 - t0, t2 - t1, 4 * len(rows) * lk * q.shape[-1]


def oracle_workers() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def head_tasks(w, heads=None, rows=None):
    """Oracle tasks for a workload: every (b, h) head (or the given ones), each
    with its own float32 [1, 1, N, D] inputs and lengths."""
    views = [t.float().numpy() for t in w.views()]
    heads = [(b, h) for b in range(w.B) for h in range(w.H)] if heads is None else heads
    tasks = []
    for b, h in heads:
        q, k, v = (x[b:b + 1, h:h + 1].copy() for x in views)
        tasks.append((q, k, v, w.qlens[b], w.kvlens[b], rows))
    return tasks


def time_oracle(tasks, workers=None):
    """Wall time of the oracle over the tasks on a pool of spawned workers.
    Returns (seconds, ops, workers used, prep seconds summed, attention seconds summed)."""
    import multiprocessing as mp
    n = min(workers or oracle_workers(), len(tasks))
    ctx = mp.get_context("spawn")
    with _OneBlasThread(), ctx.Pool(n, initializer=_oracle_worker_init) as pool:
        pool.map(abs, range(n))                               # every worker started and importing done
        t0 = time.perf_counter()
        res = pool.map(_oracle_head_task, tasks, chunksize=1)
        wall = time.perf_counter() - t0
    return wall, sum(r[2] for r in res), n, sum(r[0] for r in res), sum(r[1] for r in res)


def _head_worker_main(conn, q, k, v, lq, lk):
    """A worker that keeps one prepared head and attends batches of its rows."""
    _oracle_worker_init()
    import numpy as np

    from oracle import sage_oracle as O
    t0 = time.perf_counter()
    prep = O.prepare(q, k, v, [lq], [lk])
    conn.send(time.perf_counter() - t0)
    while True:
        rows = conn.recv()
        if rows is None:
            break
        t0 = time.perf_counter()
        O.attention_rows(prep, 0, 0, np.asarray(rows))
        conn.send(time.perf_counter() - t0)


class HeadWorkers:
    """One spawned process per sampled head of the long workload: each
    prepares its head once (timed), then attends a batch of query rows per
    step; a step ends when every worker has answered."""

    def __init__(self, w, heads):
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        self.w = w
        self.procs, self.conns = [], []
        for task in head_tasks(w, [(0, h) for h in heads]):
            parent, child = ctx.Pipe()
            p = ctx.Process(target=_head_worker_main, args=(child, *task[:5]), daemon=True)
            with _OneBlasThread():
                p.start()
            self.procs.append(p)
            self.conns.append(parent)
        self.t_prep = [c.recv() for c in self.conns]        # seconds per head
        self.next = 0

    def step(self, rows: int):
        """Wall seconds for `rows` query rows of every worker's head, plus the
        heads' preparation charged pro rata (rows / Nq of the slowest one)."""
        import numpy as np
        idx = (self.next + np.arange(rows)) % self.w.Nq
        self.next += rows
        t0 = time.perf_counter()
        for c in self.conns:
            c.send(idx)
        for c in self.conns:
            c.recv()
        wall = time.perf_counter() - t0
        ops = 4 * rows * self.w.Nkv * self.w.D * len(self.conns)
        return wall + max(self.t_prep) * rows / self.w.Nq, ops

    def close(self):
        for c in self.conns:
            c.send(None)
        for p in self.procs:
            p.join(timeout=30)


def max_over_ranks(ms: float, world: int, device=None) -> float:
    """Largest per-rank time of the timed region (ranks run independent replicas)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tops(ops_per_replica: int, world: int, ms_per_step: float) -> float:
    """All ranks' work divided by the slowest rank's time (replicas: every rank
    runs the whole workload)."""
    return world * ops_per_replica / (ms_per_step * 1e-3) / 1e12


def head_range(rank: int, world: int, H: int):
    """Heads [h0, h1) of one rank when `world` ranks split the H heads of one
    problem: contiguous ranges whose sizes differ by at most one."""
    if not 1 <= world <= H or not 0 <= rank < world:
        raise ValueError(f"cannot split {H} heads over {world} ranks")
    return H * rank // world, H * (rank + 1) // world


def config_of(w, world=1, split=False):
    par = (f"heads split over {world} ranks (each rank the sub-problem of its heads)" if split else
           "one problem per GPU" if world == 1 else f"replicas: {world} independent problems, one per GPU")
    return {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nkv": w.Nkv, "D": w.D,
            "layout": "strided NHD views into a fused [B,N,3,H,D] BF16 buffer",
            "causal": False, "l2": "inputs (302 MB) larger than L2 (129 MB); no flush",
            "parallelism": par}


def run_reference(args, world, rank):
    """The oracle (the only other implementation of the contract), timed on
    the host cores on a bounded sample of the bench workload per step."""
    if rank != 0:
        return
    from quantized_exact_attention_gb300 import workloads as W
    w = W.make_config(CONFIG_ID)
    heads = list(range(min(oracle_workers(), w.H)))
    pool = HeadWorkers(w, heads)
    rows = 32
    try:
        for _ in range(args.warmup):
            pool.step(rows)
        ts, ops = [], 0
        for _ in range(args.steps):
            t, ops = pool.step(rows)
            ts.append(t)
    finally:
        pool.close()
    t_step = sum(ts) / len(ts)
    value = ops / t_step / 1e12
    sample = (f"{rows} query rows (rotating) of each of heads {heads[0]}-{heads[-1]} x all {w.Nkv} keys per "
              f"step, one worker process per head; each head's preparation (max {max(pool.t_prep):.2f} s) "
              f"charged pro rata {rows}/{w.Nq}")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": DTYPE,
            "data": "synthetic (seeded N(0,1) + K channel offsets, as the workload states)",
            "config": config_of(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": len(heads), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def hbm_peak():
    """Measured copy bandwidth (GB/s) from the generated file, else the fallback."""
    try:
        return float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def prep_bytes(w) -> int:
    """Algorithmic bytes of the preparation: every valid element of Q, K and V
    read once as BF16 (2 B) and written once as an 8-bit code (1 B)."""
    return 3 * w.D * w.H * sum(lq + 2 * lk for lq, lk in zip(w.qlens, w.kvlens))


def attn_bytes(w) -> int:
    """Algorithmic bytes of the attention kernel: INT8 Q and K codes and e4m3 V
    codes read once (1 B each), the BF16 output written once (2 B)."""
    return w.D * w.H * sum(3 * lq + 2 * lk for lq, lk in zip(w.qlens, w.kvlens))


def prep_roofline(w, ms: float, what: str) -> dict:
    peak, src = hbm_peak()
    gbs = prep_bytes(w) / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
            "peak_basis": f"{src} copy bandwidth", "algorithmic_bytes": prep_bytes(w),
            "bytes_basis": "9 B per (token, head, channel): Q, K, V read as BF16, written as 8-bit codes",
            "ms_mean": ms, "kernels": what}


def clock_note(clocks: dict) -> str | None:
    """The measured bf16 peak was taken at the clocks MEASURED_PEAKS.json records;
    state the kernel's clock beside it."""
    try:
        d = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        at = float(d["clocks_under_load"]["sm_mhz_median"])
    except Exception:
        return None
    if not clocks or not clocks.get("sm_mhz"):
        return None
    return (f"kernel timed at {clocks['sm_mhz']:.0f} MHz median; the measured bf16 peak was taken at "
            f"{at:.0f} MHz median (power-capped), so clock for clock the fraction is "
            f"{at / clocks['sm_mhz']:.3f} x the one reported")


def run_ours(args, world, rank, local):
    import torch
    import torch.distributed as dist

    import quantized_exact_attention_gb300 as S
    from quantized_exact_attention_gb300 import build as B
    from quantized_exact_attention_gb300 import workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B.build()
    S.load_library()
    w = W.make_config(CONFIG_ID)
    phys = w.to(dev)
    q, k, v = w.views(phys)
    o_phys = torch.empty((w.B, w.Nq, w.H, w.D), dtype=torch.bfloat16, device=dev)
    o = o_phys.permute(0, 2, 1, 3)
    # Several ranks split the heads of the one problem (each head is an
    # independent problem: K mean, scales and attention are per (b, h)); a
    # rank's share is the sub-problem of head-slice views of the same tensors.
    split = world > 1 and not args.replicas
    h0, h1 = head_range(rank, world, w.H) if split else (0, w.H)
    q, k, v, o = (t[:, h0:h1] for t in (q, k, v, o))
    bufs = S.alloc_prep_buffers(w.B, h1 - h0, w.Nq, w.Nkv, dev)
    stream = torch.cuda.current_stream(dev)
    ops = w.ops()                                   # the whole problem (split) or one replica

    def barrier():
        if world > 1:
            dist.barrier()

    def step():
        S.sage_prep_qkv(q, k, v, bufs, stream=stream)
        n = S.sage_last_launch_count()
        S.sage_attn_fwd(bufs, o, stream=stream)
        return n + S.sage_last_launch_count()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if S.sage_get_device_status() != S.SAGE_OK:
        raise RuntimeError("device status reports an error after warm-up")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    sampler = ClockSampler(local)
    barrier()
    torch.cuda.synchronize()
    sampler.start()
    launches = 0
    for i in range(K):
        ev[i][0].record(stream)
        S.sage_prep_qkv(q, k, v, bufs, stream=stream)
        launches += S.sage_last_launch_count()
        ev[i][1].record(stream)
        S.sage_attn_fwd(bufs, o, stream=stream)
        launches += S.sage_last_launch_count()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    total_ms = ev[0][0].elapsed_time(ev[-1][2])
    prep_ms = [e[0].elapsed_time(e[1]) for e in ev]
    attn_ms = [e[1].elapsed_time(e[2]) for e in ev]
    ms_per_step = max_over_ranks(total_ms, world, dev) / K
    if S.sage_get_device_status() != S.SAGE_OK:
        raise RuntimeError("device status reports an error after the timed steps")
    value = whole_job_tops(ops, 1 if split else world, ms_per_step)
    rank_ops = ops * (h1 - h0) // w.H

    # roofline of the dominant kernel (the fused attention): QK runs at the
    # FP16/BF16 tensor rate, PV at the FP8 rate (2x); half the ops each.
    bf16_burst, bf16_sust, src = peaks()
    attn_avg = statistics.mean(attn_ms)
    achieved = rank_ops / (attn_avg * 1e-3) / 1e12
    p16 = bf16_burst
    p8 = 2.0 * p16
    mixed = 2.0 / (1.0 / p16 + 1.0 / p8)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": mixed, "unit": "TFLOP/s",
                "frac": achieved / mixed, "traffic": kernel_traffic(),
                "traffic_unit": "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)",
                "kernel": "sage_attn_kernel (fused QK/softmax/PV)",
                "peak_basis": (f"{src} bf16 burst {p16:.1f} TF/s for QK (FP16 codes) and 2x that for "
                               f"e4m3 PV; equal op split -> 4/3 x bf16 = {mixed:.1f}"),
                "fp8_peak": p8, "frac_of_fp8_peak": achieved / p8,
                "attn_ms_mean": attn_avg, "attn_ms_p50": statistics.median(attn_ms),
                "attn_cv": statistics.pstdev(attn_ms) / attn_avg,
                "clock_scaled": clock_note(clocks),
                "prep": prep_roofline(w, statistics.mean(prep_ms), "three launches: stats+Q, finalize, K+V")}

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, w, phys, o_phys, bufs, stream, world, ops, dev, (h0, h1), split)

    cpu = None
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        heads = list(range(min(oracle_workers(), w.H)))
        pool = HeadWorkers(w, heads)
        try:
            pool.step(32)                                      # warm-up
            tt, oo = 0.0, 0
            for _ in range(32):
                t_s, o_s = pool.step(32)
                tt += t_s
                oo += o_s
        finally:
            pool.close()
        cpu = {"value": oo / tt / 1e12, "unit": UNIT, "cores": len(heads), "kind": "oracle",
               "sample": (f"1024 query rows (32 batches of 32) of each of heads {heads[0]}-{heads[-1]} x all "
                          f"{w.Nkv} keys, one worker process (one BLAS thread) per head; each head's "
                          f"preparation (max {max(pool.t_prep):.2f} s) charged pro rata 1024/{w.Nq}"),
               "seconds": tt}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
                "scaling": "strong" if split else "weak", "vs_baseline": None, "dtype": DTYPE,
                "data": "synthetic (seeded N(0,1) Q/K/V, K channel offsets N(0,2^2))",
                "config": config_of(w, world, split), "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": launches, "clocks": clocks,
                "attn_only_tops": achieved}
        print(json.dumps(line), flush=True)


def run_e2e(args, w, phys, o_phys, bufs, stream, world, ops, dev, heads, split):
    """Same metric through the public host-memory entry points: pinned host
    inputs in, device compute, host output out, all inside the timed region.
    The headline uses sage_attention_host_overlapped (copies of one head range
    overlap the kernels of the others); sage_attention_host (all copies, then
    the kernels, then the copy back) is reported beside it.  When ranks split
    the heads, each rank copies and computes only its heads' slices (the
    overlapped entry copies the logical elements of the views it is given)."""
    import torch
    import torch.distributed as dist

    import quantized_exact_attention_gb300 as S
    h0, h1 = heads
    host_in = [t.cpu().pin_memory() for t in phys]
    host_out = torch.empty(o_phys.shape, dtype=o_phys.dtype).pin_memory()
    o_view = o_phys.permute(0, 2, 1, 3)[:, h0:h1]
    qh, kh, vh = (t[:, h0:h1] for t in w.views(host_in))
    qd, kd, vd = (t[:, h0:h1] for t in w.views(list(phys)))
    oh = host_out.permute(0, 2, 1, 3)[:, h0:h1]
    groups = min(E2E_HEAD_GROUPS, h1 - h0)

    def sequential():
        S.sage_attention_host(host_in, list(phys), w.views, bufs, o_view, host_out, stream=stream)

    def overlapped():
        S.sage_attention_host_overlapped(qh, kh, vh, oh, qd, kd, vd, o_view, bufs,
                                         head_groups=groups, stream=stream)

    def timed(fn):
        """E2E_WINDOWS windows of K back-to-back steps, an event between steps.
        Returns the median of the windows' mean step times (max over ranks),
        K, the windows' means and every step's own time."""
        for _ in range(max(args.warmup, 3)):
            fn()
        torch.cuda.synchronize()
        K = max(1, min(args.steps, 20))
        windows, steps, host = [], [], []
        for _ in range(E2E_WINDOWS):
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
            if world > 1:
                dist.barrier()
            torch.cuda.synchronize()
            ev[0].record(stream)
            for i in range(K):
                t0 = time.perf_counter()
                fn()
                host.append((time.perf_counter() - t0) * 1e3)
                ev[i + 1].record(stream)
            torch.cuda.synchronize()
            windows.append(max_over_ranks(ev[0].elapsed_time(ev[-1]) / K, world, dev))
            steps += [ev[i].elapsed_time(ev[i + 1]) for i in range(K)]
        timed.host_ms = host
        return sorted(windows)[len(windows) // 2], K, windows, steps

    ms, K, win, st = timed(overlapped)
    host_ms = timed.host_ms
    seq = None
    if not split:
        ms_seq, _, win_seq, st_seq = timed(sequential)
        seq = {"api": "sage_attention_host", "value": whole_job_tops(ops, world, ms_seq),
               "ms_per_step": ms_seq, "window_ms_per_step": [round(x, 4) for x in win_seq],
               "step_ms": {"mean": statistics.mean(st_seq), "median": statistics.median(st_seq),
                           "max": max(st_seq), "n": len(st_seq)}}
    if S.sage_get_device_status() != S.SAGE_OK:
        raise RuntimeError("device status reports an error after the end-to-end steps")
    share = (h1 - h0) / w.H
    h2d = int(sum(x.numel() * x.element_size() for x in host_in) * share)
    d2h = int(host_out.numel() * host_out.element_size() * share)
    return {"value": whole_job_tops(ops, 1 if split else world, ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": K,
            "timing": f"median of {E2E_WINDOWS} windows of {K} back-to-back steps",
            "window_ms_per_step": [round(x, 4) for x in win],
            "step_ms": {"mean": statistics.mean(st), "median": statistics.median(st), "max": max(st),
                        "min": min(st), "n": len(st), "over_2x_median": sum(x > 2 * statistics.median(st) for x in st)},
            "host_call_ms": {"median": statistics.median(host_ms), "max": max(host_ms),
                             "note": "host time inside each call (enqueueing only; the calls do not synchronize)"},
            "api": (f"sage_attention_host_overlapped (pinned host buffers, {groups} head ranges, "
                    "copies inside the timed region)"),
            "bytes_basis": "this rank's copies" if split else "one replica's copies",
            "sequential_entry": seq}


def run_forms(args):
    """Step and attention time of each form of the path on the bench workload
    shape (16K tokens, strided NHD); one JSON line per form.  Step = everything
    the form needs from BF16 inputs to BF16 output; causal forms count half
    of the 4*H*N^2*D operations."""
    import torch

    import quantized_exact_attention_gb300 as S
    from quantized_exact_attention_gb300 import build as B
    from quantized_exact_attention_gb300 import workloads as W

    B.build()
    S.load_library()
    spec = dict(W.CONFIGS[CONFIG_ID])
    forms = [("default", 128, False, 128, "two_calls"), ("causal", 128, True, 128, "two_calls"),
             ("fused_entry", 128, False, 128, "fused"), ("fused_entry_causal", 128, True, 128, "fused"),
             ("bkv64", 128, False, 64, "two_calls"), ("d64", 64, False, 128, "two_calls"),
             ("d64_causal", 64, True, 128, "two_calls"), ("cta_pairs", 128, False, 128, "pairs"),
             ("cta_pairs_causal", 128, True, 128, "pairs")]
    K = max(3, min(args.steps, 20))
    for name, d, causal, bkv, path in forms:
        sp = dict(spec, D=d, H=spec["H"] * 128 // d, name=f"{spec['name']}_D{d}")
        w = W.make_custom(**sp)
        phys = w.to("cuda")
        q, k, v = w.views(phys)
        bufs = S.alloc_prep_buffers(w.B, w.H, w.Nq, w.Nkv, "cuda", D=d)
        o = torch.empty((w.B, w.Nq, w.H, d), dtype=torch.bfloat16, device="cuda").permute(0, 2, 1, 3)

        pairs = path == "pairs"

        def step():
            if path == "fused":
                S.sage_attention(q, k, v, o, bufs, causal=causal)
            else:
                S.sage_prep_qkv(q, k, v, bufs, bkv=bkv)
                S.sage_attn_fwd(bufs, o, causal=causal, bkv=bkv, pairs=pairs)

        for _ in range(max(args.warmup, 3)):
            step()
        torch.cuda.synchronize()
        steps, attn = [], []
        for _ in range(K):
            e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            e[0].record()
            step()
            e[1].record()
            if path != "fused":
                S.sage_attn_fwd(bufs, o, causal=causal, bkv=bkv, pairs=pairs)
            e[2].record()
            torch.cuda.synchronize()
            steps.append(e[0].elapsed_time(e[1]))
            if path != "fused":
                attn.append(e[1].elapsed_time(e[2]))
        if S.sage_get_device_status() != S.SAGE_OK:
            raise RuntimeError(f"device status reports an error in form {name}")
        ops = w.ops() * (0.5 if causal else 1.0)
        st = statistics.median(steps)
        line = {"form": name, "D": d, "H": w.H, "N": w.Nq, "causal": causal, "bkv": bkv, "entry": path,
                "step_ms_p50": st, "step_tops": ops / st / 1e9, "steps": K}
        if attn:
            at = statistics.median(attn)
            line.update(attn_ms_p50=at, attn_tops=ops / at / 1e9)
        print(json.dumps(line), flush=True)
        del phys, q, k, v, bufs, o
        torch.cuda.empty_cache()


def run_configs(args):
    """One JSON line per named workload (1-5): prep, attention and step time on
    the GPU (CUDA events, L2 flushed by a 256 MB write before every timed
    step), throughput on valid lengths, fractions of the tensor and HBM
    rooflines, and the CPU oracle timed beside it on the host cores."""
    import torch

    import quantized_exact_attention_gb300 as S
    from quantized_exact_attention_gb300 import build as B
    from quantized_exact_attention_gb300 import workloads as W

    B.build()
    S.load_library()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    bf16_burst, _, src = peaks()
    p8, mixed = 2.0 * bf16_burst, 4.0 / 3.0 * bf16_burst
    hbm, hsrc = hbm_peak()
    K = max(5, min(args.steps, 50))
    for cfg in args.configs:
        w = W.make_config(cfg)
        phys = w.to("cuda")
        q, k, v = w.views(phys)
        lens = [torch.tensor(x, dtype=torch.int32, device="cuda") if x is not None else None
                for x in (w.q_len, w.kv_len)]
        bufs = S.alloc_prep_buffers(w.B, w.H, w.Nq, w.Nkv, "cuda", D=w.D)
        o = torch.zeros((w.B, w.Nq, w.H, w.D), dtype=torch.bfloat16, device="cuda").permute(0, 2, 1, 3)
        for _ in range(max(args.warmup, 3)):
            S.sage_prep_qkv(q, k, v, bufs, *lens)
            S.sage_attn_fwd(bufs, o, *lens)
        torch.cuda.synchronize()
        sampler = ClockSampler(torch.cuda.current_device())
        sampler.start()
        prep_ms, attn_ms = [], []
        for _ in range(K):
            flush.zero_()
            e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            e[0].record()
            S.sage_prep_qkv(q, k, v, bufs, *lens)
            e[1].record()
            S.sage_attn_fwd(bufs, o, *lens)
            e[2].record()
            torch.cuda.synchronize()
            prep_ms.append(e[0].elapsed_time(e[1]))
            attn_ms.append(e[1].elapsed_time(e[2]))
        clocks = sampler.stop()
        if S.sage_get_device_status() != S.SAGE_OK:
            raise RuntimeError(f"device status reports an error on workload {cfg}")
        ops = w.ops()
        pm, am = statistics.median(prep_ms), statistics.median(attn_ms)
        attn_tops = ops / am / 1e9
        abytes = attn_bytes(w)
        line = {"workload": w.name, "config": cfg,
                "shape": {"B": w.B, "H": w.H, "Nq": w.Nq, "Nkv": w.Nkv, "D": w.D, "layout": w.layout,
                          "q_len": w.q_len, "kv_len": w.kv_len},
                "ops": ops, "steps": K, "l2": "flushed by a 256 MB write before every timed step",
                "prep_ms_p50": pm, "attn_ms_p50": am, "step_ms_p50": statistics.median(
                    [a + b for a, b in zip(prep_ms, attn_ms)]),
                "attn_tops": attn_tops, "step_tops": ops / (pm + am) / 1e9,
                "tensor": {"frac_fp8_peak": attn_tops / p8, "frac_mixed_ceiling": attn_tops / mixed,
                           "fp8_peak": p8, "mixed_ceiling": mixed, "basis": f"{src} bf16 burst x2 / x4/3"},
                "attn_hbm": {"algorithmic_bytes": abytes, "achieved": abytes / (am * 1e-3) / 1e9,
                             "peak": hbm, "unit": "GB/s", "frac": abytes / (am * 1e-3) / 1e9 / hbm,
                             "basis": "INT8 Q/K and e4m3 V codes read once, BF16 output written once"},
                "prep_hbm": prep_roofline(w, pm, "three launches: stats+Q, finalize, K+V"),
                "clocks": clocks}
        if not args.no_cpu_baseline:
            if cfg == 4:
                # a bounded sample: 16 heads x 1024 query rows spread over the sequence
                import numpy as np
                tasks = head_tasks(w, [(0, h) for h in range(min(16, w.H))], rows=np.arange(0, w.Nq, 16))
                what = "16 of 24 heads, 1024 query rows each (every 16th), all 16384 keys; each head's full preparation included"
            else:
                tasks = head_tasks(w)
                what = "every (b, h) head, every valid row, preparation included"
            wall, o_ops, n, t_prep, t_att = time_oracle(tasks)
            line["oracle"] = {"seconds": wall, "tops": o_ops / wall / 1e12, "ops": o_ops, "cores": n,
                              "kind": "oracle", "sample": what, "prep_cpu_s": t_prep, "attention_cpu_s": t_att,
                              "gpu_over_oracle": attn_tops / (o_ops / wall / 1e12)}
        print(json.dumps(line), flush=True)
        del phys, q, k, v, bufs, o
        torch.cuda.empty_cache()


def run_latency(args):
    """p50 over many calls of each entry on the single-tile workload; each call
    is timed alone (events around it, a synchronize after)."""
    import torch

    import quantized_exact_attention_gb300 as S
    from quantized_exact_attention_gb300 import build as B
    from quantized_exact_attention_gb300 import workloads as W

    B.build()
    S.load_library()
    w = W.make_config(1)
    phys = w.to("cuda")
    q, k, v = w.views(phys)
    bufs = S.alloc_prep_buffers(w.B, w.H, w.Nq, w.Nkv, "cuda")
    o = torch.empty((w.B, w.Nq, w.H, w.D), dtype=torch.bfloat16, device="cuda").permute(0, 2, 1, 3)
    S.sage_prep_qkv(q, k, v, bufs)
    calls = {"attention (sage_attn_fwd)": lambda: S.sage_attn_fwd(bufs, o),
             "prep + attention (sage_prep_qkv, sage_attn_fwd)": lambda: (S.sage_prep_qkv(q, k, v, bufs),
                                                                        S.sage_attn_fwd(bufs, o)),
             "one call (sage_attention)": lambda: S.sage_attention(q, k, v, o, bufs)}
    n = max(20, args.steps)
    for name, fn in calls.items():
        for _ in range(max(args.warmup, 3)):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(n):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        print(json.dumps({"workload": w.name, "entry": name, "p50_ms": statistics.median(ts),
                          "min_ms": min(ts), "calls": n}), flush=True)
    if S.sage_get_device_status() != S.SAGE_OK:
        raise RuntimeError("device status reports an error")


def main():
    args = parse_args()
    world, rank, local = dist_env()
    if args.latency:
        if rank == 0:
            run_latency(args)
        return
    if args.forms:
        if rank == 0:
            run_forms(args)
        return
    if args.configs is not None:
        if rank == 0:
            args.configs = args.configs or [1, 2, 3, 4, 5]
            run_configs(args)
        return
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    try:
        run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
