"""Benchmark: Top-K block-sparse routed attention, plan + fwd, on one GB300.

A step is one pass of the whole path (pool, route + Top-K + lists, attention
over the lists, dense rows) over one workload, by default the H3-shaped one:
9505 packed tokens (9240 video + 265 context), 56 heads, head dim 128, BF16,
Top-K ratio 0.1, radius 1, dense tail.  Inputs are synthetic (block-clustered
random walks, seeded) and resident in HBM; Q + K + V + O = 545 MB is larger
than the 126 MB L2, so no flush is needed between steps (one extra leg times
the forward with L2 flushed before every call).

The metric is kept-block attention TFLOP/s: 4 * 128 FLOP per (real query
row, kept key) pair, summed over heads, divided by the step time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload tiny|8k|h3|32k|64k]
    python bench.py --op reweight      # Spark virtual summaries instead
    python bench.py --op spark         # Spark merged attention (plan + merged fwd)
    python bench.py --op reblock       # Spark token reblocking (landmark tree) of the H3 keys

``--op reweight`` measures the second operation of the library, the Spark
virtual summaries (sparse_attn_spark_reweight) over the same H3-shaped K/V
with one anchor per head: HBM bytes per second against the measured copy
bandwidth (K and V read once; summaries written).

Rank 0 prints one JSON line.  With N > 1 (torchrun), the heads are split
into N contiguous slices, one per rank (heads are independent: no collective
in the data path), so the job does the workload once ("scaling": "strong");
the timing is the max over ranks.  ``--impl reference`` times the CPU fp64
oracle on the host cores.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import multiprocessing as mp
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "kept-block attention TFLOP/s and ms/call at 9505 tok × 56 heads; % BF16 peak"
WORKLOAD = "h3"
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "attention_kernel_h3.md")
ATTN_SOURCE = os.path.join(ROOT, "block_sparse_routed_gb300", "csrc", "attn_kernel.cu")


# ----------------------------------------------------------------- helpers
def kept_pairs_from_lists(idx, cnt, T, nvk, nq, Nv, dense_row_start):
    """Kept (query row, key) pairs given the block lists (host count)."""
    cnt = cnt.reshape(-1, nq)
    H = cnt.shape[0]
    idx = idx.reshape(H, nq, -1)
    blk_len = np.minimum(64, T - 64 * np.arange((T + 63) // 64))
    total = 0
    for i in range(nq):
        rows = 64 if i < nvk else Nv - 64 * nvk
        for h in range(H):
            lst = idx[h, i, : cnt[h, i]]
            total += rows * int(blk_len[lst].sum())
    total += H * (T - dense_row_start) * T
    return total


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def profile_traffic():
    """Per-launch DRAM bytes of the attention kernel from the committed ncu
    summary, or None when the kernel source changed since it was taken."""
    if not os.path.exists(PROFILE_SUMMARY):
        return None
    txt = open(PROFILE_SUMMARY).read()
    m_t = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", txt)
    m_h = re.search(r"attn_kernel_sha256:\s*([0-9a-f]+)", txt)
    if not (m_t and m_h):
        return None
    cur = hashlib.sha256(open(ATTN_SOURCE, "rb").read()).hexdigest()
    if not cur.startswith(m_h.group(1)):
        return None
    return int(m_t.group(1))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- CPU oracle legs
def _oracle_worker(args):
    """Times the oracle on one head slice (runs in a spawned process)."""
    q, k, v, bias, prm = args
    import oracle as O

    sz = O.derive_sizes(prm["T"], q.shape[1], prm["video_tokens"], prm["topk_ratio"],
                        prm["radius"], prm["tail_mode"])
    t0 = time.perf_counter()
    ref = O.plan(q, k, sz)
    O.forward(q, k, v, bias, ref["idx"], ref["cnt"], sz)
    dt = time.perf_counter() - t0
    return O.kept_flops(ref["idx"], ref["cnt"], sz), dt


def _oracle_pool(ncores):
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"  # one BLAS thread per worker process
    return mp.get_context("spawn").Pool(ncores)


def oracle_timing(pool, arrays, prm, heads_per_task, ncores, heads):
    """Wall time of the oracle over `heads` (a list of head indices), spread
    over the pool; returns (kept_flops, seconds)."""
    tasks = []
    for i in range(0, len(heads), heads_per_task):
        hs = heads[i:i + heads_per_task]
        tasks.append((np.ascontiguousarray(arrays["q"][:, hs]), np.ascontiguousarray(arrays["k"][:, hs]),
                      np.ascontiguousarray(arrays["v"][:, hs]), arrays["bias"], prm))
    t0 = time.perf_counter()
    res = pool.map(_oracle_worker, tasks, chunksize=1)
    wall = time.perf_counter() - t0
    return sum(r[0] for r in res), wall


# ----------------------------------------------------------------- ranks
def max_over_ranks(x, world, device):
    """The largest of every rank's `x` (a float); the identity on one rank.
    The job's time is its slowest rank's."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(kept_flop_per_rank, ms_per_step, world):
    """Whole-job kept TFLOP/s when every rank runs its own copy of the
    workload: the job does `world` copies in the slowest rank's step time."""
    return world * kept_flop_per_rank / (ms_per_step * 1e-3) / 1e12


def head_range(H, rank, world):
    """The contiguous heads [h0, h1) of `rank` when H heads are split over
    `world` ranks (sizes differ by at most one, larger slices first)."""
    base, extra = divmod(H, world)
    h0 = rank * base + min(rank, extra)
    return h0, h0 + base + (1 if rank < extra else 0)


def split_heads(arrays, h0, h1):
    """This rank's inputs: the heads [h0, h1) of Q, K, V ([T, H, 128] BF16
    bits) as contiguous arrays; the key bias is per key and shared."""
    out = dict(arrays)
    for n in ("q", "k", "v"):
        out[n] = np.ascontiguousarray(arrays[n][:, h0:h1])
    return out


def strong_scaling_value(kept_flop_total, ms_per_step):
    """Whole-job kept TFLOP/s when the ranks split one workload: all of its
    kept work in the slowest rank's step time."""
    return kept_flop_total / (ms_per_step * 1e-3) / 1e12


def step_stats(ms):
    """Median, 10th and 90th percentile of per-step times (ms)."""
    a = np.asarray(ms, dtype=np.float64)
    return {"median": float(np.median(a)), "p10": float(np.percentile(a, 10)),
            "p90": float(np.percentile(a, 90)), "mean": float(a.mean())}


# ----------------------------------------------------------------- main legs
def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args, rank, world):
    """The oracle as it stands, timed on the host cores (rank 0 only)."""
    if rank != 0:
        return
    from workloads import make_workload

    name = getattr(args, "workload", WORKLOAD)
    arrays, prm = make_workload(name)
    ncores = host_cores()
    pool = _oracle_pool(ncores)
    H = prm["H"]
    sample_heads = list(range(min(H, ncores)))  # one head per core per step
    try:
        for _ in range(args.warmup):
            oracle_timing(pool, arrays, prm, 1, ncores, sample_heads[:1])
        flops, secs = 0, 0.0
        for _ in range(args.steps):
            f, s = oracle_timing(pool, arrays, prm, 1, ncores, sample_heads)
            flops += f
            secs += s
    finally:
        pool.close()
        pool.join()
    value = flops / secs / 1e12
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": args.gpus,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True,
        "scaling": "strong",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(prm, name),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": ncores, "kind": "oracle",
                         "sample": f"{len(sample_heads)} of {H} heads per step, all rows"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


WORKLOAD_TEXT = {
    "tiny": "tiny: 1024 video + 128 context tokens, 2 heads, i.i.d. inputs",
    "8k": "8192 video + 512 context tokens, 24 heads, block-clustered, zero key bias",
    "h3": "H3-shaped packed video sequence (9240 video + 265 context tokens)",
    "32k": "32768 video + 1024 context tokens, 40 heads, block-clustered, biased sinks",
    "64k": "65560 video (pad tail) + 2048 context tokens, 24 heads, 3-D clustered, biased sinks",
}


def workload_config(prm, name=WORKLOAD):
    qkvo = 4 * prm["T"] * prm["H"] * 128 * 2
    l2 = ("inputs larger than L2 (Q+K+V+O %d MB > 126 MB), no flush" % (qkvo // 10**6) if qkvo > 126e6
          else "inputs smaller than L2 (Q+K+V+O %d MB): L2 flushed before every step" % (qkvo // 10**6))
    return {
        "workload": WORKLOAD_TEXT[name],
        "T": prm["T"],
        "H": prm["H"],
        "head_dim": 128,
        "video_tokens": prm["video_tokens"],
        "topk_ratio": prm["topk_ratio"],
        "radius": prm["radius"],
        "tail_mode": prm["tail_mode"],
        "key_bias": None if prm.get("bias_kind", "none") == "none" else prm["bias_kind"],
        "l2": l2,
    }


def _oracle_one_core(args):
    """The oracle on a few heads in one process with one BLAS thread (runs in
    a spawned process); returns (kept_flops, seconds)."""
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    return _oracle_worker(args)


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import block_sparse_routed_gb300 as bsr
    from workloads import make_workload

    # CPU baseline pools first: spawned before the first GPU call.
    pool = pool1 = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        pool = _oracle_pool(host_cores())
        pool1 = mp.get_context("spawn").Pool(1)

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    bsr.load_library()
    name = args.workload
    arrays_all, prm = make_workload(name)
    T, H, Nv = prm["T"], prm["H"], prm["video_tokens"]
    # this rank's heads (all of them on one GPU)
    h0, h1 = head_range(H, rank, world)
    arrays = split_heads(arrays_all, h0, h1)
    Hr = h1 - h0
    P = bsr.Params(T=T, H=Hr, video_tokens=Nv, topk_ratio=prm["topk_ratio"], radius=prm["radius"],
                   tail_mode=prm["tail_mode"])
    sz = bsr.sparse_attn_query(P)

    def pinned(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).reshape(1, T, Hr, 128).pin_memory()

    hq, hk, hv = pinned(arrays["q"]), pinned(arrays["k"]), pinned(arrays["v"])
    q, k, v = hq.to(dev), hk.to(dev), hv.to(dev)
    bias = None
    if arrays["bias"] is not None:
        hbias = torch.from_numpy(arrays["bias"]).pin_memory()
        bias = hbias.to(dev)
    idx = torch.empty((1, Hr, sz.nq, sz.maxl), dtype=torch.int32, device=dev)
    cnt = torch.empty((1, Hr, sz.nq), dtype=torch.int32, device=dev)
    o = torch.empty_like(q)
    ws_plan = torch.empty(sz.plan_ws_bytes, dtype=torch.uint8, device=dev)
    ws_fwd = torch.empty(sz.fwd_ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    # small workloads fit in L2: flush it between steps (writes of a buffer
    # larger than L2, outside the timed events)
    qkvo = 4 * T * Hr * 128 * 2
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if qkvo <= 126e6 else None

    def step():
        bsr.sparse_attn_plan(P, q, k, idx=idx, cnt=cnt, ws=ws_plan, stream=stream)
        bsr.sparse_attn_fwd(P, q, k, v, idx, cnt, key_bias=bias, o=o, ws=ws_fwd, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    st = bsr.sparse_attn_last_device_status(ws_fwd, stream)
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")
    kept_mine = kept_pairs_from_lists(idx.cpu().numpy(), cnt.cpu().numpy(), T, sz.nvk, sz.nq, Nv,
                                      sz.dense_row_start) * 4 * 128
    # the whole job's kept work (every rank's heads)
    if world > 1:
        t = torch.tensor([float(kept_mine)], dtype=torch.float64, device=dev)
        dist.all_reduce(t)
        kept = float(t.item())
    else:
        kept = float(kept_mine)

    def barrier():
        if world > 1:
            dist.barrier()

    # ---- device-resident timing: per-step events split plan / fwd
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(local_rank if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for s_ in range(args.steps):
        if flush is not None:
            flush.fill_(s_ & 0xFF)
        ev[s_][0].record(stream)
        bsr.sparse_attn_plan(P, q, k, idx=idx, cnt=cnt, ws=ws_plan, stream=stream)
        ev[s_][1].record(stream)
        bsr.sparse_attn_fwd(P, q, k, v, idx, cnt, key_bias=bias, o=o, ws=ws_fwd, stream=stream)
        ev[s_][2].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    barrier()
    plan_ms = [ev[s_][0].elapsed_time(ev[s_][1]) for s_ in range(args.steps)]
    fwd_ms = [ev[s_][1].elapsed_time(ev[s_][2]) for s_ in range(args.steps)]
    step_ms = [a_ + b_ for a_, b_ in zip(plan_ms, fwd_ms)]
    total_ms = t_start.elapsed_time(t_end) if flush is None else sum(step_ms)
    if bsr.sparse_attn_last_device_status(ws_fwd, stream) != 0:
        raise RuntimeError("device status error in the timed region")
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / args.steps
    value = strong_scaling_value(kept, ms_per_step)

    # ---- one cold-L2 leg: the forward with L2 flushed before every call
    cold = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    cold_ms = []
    for i in range(max(10, min(args.steps, 50))):
        cold.fill_(i & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        bsr.sparse_attn_fwd(P, q, k, v, idx, cnt, key_bias=bias, o=o, ws=ws_fwd, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        cold_ms.append(e0.elapsed_time(e1))
    del cold

    # ---- end to end through the public API, host buffers.  Every step copies
    # its inputs in from pinned host memory and its output back; steps are
    # pipelined over two buffer sets and three streams (copy in, compute,
    # copy out), so step i+1's inputs travel while step i computes.
    h2d = 3 * T * Hr * 128 * 2 + (T * 4 if bias is not None else 0)
    d2h = T * Hr * 128 * 2
    s_in, s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    sets = []
    for _ in range(2):
        sets.append(dict(
            q=torch.empty_like(q), k=torch.empty_like(k), v=torch.empty_like(v),
            bias=None if bias is None else torch.empty_like(bias), o=torch.empty_like(q),
            idx=torch.empty_like(idx), cnt=torch.empty_like(cnt),
            wp=torch.empty_like(ws_plan), wf=torch.empty_like(ws_fwd),
            ho=torch.empty((1, T, Hr, 128), dtype=torch.bfloat16).pin_memory(),
            ev_in=torch.cuda.Event(), ev_comp=torch.cuda.Event(), ev_out=torch.cuda.Event()))

    def e2e_step(i):
        st_ = sets[i % 2]
        with torch.cuda.stream(s_in):
            s_in.wait_event(st_["ev_comp"])  # step i-2 has read this set's inputs
            st_["q"].copy_(hq, non_blocking=True)
            st_["k"].copy_(hk, non_blocking=True)
            st_["v"].copy_(hv, non_blocking=True)
            if bias is not None:
                st_["bias"].copy_(hbias, non_blocking=True)
            st_["ev_in"].record(s_in)
        s_comp.wait_event(st_["ev_in"])
        s_comp.wait_event(st_["ev_out"])  # step i-2's output has left this set
        bsr.sparse_attn_plan(P, st_["q"], st_["k"], idx=st_["idx"], cnt=st_["cnt"], ws=st_["wp"], stream=s_comp)
        bsr.sparse_attn_fwd(P, st_["q"], st_["k"], st_["v"], st_["idx"], st_["cnt"], key_bias=st_["bias"],
                            o=st_["o"], ws=st_["wf"], stream=s_comp)
        st_["ev_comp"].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(st_["ev_comp"])
            st_["ho"].copy_(st_["o"], non_blocking=True)
            st_["ev_out"].record(s_out)

    for i in range(2):
        e2e_step(i)
    barrier()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(args.steps):
        e2e_step(i)
    for st_ in sets:
        s_out.wait_event(st_["ev_out"])
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    for st_ in sets:
        if bsr.sparse_attn_last_device_status(st_["wf"], s_comp) != 0:
            raise RuntimeError("device status error in the end-to-end run")
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
    e2e_value = strong_scaling_value(kept, e2e_ms)
    # the whole job's copies (every rank's heads)
    h2d_all = 3 * T * H * 128 * 2 + (T * 4 * world if bias is not None else 0)
    d2h_all = T * H * 128 * 2

    if rank != 0:
        return

    peaks, peak_kind = measured_peaks()
    fwd_avg = sum(fwd_ms) / len(fwd_ms)
    achieved = kept_mine / (fwd_avg * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": profile_traffic() if name == WORKLOAD and world == 1 else None,
                "kernel": "attention_kernel (fwd call: status memset + attention)",
                "peak_kind": f"{peak_kind} bf16 burst"}

    cpu = cpu1 = None
    if pool is not None:
        try:
            heads = list(range(H))
            flops_c, secs_c = oracle_timing(pool, arrays_all, prm, 1, host_cores(), heads)
            cpu = {"value": flops_c / secs_c / 1e12, "unit": "TFLOP/s", "cores": host_cores(),
                   "kind": "oracle", "seconds": secs_c,
                   "sample": f"whole workload ({H} heads, all rows), one head per task, "
                             f"one BLAS thread per worker"}
            # one core: a bounded sample of whole heads, one process, one BLAS thread
            nh1 = 1 if T > 20000 else 2
            hs = list(range(nh1))
            f1, s1 = pool1.apply(_oracle_one_core, ((np.ascontiguousarray(arrays_all["q"][:, hs]),
                                                      np.ascontiguousarray(arrays_all["k"][:, hs]),
                                                      np.ascontiguousarray(arrays_all["v"][:, hs]),
                                                      arrays_all["bias"], prm),))
            cpu1 = {"value": f1 / s1 / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle", "seconds": s1,
                    "sample": f"{nh1} of {H} heads, all rows, one process, one BLAS thread"}
        finally:
            pool.close()
            pool.join()
            pool1.close()
            pool1.join()

    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "strong",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": dict(workload_config(prm, name),
                       **({"parallelism": f"heads split over {world} ranks"} if world > 1 else {})),
        "plan_ms": sum(plan_ms) / len(plan_ms),
        "fwd_ms": fwd_avg,
        "step_ms_stats": step_stats(step_ms),
        "fwd_ms_stats": step_stats(fwd_ms),
        "plan_ms_stats": step_stats(plan_ms),
        "fwd_ms_cold_l2": step_stats(cold_ms),
        "kept_tflop_per_step": kept / 1e12,
        "frac_of_bf16_peak": value / world / peak,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "cpu_baseline_1core": cpu1,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d_all,
                "d2h_bytes_per_step": d2h_all, "ms_per_step": e2e_ms,
                "pipeline": "2 buffer sets, copy-in / compute / copy-out streams"},
        "gpu_launches": args.steps * (3 + (1 if bias is not None else 0)),  # pool, route, attention (+ bias prep)
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def _reweight_worker(args):
    a, k, v = args
    import oracle as O

    t0 = time.perf_counter()
    O.spark_reweight(a, k, v)
    return time.perf_counter() - t0


def _reblock_worker(args):
    x, fanout = args
    from oracle import reblock as R

    t0 = time.perf_counter()
    R.reblock_head(x, fanout)
    return time.perf_counter() - t0


def reblock_bytes(T, H):
    """Samples read once (BF16) plus the permutation and its inverse (int32)."""
    return T * H * 256 + 2 * T * H * 4


def reblock_depth(m, fanout):
    if m <= 1:
        return 0
    c = 1
    while c * 2 <= min(fanout, m):
        c *= 2
    lo = reblock_depth(m // c, fanout)
    hi = reblock_depth(m // c + 1, fanout) if m % c else lo
    return 1 + max(lo, hi)


def run_reblock(args, rank, world, local_rank):
    """Spark token reblocking of the H3 keys: algorithmic HBM bytes per second."""
    import torch

    import block_sparse_routed_gb300 as bsr
    from workloads import make_workload

    arrays, prm = make_workload(WORKLOAD)
    T, H = prm["T"], prm["H"]
    fanout = 8
    pool = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        pool = _oracle_pool(host_cores())
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    bsr.load_library()
    hx = torch.from_numpy(np.ascontiguousarray(arrays["k"]).view(np.int16)).view(torch.bfloat16).reshape(T, H, 128).pin_memory()
    x = hx.to(dev)
    perm = torch.empty((H, T), dtype=torch.int32, device=dev)
    inv = torch.empty_like(perm)
    from block_sparse_routed_gb300 import _native

    rp = _native.SaReblockParams(_native.SA_ABI_VERSION, T, H, 128, fanout, 32, x.stride(0), x.stride(1))
    ws = torch.empty(max(_native.sparse_attn_reblock_ws_bytes(rp), 1), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        bsr.spark_reblock(x, fanout=fanout, perm=perm, inv=inv, ws=ws, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    nbytes = reblock_bytes(T, H)
    clocks = ClockSampler(local_rank if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for e0, e1 in ev:
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    per = [e0.elapsed_time(e1) for e0, e1 in ev]
    ms = max_over_ranks(sum(per) / len(per), world, dev)
    value = world * nbytes / (ms * 1e-3) / 1e9

    hperm = torch.empty((H, T), dtype=torch.int32).pin_memory()
    hinv = torch.empty_like(hperm).pin_memory()

    def e2e_step():
        x.copy_(hx, non_blocking=True)
        step()
        hperm.copy_(perm, non_blocking=True)
        hinv.copy_(inv, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
    if rank != 0:
        return
    peaks, peak_kind = measured_peaks()
    peak = float(peaks["hbm_gbs"])
    cpu = None
    if pool is not None:
        try:
            hs = list(range(H))
            tasks = [(np.ascontiguousarray(arrays["k"][:, h, :]), fanout) for h in hs]
            t0 = time.perf_counter()
            cpu_secs = sum(pool.map(_reblock_worker, tasks, chunksize=1))
            secs = time.perf_counter() - t0
            cpu = {"value": reblock_bytes(T, len(hs)) / secs / 1e9, "unit": "GB/s", "cores": host_cores(),
                   "kind": "oracle", "seconds": secs, "cpu_seconds": cpu_secs,
                   "sample": f"all {H} heads, all tokens, one head per task"}
        finally:
            pool.close()
            pool.join()
    depth = reblock_depth(T // 64, fanout)
    line = {
        "metric": "spark_reblock HBM GB/s (landmark-tree token reblocking of the H3 keys)",
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp32",
        "data": "synthetic",
        "config": {"workload": "Spark reblocking of the H3 keys (9505 tokens x 56 heads, 128 dims), "
                               "fanout 8, 32 landmarks", "T": T, "H": H, "fanout": fanout, "landmarks": 32,
                   "levels": depth, "l2": "samples 136 MB > 126 MB L2, no flush"},
        "roofline": {"bound": "hbm", "achieved": value, "peak": peak, "unit": "GB/s", "frac": value / peak,
                     "traffic": None, "kernel": f"whole call ({3 * depth + 2} launches)",
                     "peak_kind": f"{peak_kind} copy bandwidth"},
        "cpu_baseline": cpu,
        "e2e": {"value": world * nbytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": T * H * 256, "d2h_bytes_per_step": 2 * T * H * 4, "ms_per_step": e2e_ms},
        "gpu_launches": args.steps * (3 * depth + 2),
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def reweight_bytes(P, T, H):
    nblk = (T + 63) // 64
    return 2 * T * H * 256 + P * H * 256 + P * H * nblk * (2 * 256 + 4)


def run_reweight(args, rank, world, local_rank):
    """Spark virtual summaries: algorithmic HBM bytes per second."""
    import torch

    import block_sparse_routed_gb300 as bsr
    from workloads import make_reweight_workload

    name = "reweight_h3"
    arrays, prm = make_reweight_workload(name)
    T, H, P = prm["T"], prm["H"], prm["P"]
    nblk = (T + 63) // 64
    pool = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        pool = _oracle_pool(host_cores())
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    bsr.load_library()

    def pinned(bits, shape):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).reshape(shape).pin_memory()

    ha, hk, hv = pinned(arrays["a"], (1, P, H, 128)), pinned(arrays["k"], (1, T, H, 128)), pinned(arrays["v"], (1, T, H, 128))
    a, k, v = ha.to(dev), hk.to(dev), hv.to(dev)
    ak = torch.empty((1, P, H, nblk, 128), dtype=torch.bfloat16, device=dev)
    av = torch.empty_like(ak)
    lm = torch.empty((1, P, H, nblk), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        bsr.spark_reweight(a, k, v, ak=ak, av=av, lm=lm, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    nbytes = reweight_bytes(P, T, H)
    clocks = ClockSampler(local_rank if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for e0, e1 in ev:
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    per = [e0.elapsed_time(e1) for e0, e1 in ev]
    ms = max_over_ranks(sum(per) / len(per), world, dev)
    value = world * nbytes / (ms * 1e-3) / 1e9

    hak = torch.empty((1, P, H, nblk, 128), dtype=torch.bfloat16).pin_memory()
    hav = torch.empty_like(hak).pin_memory()
    hlm = torch.empty((1, P, H, nblk), dtype=torch.float32).pin_memory()

    def e2e_step():
        a.copy_(ha, non_blocking=True)
        k.copy_(hk, non_blocking=True)
        v.copy_(hv, non_blocking=True)
        step()
        hak.copy_(ak, non_blocking=True)
        hav.copy_(av, non_blocking=True)
        hlm.copy_(lm, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
    if rank != 0:
        return
    peaks, peak_kind = measured_peaks()
    peak = float(peaks["hbm_gbs"])
    cpu = None
    if pool is not None:
        try:
            hs = list(range(min(H, host_cores())))
            tasks = [(np.ascontiguousarray(arrays["a"][:, [h]]), np.ascontiguousarray(arrays["k"][:, [h]]),
                      np.ascontiguousarray(arrays["v"][:, [h]])) for h in hs]
            t0 = time.perf_counter()
            pool.map(_reweight_worker, tasks, chunksize=1)
            secs = time.perf_counter() - t0
            cpu = {"value": reweight_bytes(P, T, len(hs)) / secs / 1e9, "unit": "GB/s", "cores": host_cores(),
                   "kind": "oracle", "seconds": secs,
                   "sample": f"{len(hs)} of {H} heads, all blocks, one head per task"}
        finally:
            pool.close()
            pool.join()
    line = {
        "metric": "spark_reweight HBM GB/s (virtual summaries, H3-shaped K/V, 1 anchor per head)",
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "Spark virtual summaries over H3-shaped K/V (9505 tokens x 56 heads), "
                               "1 anchor per head", "T": T, "H": H, "P": P, "blocks": nblk,
                   "l2": "K+V 272 MB > 126 MB L2, no flush"},
        "roofline": {"bound": "hbm", "achieved": value, "peak": peak, "unit": "GB/s", "frac": value / peak,
                     "traffic": None, "kernel": "spark_reweight_kernel",
                     "peak_kind": f"{peak_kind} copy bandwidth"},
        "cpu_baseline": cpu,
        "e2e": {"value": world * nbytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": (2 * T * H + P * H) * 256,
                "d2h_bytes_per_step": P * H * nblk * (2 * 256 + 4), "ms_per_step": e2e_ms},
        "gpu_launches": args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def run_spark(args, rank, world, local_rank):
    """Spark's merged attention on the H3 workload: plan + merged forward
    (anchor, summaries, exact lists plus one summary key per skipped video
    block).  Reports the step time; the TFLOP/s figure counts the same kept
    exact work as the headline plus 4 x 128 FLOP per (row, summary key)."""
    import torch

    import block_sparse_routed_gb300 as bsr
    from block_sparse_routed_gb300 import _native
    from workloads import make_workload

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    bsr.load_library()
    arrays, prm = make_workload(WORKLOAD)
    T, H, Nv = prm["T"], prm["H"], prm["video_tokens"]
    P = bsr.Params(T=T, H=H, video_tokens=Nv, topk_ratio=prm["topk_ratio"], radius=prm["radius"],
                   tail_mode=prm["tail_mode"])
    sz = bsr.sparse_attn_query(P)
    dv = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).reshape(1, T, H, 128).to(dev)
    q, k, v = dv(arrays["q"]), dv(arrays["k"]), dv(arrays["v"])
    idx = torch.empty((1, H, sz.nq, sz.maxl), dtype=torch.int32, device=dev)
    cnt = torch.empty((1, H, sz.nq), dtype=torch.int32, device=dev)
    o = torch.empty_like(q)
    ws_plan = torch.empty(sz.plan_ws_bytes, dtype=torch.uint8, device=dev)
    ws = torch.empty(_native.sparse_attn_spark_ws_bytes(P.to_c()), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        bsr.sparse_attn_plan(P, q, k, idx=idx, cnt=cnt, ws=ws_plan, stream=stream)
        bsr.sparse_attn_spark_fwd(P, q, k, v, idx, cnt, o=o, ws=ws, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    if bsr.sparse_attn_last_device_status(ws, stream) != 0:
        raise RuntimeError("device status error after warm-up")
    ic, cc = idx.cpu().numpy().reshape(H, sz.nq, sz.maxl), cnt.cpu().numpy().reshape(H, sz.nq)
    kept = kept_pairs_from_lists(idx.cpu().numpy(), cnt.cpu().numpy(), T, sz.nvk, sz.nq, Nv,
                                 sz.dense_row_start) * 4 * 128
    summary_keys = 0
    for h in range(H):
        for i in range(sz.nq):
            listed = int(np.count_nonzero(ic[h, i, :cc[h, i]] < sz.nvk))
            rows = min(64, Nv - 64 * i) if i == sz.nvk else 64
            summary_keys += rows * (sz.nvk - listed)
    work = kept + summary_keys * 4 * 128
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    for s in range(args.steps):
        ev[s][0].record(stream)
        bsr.sparse_attn_plan(P, q, k, idx=idx, cnt=cnt, ws=ws_plan, stream=stream)
        ev[s][1].record(stream)
        bsr.sparse_attn_spark_fwd(P, q, k, v, idx, cnt, o=o, ws=ws, stream=stream)
        ev[s][2].record(stream)
    torch.cuda.synchronize(dev)
    plan_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps
    fwd_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / args.steps
    ms = max_over_ranks(plan_ms + fwd_ms, world, dev)
    if rank != 0:
        return
    line = {
        "metric": "Spark merged attention TFLOP/s (exact lists + one summary key per skipped block), H3",
        "value": weak_scaling_value(work, ms, world),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "plan_ms": plan_ms,
        "fwd_ms": fwd_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": dict(workload_config(prm), summary_keys_per_step=summary_keys),
        "work_tflop_per_step": work / 1e12,
        "exact_kept_tflop_per_step": kept / 1e12,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--op", choices=["attention", "reweight", "spark", "reblock"], default="attention")
    ap.add_argument("--workload", choices=["tiny", "8k", "h3", "32k", "64k"], default=WORKLOAD)
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        if args.op == "reweight":
            run_reweight(args, rank, world, local_rank)
        elif args.op == "spark":
            run_spark(args, rank, world, local_rank)
        elif args.op == "reblock":
            run_reblock(args, rank, world, local_rank)
        else:
            run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
