"""Benchmark of the paged-attention hot path on GB300.

Headline (one JSON line on rank 0): split-KV paged decode on the pages' decode
microbench shape -- B=32, GQA 32/8, head_dim 128, seq_lens uniform in [200, 2000],
page_size=1 random slot table, bf16 -- reported as K+V bytes read per second (GB/s),
microseconds per call and the fraction of the measured HBM copy bandwidth.  A step is
one decode call (split kernel + combine kernel) through the C ABI on inputs already in
HBM.  L2 is defeated by rotating through several copies of the KV pools (working set
well above the 126 MB L2), so every call reads its keys from DRAM.  Each timed region
starts with the GPU busy (a short spin kernel queued before the start event), so the host's
latency to launch the first call is not counted; the e2e object counts everything.  The timed region of
`--steps` calls runs `--repeats` times (each between a barrier and a synchronize); the
line reports the median region and the spread of all of them.

Also reported in the same line:
  * roofline     -- the split kernel alone (the dominant kernel), timed with CUDA events
                    on its stream: algorithmic K+V bytes per launch / mean duration;
                    stable_indices: the same, and the call, with ASTR_DIMS_STABLE_INDICES
                    (chunks planned before the dependency wait; valid here: the index arrays
                    are never written between calls).
  * prefill      -- the ragged prefill entry point on the 16-request extend workload,
                    FLOP/s against the measured dense bf16 tensor-core peak (rotating
                    query / pool / output copies, so each call is cold in L2), with the
                    batch's host work plan attached (made once outside the timed region, as a
                    serving step makes it once for all layers); us_per_call_unplanned is the
                    same call without a plan (the kernel orders the work itself),
                    us_per_call_graph the planned calls replayed from a CUDA graph.
  * decode_workloads -- the other decode workloads (B=4 d=64 tiny, B=8 long context, B=256
                    large batch): us per call, K+V GB/s and the fraction of the copy peak.
  * masked       -- the explicit-mask entry points on the same workloads: prefill with a 3-D
                    mask (causal on) and decode with a 2-D mask, each byte kept with
                    probability 0.75; FLOP/s and GB/s count the same work as the unmasked calls
                    (masked keys are still read and scored).
  * contiguous   -- decode over a contiguous "bhld" K/V cache (stride addressing, no slot
                    table; 2 rotating copies) and prefill over a "blhd" cache, same workloads.
  * kv_append    -- the KV-append step (the extend workload's new K/V rows written into their
                    pool slots), bytes moved per second against the measured HBM copy peak.
  * e2e          -- the same decode metric with every input in pinned host memory, the
                    host->device copies and the device->host read of `out` inside the
                    timed region (and a variant where only q and the index arrays move).
  * cpu_baseline -- the fp64 CPU oracle timed on this host on a bounded sample (decode: whole
                    batches; prefill_cpu_baseline: a sample of (query row, head) rows).

--impl reference times the fp64 oracle (the only reference implementation this build
has) on the same workload and prints the same line with "impl": "reference".
Multi-GPU (torchrun): every rank runs its own replica (weak scaling); the elapsed time is
the max over ranks and value sums all ranks' bytes.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workload  # noqa: E402

METRIC = "paged decode KV GB/s (fraction of HBM peak) & us/call, B=32 GQA 32/8 d128"
DECODE_CFG = 2
PREFILL_CFG = 5
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
POOL_COPIES = 4          # rotate KV-pool copies so each call's working set is cold in L2
                         # (fewer when one pool alone is several times the L2)
MAX_SPLITS = 64
SPIN_CYCLES = 1_000_000  # GPU clock cycles of the pre-region spin (~0.5 ms at 2 GHz)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"]))}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def prefill_flops(w) -> float:
    """Causal-attended (query, key) pairs x 4 d Hq (QK^T and PV, 2 FLOP per MAC)."""
    ql = w.q_lens.astype(np.int64)
    c = w.seq_lens.astype(np.int64) - ql
    pairs = int((ql * c + ql * (ql + 1) // 2).sum())
    return 4.0 * w.head_dim * w.num_qo_heads * pairs


def decode_bytes(w) -> dict:
    kv = w.kv_bytes()
    idx = 4 * int(w.seq_lens.sum()) + 8 * w.batch
    qo = 2 * 2 * w.batch * w.num_qo_heads * w.head_dim
    return {"kv": kv, "all": kv + idx + qo}


# ------------------------------------------------------------------ traffic record


def source_digest(path: str) -> str:
    """sha-256 (first 16 hex digits) of a CUDA source with comments and whitespace removed, so
    that a counter record survives comment edits but not code changes."""
    import re
    with open(path, "r") as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    text = re.sub(r"\s+", "", text)
    return hashlib.sha256(text.encode()).hexdigest()[:16]


def recorded_traffic(kernel: str, source: str):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken on this source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel)
    if not rec:
        return None
    if rec.get("source_digest") != source_digest(os.path.join(ROOT, "prefill_attention_gb300", "csrc", source)):
        return None
    return rec.get("bytes_per_launch")


# ------------------------------------------------------------------ multi-rank aggregation


def rank_reduce(dist, x: float, op: str, device=None) -> float:
    """Reduce one float over ranks ("max" or "sum"); identity without a process group."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def aggregate_weak(dist, elapsed_s: float, units: float, device=None):
    """Weak scaling: job time = slowest rank, job work = every rank's units."""
    t = rank_reduce(dist, elapsed_s, "max", device)
    u = rank_reduce(dist, units, "sum", device)
    return t, u, (u / t if t > 0 else 0.0)


# ------------------------------------------------------------------ clocks


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")  # removed again by stop()
        os.close(fd)

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.dev), "-lms", "50"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            if getattr(self, "fh", None) is not None:
                self.fh.close()
            try:
                os.remove(self.path)
            except OSError:
                pass
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        try:
            os.remove(self.path)
        except OSError:
            pass
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ reference arm (oracle)


def oracle_gbs(w, seconds: float, nthreads: int):
    """Time the fp64 oracle on whole-batch decode calls for ~`seconds`; GB/s of K+V."""
    import oracle
    oracle.build()
    t0 = time.perf_counter()
    oracle.decode(w, nthreads=nthreads)  # one call also warms caches
    one = time.perf_counter() - t0
    reps = max(1, int(seconds / max(one, 1e-3)))
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.decode(w, nthreads=nthreads)
    dt = (time.perf_counter() - t0) / reps
    return w.kv_bytes() / dt / 1e9, dt, reps


def oracle_prefill_tflops(wp, seconds: float, nthreads: int, seed: int = 1):
    """Time the fp64 oracle on a random sample of (flat query row, head) rows of prefill workload
    ``wp`` for ~`seconds`; TFLOP/s counted as for the GPU (4 d per attended (query, key) pair)."""
    import oracle
    oracle.build()
    rng = np.random.default_rng(seed)
    qo = np.asarray(wp.qo_indptr, dtype=np.int64)
    req = np.searchsorted(qo, np.arange(wp.total_q), side="right") - 1
    vis = (wp.seq_lens[req].astype(np.int64) - (qo[req + 1] - qo[req])) + (np.arange(wp.total_q) - qo[req]) + 1

    def sample(n):
        rows = np.stack([rng.integers(0, wp.total_q, n), rng.integers(0, wp.num_qo_heads, n)], 1).astype(np.int32)
        return rows, 4.0 * wp.head_dim * float(vis[rows[:, 0]].sum())

    rows, fl = sample(256)
    t0 = time.perf_counter()
    oracle.prefill(wp, rows=rows, nthreads=nthreads)
    one = max(time.perf_counter() - t0, 1e-4)
    rows, fl = sample(max(256, min(int(256 * seconds / one), 4_000_000)))
    t0 = time.perf_counter()
    oracle.prefill(wp, rows=rows, nthreads=nthreads)
    dt = time.perf_counter() - t0
    return fl / dt / 1e12, rows.shape[0], dt


def run_reference(args, rank: int, world: int):
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = workload.config(args.decode_workload)
    cores = os.cpu_count() or 1
    # each step: the whole B=32 batch (all 1024 (request, head) rows), fp64, all host cores
    for _ in range(args.warmup):
        oracle.decode(w, nthreads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.decode(w, nthreads=cores)
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    val = w.kv_bytes() / dt / 1e9
    line = {
        "impl": "reference",
        "metric": METRIC if args.decode_workload == DECODE_CFG else METRIC.split(", B=")[0] + f", {w.name}",
        "value": round(val, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "seed": w.seed, "sample": "whole batch per step"},
        "cpu_baseline": {"value": round(val, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"whole decode batch ({w.batch} requests x {w.num_qo_heads} heads) per step, fp64 C oracle"},
        "e2e": {"value": round(val, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--repeats", type=int, default=7, help="timed regions of --steps calls (median reported)")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU-baseline sample budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--num-splits", type=int, default=0, help="force the decode split count (0 = planned)")
    ap.add_argument("--decode-workload", type=int, default=DECODE_CFG, choices=[1, 2, 3, 4],
                    help="decode workload of the step (default 2, the headline; 3 = long context, "
                         "4 = large batch are extra measurements, not the headline)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch
    import prefill_attention_gb300 as pa
    from prefill_attention_gb300 import build as pbuild

    pbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    def max_over_ranks(x: float) -> float:
        return rank_reduce(dist, x, "max", dev)

    def sum_over_ranks(x: float) -> float:
        return rank_reduce(dist, x, "sum", dev)

    peaks, peaks_src = load_peaks()

    # ---------------- decode inputs (replica per rank, same seed so every rank does equal work)
    w = workload.config(args.decode_workload)
    nbytes = decode_bytes(w)

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)

    q = bf(w.q)
    n_copies = max(1, min(POOL_COPIES, -(-int(6e8) // max(int(nbytes["kv"]), 1))))
    pools = [(bf(w.k_pool), bf(w.v_pool)) for _ in range(n_copies)]
    r2t, seq, kvi = i32(w.req_to_token), i32(w.seq_lens), i32(w.kv_indptr)
    dims = pa.make_dims(w.batch, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.num_slots, w.r2t_stride,
                        w.max_seq_len, max_splits=MAX_SPLITS, num_splits=args.num_splits)
    S = pa.astr_attn_decode_num_splits(dims, local)
    o_part, ml_part = pa.alloc_decode_workspace(dims, device=dev)
    out = torch.empty_like(q)
    stream = torch.cuda.Stream(device=dev)
    sh = int(stream.cuda_stream)

    def decode(i):
        k, v = pools[i % n_copies]
        pa.astr_attn_paged_decode(q, k, v, r2t, seq, kvi, o_part, ml_part, out, dims, w.sm_scale, stream=sh)

    def split_only(i):
        k, v = pools[i % n_copies]
        pa.astr_attn_decode_split(q, k, v, r2t, seq, kvi, o_part, ml_part, dims, w.sm_scale, stream=sh)

    def timed(fn, n):
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            # a ~0.5 ms spin before the start event keeps the GPU busy while the host queues the
            # first calls, so the region times the calls back to back rather than the host's
            # launch of the first one (outside the region; not one of this library's kernels)
            if hasattr(torch.cuda, "_sleep"):
                torch.cuda._sleep(SPIN_CYCLES)
            ev0.record(stream)
            for i in range(n):
                fn(i)
            ev1.record(stream)
        ev1.synchronize()
        return ev0.elapsed_time(ev1) / 1e3  # seconds

    clocks = ClockSampler(local)
    clocks.start()
    # warm-up (also keeps the GPU loaded ~0.3 s so the clock samples reflect load)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            decode(i)
    stream.synchronize()
    t_end = time.perf_counter() + 0.3
    while time.perf_counter() < t_end:
        timed(decode, 200)

    # ---------------- timed regions: K decode steps each, repeated; the median region counts
    regions = []
    for _ in range(max(1, args.repeats)):
        barrier()
        elapsed = timed(decode, args.steps)
        barrier()
        regions.append(aggregate_weak(dist, elapsed, float(nbytes["kv"]) * args.steps, dev))
    clk = clocks.stop()
    region_us = sorted(r[0] / args.steps * 1e6 for r in regions)
    elapsed_max, total_kv, bytes_per_s = sorted(regions)[len(regions) // 2]
    value = bytes_per_s / 1e9
    us_per_call = elapsed_max / args.steps * 1e6

    # ---------------- the split kernel alone (roofline of the dominant kernel)
    n_split = max(200, min(args.steps, 2000))
    timed(split_only, 20)
    t_split = timed(split_only, n_split) / n_split
    split_gbs = nbytes["kv"] / t_split / 1e9
    # the same with ASTR_DIMS_STABLE_INDICES (the index arrays are never written here, so the
    # split step may plan its chunks before waiting for the preceding kernel), and the call
    sdims = pa.make_dims(w.batch, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.num_slots, w.r2t_stride,
                         w.max_seq_len, max_splits=MAX_SPLITS, num_splits=args.num_splits,
                         flags=pa.ASTR_DIMS_STABLE_INDICES)

    def split_stable(i):
        k, v = pools[i % n_copies]
        pa.astr_attn_decode_split(q, k, v, r2t, seq, kvi, o_part, ml_part, sdims, w.sm_scale, stream=sh)

    def decode_stable(i):
        k, v = pools[i % n_copies]
        pa.astr_attn_paged_decode(q, k, v, r2t, seq, kvi, o_part, ml_part, out, sdims, w.sm_scale, stream=sh)

    timed(split_stable, 20)
    t_split_s = timed(split_stable, n_split) / n_split
    timed(decode_stable, 20)
    t_call_s = timed(decode_stable, n_split) / n_split

    # ---------------- CUDA-graph replay (launch overhead amortised)
    graph_us = None
    try:
        g = torch.cuda.CUDAGraph()
        n_graph = 64
        with torch.cuda.graph(g, stream=stream):
            for i in range(n_graph):
                decode(i)
        g.replay()
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(10):
                g.replay()
            ev1.record(stream)
        ev1.synchronize()
        graph_us = ev0.elapsed_time(ev1) * 1e3 / (10 * n_graph)
        del g
    except Exception as e:  # capture problems are reported, not hidden
        graph_us = f"capture failed: {e}"

    # ---------------- e2e through the public API with host buffers
    def pinned(t):
        h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        h.copy_(t)
        return h

    hq, hk, hv = pinned(q), pinned(pools[0][0]), pinned(pools[0][1])
    hr, hs, hi = pinned(r2t), pinned(seq), pinned(kvi)
    hout = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(pools[0][0]), torch.empty_like(pools[0][1])
    dr, ds, di = torch.empty_like(r2t), torch.empty_like(seq), torch.empty_like(kvi)
    n_e2e = max(5, min(args.steps // 20, 100))

    def e2e_step(full: bool):
        with torch.cuda.stream(stream):
            dq.copy_(hq, non_blocking=True)
            if full:
                dk.copy_(hk, non_blocking=True)
                dv.copy_(hv, non_blocking=True)
            dr.copy_(hr, non_blocking=True)
            ds.copy_(hs, non_blocking=True)
            di.copy_(hi, non_blocking=True)
            k, v = (dk, dv) if full else pools[0]
            pa.astr_attn_paged_decode(dq, k, v, dr, ds, di, o_part, ml_part, out, dims, w.sm_scale, stream=sh)
            hout.copy_(out, non_blocking=True)
        stream.synchronize()

    def e2e_time(full):
        for _ in range(3):
            e2e_step(full)
        barrier()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            e2e_step(full)
        barrier()
        return max_over_ranks((time.perf_counter() - t0) / n_e2e)

    t_e2e_full = e2e_time(True)
    t_e2e_res = e2e_time(False)
    h2d_full = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hr, hs, hi))
    h2d_res = sum(t.numel() * t.element_size() for t in (hq, hr, hs, hi))
    d2h = hout.numel() * hout.element_size()

    # ---------------- the other decode workloads, each timed on its own (one pool copy when it
    # is several times the L2 already)
    decode_workloads = {}
    for cfg in (1, 3, 4):
        if cfg == args.decode_workload:
            continue
        wx = workload.config(cfg)
        bx = decode_bytes(wx)
        nx = max(1, min(POOL_COPIES, -(-int(6e8) // max(int(bx["kv"]), 1))))
        xpools = [(bf(wx.k_pool), bf(wx.v_pool)) for _ in range(nx)]
        xq, xr, xs, xi = bf(wx.q), i32(wx.req_to_token), i32(wx.seq_lens), i32(wx.kv_indptr)
        xdims = pa.make_dims(wx.batch, wx.num_qo_heads, wx.num_kv_heads, wx.head_dim, wx.num_slots, wx.r2t_stride,
                             wx.max_seq_len, max_splits=MAX_SPLITS)
        xo, xm = pa.alloc_decode_workspace(xdims, device=dev)
        xout = torch.empty_like(xq)

        def decode_x(i, xpools=xpools, xq=xq, xr=xr, xs=xs, xi=xi, xdims=xdims, xo=xo, xm=xm, xout=xout, wx=wx,
                     nx=nx):
            k, v = xpools[i % nx]
            pa.astr_attn_paged_decode(xq, k, v, xr, xs, xi, xo, xm, xout, xdims, wx.sm_scale, stream=sh)

        n_x = max(20, min(args.steps, int(0.3 / max(bx["kv"] / 5e12, 2e-6))))
        timed(decode_x, 10)
        t_x = statistics.median(timed(decode_x, n_x) / n_x for _ in range(3))
        rec = {"workload": wx.name, "seed": wx.seed, "us_per_call": round(t_x * 1e6, 3),
               "kv_bytes_per_call": bx["kv"], "gbs": round(bx["kv"] / t_x / 1e9, 2),
               "frac_of_hbm": round(bx["kv"] / t_x / 1e9 / peaks["hbm_gbs"], 4),
               "l2": f"{nx} KV-pool copies ({nx * bx['kv'] / 1e6:.0f} MB)"}
        if cfg == 1:  # launch-bound: the CUDA-graph replay time is the meaningful one
            try:
                gx = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gx, stream=stream):
                    for i in range(64):
                        decode_x(i)
                gx.replay()
                torch.cuda.synchronize()
                ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(stream):
                    ev0.record(stream)
                    for _ in range(10):
                        gx.replay()
                    ev1.record(stream)
                ev1.synchronize()
                rec["us_per_call_graph"] = round(ev0.elapsed_time(ev1) * 1e3 / 640, 3)
                del gx
            except Exception as e:
                rec["us_per_call_graph"] = f"capture failed: {e}"
        decode_workloads[f"workload_{cfg}"] = rec
        del xpools, xo, xm
    torch.cuda.empty_cache()

    # ---------------- prefill entry point on the extend workload (rotating query / pool /
    # output copies: one copy, ~135 MB, is about the L2's size)
    wp = workload.config(PREFILL_CFG)
    n_pcp = 3
    pcopies = [(bf(wp.q), bf(wp.k_pool), bf(wp.v_pool)) for _ in range(n_pcp)]
    pq, pk, pv = pcopies[0]
    pqo, pr, ps_, pki = i32(wp.qo_indptr), i32(wp.req_to_token), i32(wp.seq_lens), i32(wp.kv_indptr)
    pdims = pa.make_dims(wp.batch, wp.num_qo_heads, wp.num_kv_heads, wp.head_dim, wp.num_slots, wp.r2t_stride,
                         wp.max_seq_len, total_q=wp.total_q, max_q_len=wp.max_q_len)
    pouts = [torch.empty_like(pq) for _ in range(n_pcp)]
    pout = pouts[0]
    # the host work plan of this batch, made once outside the timed region (a serving step makes
    # it once per batch and every layer's call reuses it); the call without it is timed as well
    pplan = pa.make_prefill_plan(wp.qo_indptr, wp.seq_lens, pdims)
    udims = pdims
    pdims = pa.attach_prefill_plan(pa.make_dims(wp.batch, wp.num_qo_heads, wp.num_kv_heads, wp.head_dim,
                                                wp.num_slots, wp.r2t_stride, wp.max_seq_len, total_q=wp.total_q,
                                                max_q_len=wp.max_q_len), pplan)

    def prefill_with(dims_):
        def run(i):
            q_, k_, v_ = pcopies[i % n_pcp]
            pa.astr_attn_prefill_ragged(q_, pqo, k_, v_, pr, ps_, pki, pouts[i % n_pcp], dims_, wp.sm_scale,
                                        stream=sh)
        return run

    prefill, prefill_unplanned = prefill_with(pdims), prefill_with(udims)
    timed(prefill, 6)
    timed(prefill_unplanned, 6)
    n_pf = max(21, min(args.steps // 10, 399))
    t_pf = statistics.median(timed(prefill, n_pf) / n_pf for _ in range(3))
    t_pfu = statistics.median(timed(prefill_unplanned, n_pf) / n_pf for _ in range(3))
    # the planned calls replayed from a CUDA graph (a fixed batch's calls are capturable: the
    # plan and every argument stay the same), which removes the per-launch gap of the stream
    try:
        gp = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gp, stream=stream):
            for i in range(30):
                prefill(i)
        gp.replay()
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            torch.cuda._sleep(SPIN_CYCLES)
            ev0.record(stream)
            for _ in range(5):
                gp.replay()
            ev1.record(stream)
        ev1.synchronize()
        t_pfg = ev0.elapsed_time(ev1) * 1e-3 / 150
        del gp
    except Exception as e:  # noqa: BLE001 (reported in the line)
        t_pfg = f"capture failed: {e}"
    flops = prefill_flops(wp)
    pf_tflops = flops / t_pf / 1e12
    pf_copy_mb = (wp.q.nbytes * 2 + wp.k_pool.nbytes * 2) / 1e6

    # ---------------- explicit-mask entry points (prefill: 3-D mask; decode: 2-D mask)
    pmask = torch.from_numpy(workload.make_mask(wp, 3, seed=wp.seed + 7, keep=0.75)).to(dev)
    pm = pa.make_mask(pmask, causal=True)

    def prefill_masked(i):
        q_, k_, v_ = pcopies[i % n_pcp]
        pa.astr_attn_prefill_ragged_masked(q_, pqo, k_, v_, pr, ps_, pki, pm, pouts[i % n_pcp], pdims, wp.sm_scale,
                                           stream=sh)

    timed(prefill_masked, 5)
    t_pfm = timed(prefill_masked, n_pf) / n_pf
    dmask = torch.from_numpy(workload.make_mask(w, 2, seed=w.seed + 7, keep=0.75)).to(dev)
    dm = pa.make_mask(dmask)

    def decode_masked(i):
        k, v = pools[i % n_copies]
        pa.astr_attn_paged_decode_masked(q, k, v, r2t, seq, kvi, dm, o_part, ml_part, out, dims, w.sm_scale,
                                         stream=sh)

    timed(decode_masked, 20)
    t_dm = timed(decode_masked, n_split) / n_split

    # ---------------- contiguous K/V caches (stride addressing instead of the slot table)
    def contiguous(wl, head_major):
        """The workload's K and V rows by request position: [B, L, Hkv, d] views ("bhld" storage
        when head_major)."""
        L = wl.max_seq_len
        kc = np.zeros((wl.batch, L, wl.num_kv_heads, wl.head_dim), np.uint16)
        vc = np.zeros_like(kc)
        for b in range(wl.batch):
            n = int(wl.seq_lens[b])
            sl_ = wl.req_to_token[b, :n].astype(np.int64)
            kc[b, :n], vc[b, :n] = wl.k_pool[sl_], wl.v_pool[sl_]
        if head_major:
            return [bf(a.transpose(0, 2, 1, 3)).transpose(1, 2) for a in (kc, vc)]
        return [bf(a) for a in (kc, vc)]

    dcaches = [contiguous(w, True) for _ in range(2)]
    dlay = pa.make_kv_layout(dcaches[0][0])

    def decode_contig(i):
        kc, vc = dcaches[i % 2]
        pa.astr_attn_decode_contiguous(q, kc, vc, dlay, seq, kvi, o_part, ml_part, out, dims, w.sm_scale, stream=sh)

    timed(decode_contig, 20)
    t_dc = timed(decode_contig, n_split) / n_split
    del dcaches
    pkc, pvc = contiguous(wp, False)
    play = pa.make_kv_layout(pkc)

    def prefill_contig(i):
        pa.astr_attn_prefill_contiguous(pq, pqo, pkc, pvc, play, ps_, pki, pout, pdims, wp.sm_scale, stream=sh)

    timed(prefill_contig, 5)
    t_pc = timed(prefill_contig, n_pf) / n_pf
    del pkc, pvc

    # ---------------- KV-append step on the extend workload (rotating copies: cold in L2)
    aqo_np, akn_np, avn_np = workload.append_rows(wp, seed=wp.seed + 1)
    a_rows = int(aqo_np[-1])
    a_bytes = 4 * a_rows * wp.num_kv_heads * wp.head_dim * 2  # read K and V rows, write them
    a_copy_bytes = 2 * akn_np.nbytes + 2 * wp.k_pool.nbytes
    n_app = max(2, min(8, -(-int(8e8) // a_copy_bytes)))
    aqo = i32(aqo_np)
    app_sets = [(bf(akn_np), bf(avn_np), bf(wp.k_pool), bf(wp.v_pool)) for _ in range(n_app)]
    adims = pa.make_dims(wp.batch, wp.num_qo_heads, wp.num_kv_heads, wp.head_dim, wp.num_slots, wp.r2t_stride,
                         wp.max_seq_len, total_q=a_rows)

    def kv_append(i):
        kn, vn, kp_, vp_ = app_sets[i % n_app]
        pa.astr_attn_kv_append(kn, vn, aqo, pr, ps_, kp_, vp_, adims, stream=sh)

    timed(kv_append, 3 * n_app)
    n_a = max(40, min(args.steps // 10, 400))
    t_app = timed(kv_append, n_a) / n_a
    app_gbs = a_bytes / t_app / 1e9
    del app_sets
    # context for the fraction: a plain contiguous device-to-device copy of the same bytes
    cp_src = [torch.empty(a_bytes // 2, dtype=torch.uint8, device=dev) for _ in range(n_app)]
    cp_dst = [torch.empty_like(x) for x in cp_src]

    def plain_copy(i):
        cp_dst[i % n_app].copy_(cp_src[i % n_app])

    timed(plain_copy, 3 * n_app)
    t_copy = timed(plain_copy, n_a) / n_a
    del cp_src, cp_dst

    # ---------------- CPU baseline: the oracle on this host (rank 0 at N=1 only)
    cpu = cpu_pf = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = os.cpu_count() or 1
        gbs, dt, reps = oracle_gbs(w, args.cpu_seconds, cores)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": f"whole B=32 decode batch, fp64 C oracle, {reps} calls of {dt:.3f} s"}
        tf, n_rows, dtp = oracle_prefill_tflops(wp, args.cpu_seconds / 2, cores)
        cpu_pf = {"value": round(tf, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                  "sample": f"{n_rows} random (query row, head) rows of the extend workload, fp64 C oracle, "
                            f"{dtp:.2f} s"}

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    traffic = recorded_traffic("decode_split", "decode.cu")
    line = {
        "metric": METRIC if args.decode_workload == DECODE_CFG else METRIC.split(", B=")[0] + f", {w.name}",
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(elapsed_max / args.steps * 1e3, 6),
        "us_per_call": round(us_per_call, 3),
        "repeats": {"regions": len(region_us), "steps_each": args.steps, "us_per_call_min": round(region_us[0], 3),
                    "us_per_call_median": round(us_per_call, 3), "us_per_call_max": round(region_us[-1], 3)},
        "us_per_call_graph": round(graph_us, 3) if isinstance(graph_us, float) else graph_us,
        "frac_of_hbm": round(value / world / peaks["hbm_gbs"], 4),
        "frac_of_nominal_8tbs": round(value / world / 7900.0, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "seed": w.seed, "page_size": 1, "num_splits": S,
                   "kv_bytes_per_call": nbytes["kv"], "total_keys": int(w.seq_lens.sum()),
                   "l2": f"rotating {n_copies} KV-pool copies ({n_copies * nbytes['kv'] / 1e6:.0f} MB > L2)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "kernel": "decode_split_kernel<128,4>", "achieved": round(split_gbs, 2),
                     "peak": peaks["hbm_gbs"], "peak_source": f"hbm_gbs ({peaks_src})", "unit": "GB/s",
                     "frac": round(split_gbs / peaks["hbm_gbs"], 4), "us_per_launch": round(t_split * 1e6, 3),
                     "stable_indices": {"us_per_launch": round(t_split_s * 1e6, 3),
                                        "frac": round(nbytes["kv"] / t_split_s / 1e9 / peaks["hbm_gbs"], 4),
                                        "us_per_call": round(t_call_s * 1e6, 3)},
                     "traffic": traffic},
        "prefill": {"workload": wp.name, "seed": wp.seed, "us_per_call": round(t_pf * 1e6, 3),
                    "plan": "host work plan of the batch (made once, outside the timed region)"
                    if pplan is not None else "none applies",
                    "us_per_call_unplanned": round(t_pfu * 1e6, 3),
                    "us_per_call_graph": round(t_pfg * 1e6, 3) if isinstance(t_pfg, float) else t_pfg,
                    "frac_unplanned": round(flops / t_pfu / 1e12 / peaks["bf16_tflops"], 4),
                    "flops_per_call": flops,
                    "l2": f"rotating {n_pcp} query/pool/output copies ({n_pcp * pf_copy_mb:.0f} MB)",
                    "roofline": {"bound": "tensor", "achieved": round(pf_tflops, 2), "peak": peaks["bf16_tflops"],
                                 "peak_source": f"bf16_tflops burst ({peaks_src})", "unit": "TFLOP/s",
                                 "frac": round(pf_tflops / peaks["bf16_tflops"], 4),
                                 "traffic": recorded_traffic("prefill", "prefill.cu")}},
        "masked": {"prefill": {"workload": wp.name, "mask": "3-D [B, max_q_len, kv_pitch], keep 0.75, causal on",
                               "us_per_call": round(t_pfm * 1e6, 3),
                               "tflops": round(flops / t_pfm / 1e12, 2),
                               "frac": round(flops / t_pfm / 1e12 / peaks["bf16_tflops"], 4)},
                   "decode": {"workload": w.name, "mask": "2-D [B, kv_pitch], keep 0.75",
                              "us_per_call": round(t_dm * 1e6, 3),
                              "gbs": round(nbytes["kv"] / t_dm / 1e9, 2),
                              "frac": round(nbytes["kv"] / t_dm / 1e9 / peaks["hbm_gbs"], 4)}},
        "contiguous": {"decode": {"workload": w.name, "layout": "bhld", "us_per_call": round(t_dc * 1e6, 3),
                                  "gbs": round(nbytes["kv"] / t_dc / 1e9, 2),
                                  "frac": round(nbytes["kv"] / t_dc / 1e9 / peaks["hbm_gbs"], 4)},
                       "prefill": {"workload": wp.name, "layout": "blhd", "us_per_call": round(t_pc * 1e6, 3),
                                   "tflops": round(flops / t_pc / 1e12, 2),
                                   "frac": round(flops / t_pc / 1e12 / peaks["bf16_tflops"], 4)}},
        "kv_append": {"workload": wp.name, "rows": a_rows, "us_per_call": round(t_app * 1e6, 3),
                      "bytes_per_call": a_bytes,
                      "same_bytes_device_copy_us": round(t_copy * 1e6, 3),
                      "l2": f"rotating {n_app} input/pool copies ({n_app * a_copy_bytes / 1e6:.0f} MB)",
                      "roofline": {"bound": "hbm", "achieved": round(app_gbs, 2), "peak": peaks["hbm_gbs"],
                                   "peak_source": f"hbm_gbs ({peaks_src})", "unit": "GB/s",
                                   "frac": round(app_gbs / peaks["hbm_gbs"], 4),
                                   "traffic": recorded_traffic("kv_append", "append.cu")}},
        "e2e": {"value": round(sum_over_ranks(nbytes["kv"]) / t_e2e_full / 1e9, 3), "unit": "GB/s",
                "h2d_bytes_per_step": h2d_full, "d2h_bytes_per_step": d2h,
                "resident_kv": {"value": round(sum_over_ranks(nbytes["kv"]) / t_e2e_res / 1e9, 3), "unit": "GB/s",
                                "h2d_bytes_per_step": h2d_res, "d2h_bytes_per_step": d2h}},
        "decode_workloads": decode_workloads,
        "gpu_launches": 2 * args.steps * len(region_us),
        "cpu_baseline": cpu,
        "prefill_cpu_baseline": cpu_pf,
        "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"],
                   "samples": clk["samples"]},
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
