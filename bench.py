#!/usr/bin/env python
"""TBE fwd+bwd (rowwise Adagrad) benchmark on GB300.

One step = tbe_forward (pooled lookup with fused bounds check; on the large
Zipf workload the batch inversion -- linearise, radix sort, RLE -- runs
inside it) + tbe_backward_rowwise_adagrad (per-unique-row reduction routed
by segment length, one exact rowwise Adagrad update per touched row), over
one synthetic batch already resident in HBM.

Prints one JSON line (rank 0).  Default workload: the large Zipf
configuration (T=32, E=2M, D=128, bf16, B=131072, L~Poisson(20), ~84M
lookups, ~3M unique rows, hottest row ~125K lookups).

  python bench.py [--gpus N --steps K --warmup W] [--workload large|mid|hist|demo|tiny]
  python bench.py --impl reference      # the CPU oracle on a bounded sample

With N > 1 (torchrun) every rank runs an independent replica of the whole
workload (the path has no exchange step on one batch); the value is the
lookups of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import re
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "TBE fwd+bwd (rowwise Adagrad) lookups/s"
UNIT = "lookups/s"
PREPROCESS_IN_FORWARD = {"large": True, "mid": False, "demo": False, "tiny": False, "hist": False}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="large", choices=sorted(workloads.PRESETS))
    ap.add_argument("--long-mode", type=int, default=0, help="0 auto, 1 two-kernel, 2 fused")
    ap.add_argument("--hist-mode", type=int, default=0, help="0 auto, 1 off, 2 force")
    ap.add_argument("--preprocess", default="config", choices=["config", "forward", "backward"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--eager", action="store_true", help="time eager calls instead of CUDA graphs")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quick", action="store_true", help="skip e2e, cpu baseline and clocks (profiling runs)")
    ap.add_argument("--batch", type=int, default=None, help="override B (profiling a smaller case)")
    ap.add_argument("--rows", type=int, default=None, help="override E per table (large/mid)")
    return ap.parse_args()


def make_workload(args):
    kw = {}
    if args.batch is not None:
        kw["B"] = args.batch
    if args.rows is not None and args.workload in ("large", "mid"):
        kw["E"] = args.rows
    return workloads.PRESETS[args.workload](**kw)


# ----------------------------------------------------------------- helpers

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(x: float, device, world: int) -> float:
    """Max of a per-rank float over all ranks (the slowest replica's time)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.f = None

    def start(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.flush()
        rows = []
        for line in open(self.f.name):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.f.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if re.match(r"^[0-9.]+$", r[1])]
        mx = [float(r[2]) for r in rows if re.match(r"^[0-9.]+$", r[2])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


_BWD = ("backward.cu", "backward_kernels.cuh", "backward_f32.cu", "backward_f16.cu", "backward_bf16.cu")
KERNEL_SOURCE = [("tbe_fwd_", ("forward.cu",)), ("tbe_linearize", ("forward.cu",)),
                 ("tbe_offsets_fixup", ("forward.cu",)), ("tbe_sort_", ("sort.cu",)), ("tbe_rle_", ("rle.cu",)),
                 ("tbe_route", ("rle.cu",)), ("tbe_chunk_", ("rle.cu",)), ("tbe_zero_counters", ("rle.cu",)),
                 ("tbe_bwd_", _BWD), ("tbe_hist_", ("hist.cu",))]


def src_hash(kernel: str):
    """Hash of the source files that hold `kernel` and of the shared internal
    header: an ncu summary is current only while they are unchanged."""
    fns = next((f for pre, f in KERNEL_SOURCE if kernel.startswith(pre)), None)
    if fns is None:
        return None
    d = os.path.join(ROOT, "recsys_table_embedding_gb300", "csrc")
    h = hashlib.sha256()
    for f in fns + ("tbe_internal.cuh",):
        h.update(open(os.path.join(d, f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from a committed ncu summary, or None
    when there is none or the kernel's source changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    h = re.search(r"source_sha256_16:\s*([0-9a-f]+)", txt)
    if not m or not h or h.group(1) != src_hash(kernel):
        return None
    return float(m.group(1))


# ----------------------------------------------------------------- bytes

def run_stats(wl, tbe):
    """Realised batch statistics from the device metadata (generic path)."""
    import torch
    from recsys_table_embedding_gb300 import meta_view
    st = {"N": wl.N, "NB": wl.NB}
    if tbe.path != 1:
        return st
    U, nv, nlong, nchunks = tbe.counters()
    seg = meta_view(tbe.meta, "seg_off", U + 1, torch.int32).cpu().numpy().astype(np.int64)
    rl = np.diff(seg)
    long = rl >= 256
    st.update(U=U, n_valid=nv, num_long=nlong, num_chunks=nchunks, max_run=int(rl.max()) if U else 0,
              N_long=int(rl[long].sum()), N_short=int(rl[~long].sum()), U_short=int((~long).sum()))
    return st


def step_bytes(wl, st, pif: bool):
    """Algorithmic bytes of one step: what the method moves (no re-reads)."""
    N, NB, D = wl.N, wl.NB, wl.D
    sw = workloads.DTYPE_BYTES[wl.dtype]
    nw = 0
    if wl.per_sample_weights is not None:
        wt = wl.weighted_tables if wl.weighted_tables is not None else np.ones(wl.T, np.uint8)
        per_t = np.diff(wl.offsets[::wl.B].astype(np.int64))
        nw = int(per_t[wt.astype(bool)].sum())
    if st.get("U") is None:   # histogram path
        E = 64
        fwd = 4 * N + 4 * (NB + 1) + NB * D * 4 + NB * E * 2 + int(wl.rows_total) * D * sw
        bwd = NB * D * 4 + NB * E * 2 + 2 * int(wl.rows_total) * D * sw + 8 * int(wl.rows_total)
        return {"forward": fwd, "preprocess": 0, "backward": bwd, "total": fwd + bwd}
    U = st["U"]
    fwd = 4 * N + 4 * (NB + 1) + 4 * nw + N * D * sw + NB * D * 4
    pre = 8 * N + 16 * N + 4 * N + 12 * U
    bwd = 4 * N + 8 * U + 4 * nw + N * D * 4 + 2 * U * D * sw + 8 * U
    return {"forward": fwd, "preprocess": pre, "backward": bwd, "total": fwd + pre + bwd}


def kernel_bytes(name: str, wl, st, pif: bool):
    """Algorithmic bytes of one launch of the named kernel, or None."""
    N, NB, D = wl.N, wl.NB, wl.D
    sw = workloads.DTYPE_BYTES[wl.dtype]
    if name == "tbe_fwd_gather":
        return 4 * N + 4 * (NB + 1) + N * D * sw + NB * D * 4 + (8 * N if pif else 0)
    if name == "tbe_bwd_fused_long" or name == "tbe_bwd_grad_accum":
        nl = st.get("num_long", 0)
        b = 4 * st.get("N_long", 0) + st.get("N_long", 0) * D * 4
        if name == "tbe_bwd_fused_long":
            b += nl * (2 * D * sw + 8 + 8)
        return b
    if name == "tbe_bwd_short_run":
        us = st.get("U_short", 0)
        return 4 * st.get("N_short", 0) + st.get("N_short", 0) * D * 4 + us * (2 * D * sw + 8 + 8)
    if name == "tbe_sort_onesweep":
        return 16 * N
    if name in ("tbe_sort_histogram", "tbe_rle_count"):
        return 4 * N
    if name == "tbe_rle_write":
        return 4 * N + 8 * st.get("U", 0)
    if name == "tbe_linearize":
        return 4 * N + 4 * (NB + 1) + 8 * N
    if name == "tbe_bwd_apply":
        return st.get("num_long", 0) * (2 * D * sw + 8)
    if name == "tbe_hist_fwd_umma":
        return 4 * N + 4 * (NB + 1) + NB * D * 4 + NB * 64 * 2
    if name == "tbe_hist_bwd_umma":
        return NB * D * 4 + NB * 64 * 2
    return None


# ----------------------------------------------------------------- ours

def run_ours(args):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from recsys_table_embedding_gb300 import TBE, Batch, Tables, config, tbe as T

    wl = make_workload(args)
    pif = PREPROCESS_IN_FORWARD[args.workload] if args.preprocess == "config" else args.preprocess == "forward"
    cfg = config(long_run_mode=args.long_mode, hist_mode=args.hist_mode)

    W = wl.weights(device=str(dev))
    tables = Tables(W, wl.table_offset)
    idx_h = torch.from_numpy(wl.indices)
    off_h = torch.from_numpy(wl.offsets)
    G_h = torch.from_numpy(wl.grad_out())
    psw_h = torch.from_numpy(wl.per_sample_weights) if wl.per_sample_weights is not None else None
    wt = torch.from_numpy(wl.weighted_tables).to(dev) if wl.weighted_tables is not None else None
    idx, off, G = idx_h.to(dev), off_h.to(dev), G_h.to(dev)
    psw = psw_h.to(dev) if psw_h is not None else None
    batch = Batch(idx, off, wl.B, psw, wt)
    mom = torch.zeros(wl.rows_total, dtype=torch.float32, device=dev)
    out = torch.empty((wl.B, wl.T * wl.D), dtype=torch.float32, device=dev)
    tbe = TBE(tables, batch, cfg, preprocess_in_forward=pif)
    stream = torch.cuda.current_stream(dev)

    def step(b=batch, o=out, g=G):
        tbe.forward(b, o)
        tbe.backward(b, mom, g, wl.lr, wl.eps)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    st = run_stats(wl, tbe)
    status = tbe.status.cpu().numpy()

    # Per-kernel CUDA events recorded by the library around each of its
    # launches on the step's stream; one set per timed step.  The span of a
    # step (and of its forward and backward) runs from its first kernel's
    # start event to its last kernel's end event.
    max_pairs = 64

    class Slot:
        def __init__(self):
            self.evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * max_pairs)]
            for e in self.evs:
                e.record(stream)     # creates the CUDA event so its handle exists
            self.handles = (ctypes.c_void_p * (2 * max_pairs))(*[e.cuda_event for e in self.evs])
            self.names = (ctypes.c_char_p * max_pairs)()
            self.used = ctypes.c_int32(0)
            self.n_fwd = 0

        def arm(self):
            self.used.value = 0
            cfg.kernel_events = ctypes.cast(self.handles, ctypes.c_void_p)
            cfg.kernel_names = ctypes.cast(self.names, ctypes.c_void_p)
            cfg.n_kernel_events = max_pairs
            cfg.kernel_events_used = ctypes.cast(ctypes.pointer(self.used), ctypes.c_void_p)

        def run(self, strm=None):
            self.arm()
            tbe.forward(batch, out, stream=strm)
            self.n_fwd = self.used.value
            tbe.backward(batch, mom, G, wl.lr, wl.eps, stream=strm)

        def spans(self):
            """(step, forward, backward) milliseconds and per-kernel (name, ms)."""
            n = self.used.value
            e = self.evs
            kern = [(self.names[i].decode(), e[2 * i].elapsed_time(e[2 * i + 1])) for i in range(n)]
            stp = e[0].elapsed_time(e[2 * n - 1])
            fwd = e[0].elapsed_time(e[2 * self.n_fwd - 1])
            bwd = e[2 * self.n_fwd].elapsed_time(e[2 * n - 1]) if n > self.n_fwd else 0.0
            return stp, fwd, bwd, kern

    def disarm():
        cfg.kernel_events = None
        cfg.kernel_events_used = None

    # the timed steps run as CUDA graphs, one per step (each holds its own
    # events), captured after the warm-up: replaying a graph enqueues the
    # whole step at once, so the GPU never waits for the host between kernels
    slots = [Slot() for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    graphs = []
    mode = "cuda_graph"
    if not args.eager:
        try:
            cap = torch.cuda.Stream(dev)
            for sl in slots:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=cap, capture_error_mode="thread_local"):
                    sl.run()
                graphs.append(g)
            disarm()
            for g in graphs:          # upload and warm each graph once
                g.replay()
            torch.cuda.synchronize(dev)
        except Exception as e:       # graphs are an optimisation of the timed loop only
            disarm()
            graphs = []
            mode = f"eager (graph capture failed: {type(e).__name__}: {str(e)[:120]})"
            torch.cuda.synchronize(dev)
    else:
        mode = "eager"

    clocks = ClockSampler(local) if not args.quick else None
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    if clocks:
        clocks.start()
        time.sleep(0.3)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    h0 = time.perf_counter()
    t0.record(stream)
    for k in range(args.steps):
        if graphs:
            graphs[k].replay()
        else:
            slots[k].run()
    t1.record(stream)
    host_ms = (time.perf_counter() - h0) * 1e3
    torch.cuda.synchronize(dev)
    disarm()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop() if clocks else None
    ms_total = t0.elapsed_time(t1)

    # per-kernel durations and per-step spans
    kern = {}
    launches = 0
    steps_ms, fwd_ms, bwd_ms = [], [], []
    for sl in slots:
        stp, fwd, bwd, kl = sl.spans()
        steps_ms.append(stp)
        fwd_ms.append(fwd)
        bwd_ms.append(bwd)
        launches += len(kl)
        for nm, dt in kl:
            d = kern.setdefault(nm, [0, 0.0])
            d[0] += 1
            d[1] += dt
    kern_sum = sum(v[1] for v in kern.values())

    # the same steps launched one call at a time (no graph), for comparison:
    # shows what host-side enqueueing costs the eager API
    eager = None
    if graphs and not args.quick:
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        h1 = time.perf_counter()
        e0.record(stream)
        for k in range(args.steps):
            slots[k].run()
        e1.record(stream)
        eh = (time.perf_counter() - h1) * 1e3
        torch.cuda.synchronize(dev)
        disarm()
        eks = sum(sum(dt for _, dt in sl.spans()[3]) for sl in slots)
        et = e0.elapsed_time(e1)
        eager = {"ms_per_step": round(et / args.steps, 4),
                 "host_enqueue_ms_per_step": round(eh / args.steps, 4),
                 "gpu_gap_ms_per_step": round((et - eks) / args.steps, 4)}

    ms_total = reduce_max(ms_total, dev, world)
    ms_step = ms_total / args.steps
    value = wl.N * world * args.steps / (ms_total / 1e3)

    # e2e: host pinned inputs -> device, step, result -> host, every step
    e2e = None
    if not args.no_e2e and not args.quick:
        e2e = run_e2e(args, wl, tables, tbe, cfg, idx_h, off_h, G_h, psw_h, wt, mom, dev, world)

    peaks = measured_peaks()
    hbm_peak = peaks["hbm_gbs"] if peaks else 6800.0
    peak_src = "measured" if peaks else "fallback"
    sb = step_bytes(wl, st, pif)
    roof = None
    if kern:
        dom = max(kern, key=lambda n: kern[n][1])
        cnt, tot = kern[dom]
        avg_s = tot / cnt / 1e3
        kb = kernel_bytes(dom, wl, st, pif)
        if kb is not None:
            ach = kb / avg_s / 1e9
            traffic = ncu_traffic(dom, args.workload)
            roof = {"kernel": dom, "bound": "hbm", "achieved": round(ach, 1), "peak": hbm_peak,
                    "unit": "GB/s", "frac": round(ach / hbm_peak, 4),
                    "traffic": traffic, "bytes_per_launch": kb,
                    "avg_launch_ms": round(avg_s * 1e3, 4), "peak_source": peak_src,
                    "frac_basis": "algorithmic bytes: each lookup's row read counted once, "
                                  "re-reads that L2 serves included, so frac can exceed 1; "
                                  "dram_frac is the HBM figure"}
            if traffic:
                # what DRAM itself delivered
                dach = traffic / avg_s / 1e9
                roof["dram_achieved"] = round(dach, 1)
                roof["dram_frac"] = round(dach / hbm_peak, 4)
    step_ach = sb["total"] / (ms_step / 1e3) / 1e9
    kernels = {}
    for n, (c, t) in sorted(kern.items(), key=lambda kv: -kv[1][1]):
        kernels[n] = {"launches": c, "avg_ms": round(t / c, 4), "share": round(t / kern_sum, 4)}
        kb_n = kernel_bytes(n, wl, st, pif)
        if kb_n:
            kernels[n]["algo_gbs"] = round(kb_n / (t / c / 1e3) / 1e9, 1)
        tr = ncu_traffic(n, args.workload)
        if tr:
            kernels[n]["dram_gbs"] = round(tr / (t / c / 1e3) / 1e9, 1)

    res = None
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and not args.quick and world == 1:
            cpu = cpu_baseline(args.workload)
        res = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "ms_per_step_median": round(float(np.median(steps_ms)), 4),
            "forward_ms_median": round(float(np.median(fwd_ms)), 4),
            "backward_ms_median": round(float(np.median(bwd_ms)), 4),
            "launch_mode": mode,
            "host_enqueue_ms_per_step": round(host_ms / args.steps, 4),
            "gpu_gap_ms_per_step": round((ms_total - kern_sum) / args.steps, 4),
            "eager": eager,
            "config": {"workload": wl.name + ": " + wl.desc,
                       "weights": wl.dtype, "accumulate": "f64" if wl.dtype == "f32" else "f32",
                       "preprocess_in_forward": pif, "path": "histogram" if tbe.path == 2 else "generic",
                       "long_run_mode": args.long_mode, "lookups": wl.N, "bags": wl.NB,
                       "unique_rows": st.get("U"), "max_run": st.get("max_run"),
                       "long_runs": st.get("num_long"), "chunks": st.get("num_chunks"),
                       "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas{world}",
                       "status_words": [int(x) for x in status[:2]]},
            "roofline": roof,
            "step_roofline": {"bytes": sb["total"], "achieved": round(step_ach, 1), "peak": hbm_peak,
                              "unit": "GB/s", "frac": round(step_ach / hbm_peak, 4),
                              "frac_of_8tbs_nominal": round(step_ach / 8000.0, 4),
                              "bytes_split": sb},
            "kernels": kernels,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clk,
        }
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return res


E2E_WARM = 3      # untimed replays of the captured end-to-end pipeline
E2E_REPEATS = 5   # timed ones (median reported)


def run_e2e(args, wl, tables, tbe, cfg, idx_h, off_h, G_h, psw_h, wt, mom, dev, world):
    """The step through the public API from pinned host memory.  Every step
    uploads its inputs -- the batch (indices, offsets, weights) and the
    upstream gradient of the pooled output -- and reads back its result on
    the host: the status words (out-of-range count and error flags), which a
    caller must check after every step.  Uploads run on one copy stream and
    the read-back on another, into double-buffered device tensors, so step
    i+1's upload overlaps step i's compute.  The pipeline of all the timed
    steps is captured once as a CUDA graph (the same calls, enqueued ahead),
    so host speed does not pace it.  A second figure also downloads each
    step's pooled output [B, T*D] (the forward's activations)."""
    import torch
    from recsys_table_embedding_gb300 import Batch
    idx_p, off_p, G_p = idx_h.pin_memory(), off_h.pin_memory(), G_h.pin_memory()
    psw_p = psw_h.pin_memory() if psw_h is not None else None
    steps = max(3, min(args.steps, 10))
    out_p = [torch.empty((wl.B, wl.T * wl.D), dtype=torch.float32).pin_memory() for _ in range(2)]
    stat_p = torch.zeros((steps, 4), dtype=torch.int32).pin_memory()
    bufs = []
    for _ in range(2):
        idx_d, off_d = torch.empty_like(idx_h, device=dev), torch.empty_like(off_h, device=dev)
        psw_d = torch.empty_like(psw_h, device=dev) if psw_h is not None else None
        bufs.append(dict(idx=idx_d, off=off_d, psw=psw_d, G=torch.empty_like(G_h, device=dev),
                         out=torch.empty((wl.B, wl.T * wl.D), dtype=torch.float32, device=dev),
                         batch=Batch(idx_d, off_d, wl.B, psw_d, wt)))
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    h2d = (idx_h.numel() * idx_h.element_size() + off_h.numel() * off_h.element_size()
           + G_h.numel() * 4 + (psw_h.numel() * 4 if psw_h is not None else 0))
    d2h_status = 4 * 4
    d2h_out = out_p[0].numel() * 4

    def pipeline(main, with_out):
        """Enqueue `steps` end-to-end steps; returns after joining the copy
        streams back into `main`."""
        fork = torch.cuda.Event()
        fork.record(main)
        up.wait_event(fork)
        down.wait_event(fork)
        state = [dict(bwd_done=None, out_copied=None) for _ in range(2)]
        last_down = None
        for i in range(steps):
            bf, sv = bufs[i & 1], state[i & 1]
            # buffers of step i-2: its backward read G and the batch, its
            # download read out
            with torch.cuda.stream(up):
                if sv["bwd_done"] is not None:
                    up.wait_event(sv["bwd_done"])
                bf["idx"].copy_(idx_p, non_blocking=True)
                bf["off"].copy_(off_p, non_blocking=True)
                if bf["psw"] is not None:
                    bf["psw"].copy_(psw_p, non_blocking=True)
                in_ready = torch.cuda.Event()
                in_ready.record(up)
                bf["G"].copy_(G_p, non_blocking=True)
                g_ready = torch.cuda.Event()
                g_ready.record(up)
            main.wait_event(in_ready)
            if sv["out_copied"] is not None:
                main.wait_event(sv["out_copied"])
            tbe.forward(bf["batch"], bf["out"], stream=main)
            if with_out:
                fwd_done = torch.cuda.Event()
                fwd_done.record(main)
                with torch.cuda.stream(down):
                    down.wait_event(fwd_done)
                    out_p[i & 1].copy_(bf["out"], non_blocking=True)
                    oc = torch.cuda.Event()
                    oc.record(down)
                sv["out_copied"] = oc
            main.wait_event(g_ready)
            tbe.backward(bf["batch"], mom, bf["G"], wl.lr, wl.eps, stream=main)
            bwd_done = torch.cuda.Event()
            bwd_done.record(main)
            sv["bwd_done"] = bwd_done
            with torch.cuda.stream(down):
                down.wait_event(bwd_done)
                stat_p[i].copy_(tbe.status, non_blocking=True)
                last_down = torch.cuda.Event()
                last_down.record(down)
        last_up = torch.cuda.Event()
        last_up.record(up)
        main.wait_event(last_up)
        main.wait_event(last_down)     # the last step's result is on the host

    def measure(with_out):
        main = torch.cuda.current_stream(dev)
        graph, mode = None, "cuda_graph"
        if not args.eager:
            try:
                cap = torch.cuda.Stream(dev)
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=cap, capture_error_mode="thread_local"):
                    pipeline(torch.cuda.current_stream(dev), with_out)
                # upload and warm: the first replays of a fresh pipeline ran
                # 2-3x slower (29.7, 15.6, then 12.8 ms per step) on one box
                for _ in range(E2E_WARM):
                    graph.replay()
            except Exception as e:
                graph, mode = None, f"eager (graph capture failed: {type(e).__name__}: {str(e)[:120]})"
        else:
            mode = "eager"
        if graph is None:
            pipeline(main, with_out)   # warm
        torch.cuda.synchronize(dev)
        # E2E_REPEATS timed runs of the whole pipeline; the median run is
        # reported, every run alongside it (single runs ~2x slower than the
        # others come and go: 12.31, 12.31, 22.39, 12.31, 12.31 ms per step)
        runs, host = [], 0.0
        for _ in range(E2E_REPEATS):
            if world > 1:
                torch.distributed.barrier()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            h0 = time.perf_counter()
            a.record(main)
            if graph is not None:
                graph.replay()
            else:
                pipeline(main, with_out)
            b.record(main)
            host = (time.perf_counter() - h0) * 1e3
            torch.cuda.synchronize(dev)
            runs.append(reduce_max(a.elapsed_time(b), dev, world))
        return float(np.median(runs)), mode, host, runs

    ms, mode, host, runs = measure(False)
    res = {"value": round(wl.N * world * steps / (ms / 1e3), 1), "unit": UNIT,
           "ms_per_step": round(ms / steps, 4), "steps": steps,
           "runs_ms_per_step": [round(r / steps, 4) for r in runs],
           "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h_status),
           "launch_mode": mode, "host_enqueue_ms_per_step": round(host / steps, 4),
           "result_read_back": "status words (out-of-range count, error flags) of every step",
           "pipeline": "uploads and read-backs on two copy streams, double-buffered, overlapping compute"}
    ms2, _, _, runs2 = measure(True)
    res["with_output_download"] = {"value": round(wl.N * world * steps / (ms2 / 1e3), 1),
                                   "ms_per_step": round(ms2 / steps, 4),
                                   "runs_ms_per_step": [round(r / steps, 4) for r in runs2],
                                   "d2h_bytes_per_step": int(d2h_status + d2h_out)}
    # copy rates alone, for reading the figures above
    x = torch.empty_like(G_h, device=dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    x.copy_(G_p, non_blocking=True)
    b.record()
    torch.cuda.synchronize(dev)
    res["h2d_gbs"] = round(G_h.numel() * 4 / (a.elapsed_time(b) / 1e3) / 1e9, 1)
    a.record()
    out_p[0].copy_(bufs[0]["out"], non_blocking=True)
    b.record()
    torch.cuda.synchronize(dev)
    res["d2h_gbs"] = round(d2h_out / (a.elapsed_time(b) / 1e3) / 1e9, 1)
    del x
    return res


# ----------------------------------------------------------------- oracle

def oracle_sample(workload: str, tables: int, min_tables: int = 1, max_weight_bytes: float = 0):
    """A bounded sample of the workload for the CPU oracle: its first `tables`
    tables (at least `min_tables`, fewer if their float32 weights would pass
    `max_weight_bytes`) with all their bags (same indices and offsets), fresh
    weights of the same distribution and an upstream gradient for them."""
    wl = workloads.PRESETS[workload]()
    k = min(tables, wl.T)
    if max_weight_bytes:
        per_table = float(np.max(wl.table_rows)) * wl.D * 4
        k = min(k, max(1, int(max_weight_bytes // per_table)))
    k = max(k, min(min_tables, wl.T))
    end = int(wl.offsets[k * wl.B])
    sub = workloads.Workload(
        name=wl.name, T=k, B=wl.B, D=wl.D, dtype=wl.dtype, table_rows=wl.table_rows[:k].copy(),
        offsets=wl.offsets[:k * wl.B + 1].copy(), indices=wl.indices[:end].copy(),
        per_sample_weights=wl.per_sample_weights[:end].copy() if wl.per_sample_weights is not None else None,
        weighted_tables=wl.weighted_tables[:k].copy() if wl.weighted_tables is not None else None,
        lr=wl.lr, eps=wl.eps, seed=wl.seed)
    rng = np.random.default_rng(99)
    Wf = rng.uniform(-wl.w_init, wl.w_init, size=(sub.rows_total, wl.D)).astype(np.float32)
    if wl.dtype == "f32":
        W = Wf
    else:
        import torch
        W = torch.from_numpy(Wf).to(sub.torch_dtype()).view(torch.int16).numpy().view(np.uint16)
    G = rng.standard_normal((wl.B, k * wl.D), dtype=np.float32)
    return sub, W, G, wl


def oracle_step(sub, W, G):
    import oracle
    oracle.forward(sub, W)
    oracle.backward_adagrad(sub, W, sub.momentum(), G)


def _table_slice(sub, W, G, j):
    """Table j of an oracle sample as a one-table problem (same lookups)."""
    B, D = sub.B, sub.D
    s0, s1 = int(sub.offsets[j * B]), int(sub.offsets[(j + 1) * B])
    r0, r1 = int(sub.table_offset[j]), int(sub.table_offset[j + 1])
    one = workloads.Workload(
        name=sub.name, T=1, B=B, D=D, dtype=sub.dtype, table_rows=sub.table_rows[j:j + 1].copy(),
        offsets=(sub.offsets[j * B:(j + 1) * B + 1] - s0).astype(sub.offsets.dtype),
        indices=sub.indices[s0:s1].copy(),
        per_sample_weights=sub.per_sample_weights[s0:s1].copy() if sub.per_sample_weights is not None else None,
        weighted_tables=sub.weighted_tables[j:j + 1].copy() if sub.weighted_tables is not None else None,
        lr=sub.lr, eps=sub.eps, seed=sub.seed)
    return one, W[r0:r1], np.ascontiguousarray(G[:, j * D:(j + 1) * D])


_START = None


def _oracle_worker_init(barrier):
    global _START
    _START = barrier


def _oracle_table_job(job):
    one, W, G = job
    import oracle
    oracle.build()
    _START.wait(timeout=120)   # every worker holds its table before any starts
    t0 = time.perf_counter()   # CLOCK_MONOTONIC: comparable across processes
    oracle_step(one, W, G)
    return one.N, t0, time.perf_counter()


def cpu_baseline(workload: str):
    """The oracle as it stands on host cores: single-threaded on the first k
    tables, and one table per process over all cores (tables are independent
    problems; processes started with spawn)."""
    import multiprocessing as mp
    import oracle
    oracle.build()
    k = {"large": 4, "mid": 4, "hist": 8, "demo": 16, "tiny": 2}[workload]
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    # one table per core for the multi-process figure, ~4 GB of weights at most
    sub, W, G, wl = oracle_sample(workload, cores, min_tables=k, max_weight_bytes=4e9)
    first, Wf, Gf = sub, W, G
    if sub.T > k:   # the single-threaded sample: the first k tables
        end = int(sub.offsets[k * sub.B])
        first = workloads.Workload(
            name=sub.name, T=k, B=sub.B, D=sub.D, dtype=sub.dtype, table_rows=sub.table_rows[:k].copy(),
            offsets=sub.offsets[:k * sub.B + 1].copy(), indices=sub.indices[:end].copy(),
            per_sample_weights=sub.per_sample_weights[:end].copy() if sub.per_sample_weights is not None else None,
            weighted_tables=sub.weighted_tables[:k].copy() if sub.weighted_tables is not None else None,
            lr=sub.lr, eps=sub.eps, seed=sub.seed)
        Wf = W[:int(sub.table_offset[k])]
        Gf = np.ascontiguousarray(G[:, :k * sub.D])
    t = time.perf_counter()
    oracle_step(first, Wf, Gf)
    dt = time.perf_counter() - t
    res = {"value": round(first.N / dt, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
           "seconds": round(dt, 2),
           "sample": f"first {first.T} tables of the workload with all their bags ({first.N} lookups): "
                     f"forward + batch inversion + backward with Adagrad, single-threaded plain C, "
                     f"double accumulation"}
    nproc = min(cores, sub.T)
    if nproc > 1 and dt >= 1.0:
        # one table per process, all released together by a barrier; the
        # compute window is from the first start to the last end
        try:
            ctx = mp.get_context("spawn")
            jobs = [_table_slice(sub, W, G, j) for j in range(nproc)]
            with ctx.Pool(nproc, initializer=_oracle_worker_init, initargs=(ctx.Barrier(nproc),)) as pool:
                # bounded: a worker that dies would otherwise leave map() waiting forever
                out = pool.map_async(_oracle_table_job, jobs, chunksize=1).get(timeout=600)
            n = sum(o[0] for o in out)
            dta = max(o[2] for o in out) - min(o[1] for o in out)
            res["all_cores"] = {"value": round(n / dta, 1), "cores": nproc, "seconds": round(dta, 2),
                                "sample": f"{nproc} tables ({n} lookups), one table per process, "
                                          f"timed from the first start to the last end"}
        except Exception as e:   # the figure is optional: never fail the benchmark for it
            res["all_cores"] = {"unavailable": f"{type(e).__name__}: {e}"[:200]}
    return res


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    oracle.build()
    sub, W, G, wl = oracle_sample(args.workload, 1)
    for _ in range(args.warmup):
        oracle_step(sub, W, G)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(sub, W, G)
    dt = time.perf_counter() - t
    value = sub.N * args.steps / dt
    pif = PREPROCESS_IN_FORWARD[args.workload]
    sample = (f"table 0 of the {wl.T}-table workload with all its {wl.B} bags ({sub.N} lookups) per step: "
              f"forward + batch inversion + backward with Adagrad, single-threaded plain C oracle")
    res = {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT,
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": wl.name + ": " + wl.desc, "weights": wl.dtype,
                      "preprocess_in_forward": pif},
           "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)
    return res


def main():
    args = parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
