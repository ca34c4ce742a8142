#!/usr/bin/env python
"""Benchmark of the Kamera relocate + patch operator on GB300.

Default workload (the configuration the metric is quoted on): GQA reorder shaped like
Qwen2-VL-7B — 28 layers, 4 KV heads × 128, θ=1e6, three T=1024 chunks placed in all 6
orderings (18 placements), one rank-32 orbit patch per chunk on layers 14–27, pages of 16
shuffled over the pool. One step = one kamera_batch_reuse over the 18 placements.

Prints one JSON line (rank 0). ``--impl reference`` times the float64 CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KV GB/s written by relocate+patch (fraction of HBM peak); chunks/s at T=1024"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["kamera", "reference"], default="kamera")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU work of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip the brief timings of the MLA, survival and recall-sweep workloads")
    ap.add_argument("--workload", choices=OTHER_WORKLOADS, default=None,
                    help="time only this one of the other workloads and print it (a profiling "
                         "entry point; not the bench line)")
    ap.add_argument("--mla-chunks", type=int, default=64,
                    help="chunks of the MLA recall batch (64; fewer shrink it for profilers)")
    ap.add_argument("--sweep-requests", type=int, default=256,
                    help="requests of the recall sweep, 4 recalls each (256: 1024 items; fewer "
                         "shrink it for profilers)")
    ap.add_argument("--survivors-seqs", type=int, default=64,
                    help="sequences of the sliding-window survival workload (64: the full "
                         "77 GB K pool; fewer shrink it for profilers that replay the kernel)")
    return ap.parse_args()


# ----------------------------------------------------------------------------------------
# workload accounting
# ----------------------------------------------------------------------------------------

def accounting(w, items=None):
    """Algorithmic bytes of one step of a reuse workload (bf16 = 2 bytes), in total and per
    kernel: the streaming kernel takes the unpatched layers, the tensor-core kernel the patched
    ones. Canonical bytes count each distinct canonical once (placements that share it read
    it from L2); patch bytes count each distinct factor once."""
    items = w.items if items is None else items
    lay = w.layout
    row = lay.row_k + lay.row_v

    def patched(it, layer):
        return it.patch_m > 0 and it.patch_l0 <= layer < it.patch_l1

    out = {"copy": dict(written=0, canon=0), "tensor": dict(written=0, canon=0, patch=0)}
    seen_c, seen_p = set(), set()
    for it in items:
        for layer in range(lay.num_layers):
            kind = "tensor" if patched(it, layer) else "copy"
            nbytes = it.num_tokens * row * 2
            out[kind]["written"] += nbytes
            key = (it.canon_k.data_ptr(), layer)
            if key not in seen_c:
                seen_c.add(key)
                out[kind]["canon"] += nbytes
        if it.patch_u is not None and it.patch_u.data_ptr() not in seen_p:
            seen_p.add(it.patch_u.data_ptr())
            out["tensor"]["patch"] += (it.patch_u.numel() + it.patch_vt.numel()) * 2
    meta = 64 * len(items) + w.page_table.numel() * 4
    for k in out:
        out[k]["algorithmic"] = sum(out[k].values()) + meta
    written = out["copy"]["written"] + out["tensor"]["written"]
    canon = out["copy"]["canon"] + out["tensor"]["canon"]
    return dict(written=written, canon_distinct=canon, canon_naive=written,
                patch=out["tensor"]["patch"], meta=meta,
                algorithmic=written + canon + out["tensor"]["patch"] + meta,
                per_kernel={"reuse_copy_kernel": out["copy"]["algorithmic"],
                            "reuse_tile_kernel": out["tensor"]["algorithmic"],
                            "reuse_persist_kernel": out["tensor"]["algorithmic"]})


def recorded_traffic(kernel: str, workload: str = "gqa_reorder"):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu record, or None
    when there is no record or the kernel's sources changed since it was taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}_traffic.txt")
    try:
        rec = {}
        for line in open(path):
            line = line.strip()
            if line and not line.startswith("#") and "=" in line:
                k, v = line.split("=", 1)
                rec[k.strip()] = v.strip()
        csrc = os.path.join(ROOT, "position_independent_multimodal_gb300", "csrc")
        h = hashlib.sha256()
        for f in ("kamera_reuse_tile.cu", "kamera_dev.cuh", "kamera_ptx.cuh", "kamera_smem.cuh"):
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(fh.read())
        if rec.get("kernel") != kernel or rec.get("source_sha256") != h.hexdigest():
            return None
        return int(rec["dram_bytes_per_launch"])
    except Exception:
        return None


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ----------------------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------------------
# the float64 oracle on host cores (CPU baseline and reference arm)
# ----------------------------------------------------------------------------------------

_W = None


def _worker_init():
    os.environ["OMP_NUM_THREADS"] = "1"
    os.environ["OPENBLAS_NUM_THREADS"] = "1"
    import torch
    torch.set_num_threads(1)
    import workloads as wl
    global _W
    w = wl.config2(device="cpu")
    from oracle import kamera_oracle as ora
    items = [ora.as_item(canon_k=wl.bf16_bits(it.canon_k), canon_v=wl.bf16_bits(it.canon_v),
                         patch_u=None if it.patch_u is None else wl.bf16_bits(it.patch_u),
                         patch_vt=None if it.patch_vt is None else wl.bf16_bits(it.patch_vt),
                         delta=it.delta, num_tokens=it.num_tokens, req=it.req,
                         start_tok=it.start_tok, patch_m=it.patch_m, patch_l0=it.patch_l0,
                         patch_l1=it.patch_l1, delta_h=it.delta_h, delta_w=it.delta_w)
             for it in w.items]
    _W = (w.layout, items)


def _worker_units(units):
    from oracle import kamera_oracle as ora
    lay, items = _W
    t = time.perf_counter()
    nbytes = 0
    for i, layer, ch in units:
        bits = ora.reuse_layer_bits(lay, items[i], layer, ch)
        nbytes += bits.nbytes
    return nbytes, time.perf_counter() - t


def unit_order(n_items, L, n_ch):
    """(item, layer, channel) units in an order that mixes patched and unpatched layers in
    the workload's proportion."""
    import random
    out = [(i, layer, ch) for layer in range(L) for i in range(n_items) for ch in range(n_ch)]
    random.Random(0).shuffle(out)
    return out


class OraclePool:
    def __init__(self, cores: int):
        ctx = mp.get_context("spawn")
        self.cores = cores
        self.pool = ctx.Pool(cores, initializer=_worker_init)
        # warm every worker (input generation happens in the initializer)
        self.pool.map(_worker_units, [[] for _ in range(cores)])
        self.units = unit_order(18, 28, 2)
        self.pos = 0

    def calibrate(self):
        nb, dt = self.pool.apply(_worker_units, ([self.units[0], self.units[14 * 36]],))
        return dt / 2

    def run(self, n_units):
        chunks = [[] for _ in range(self.cores)]
        for k in range(n_units):
            chunks[k % self.cores].append(self.units[(self.pos + k) % len(self.units)])
        self.pos += n_units
        t = time.perf_counter()
        res = self.pool.map(_worker_units, chunks)
        wall = time.perf_counter() - t
        return sum(r[0] for r in res), wall

    def close(self):
        self.pool.close()
        self.pool.join()


def cpu_baseline(target_s: float):
    cores = os.cpu_count() or 1
    op = OraclePool(cores)
    try:
        per_unit = op.calibrate()
        n = max(cores, int(target_s * cores / max(per_unit, 1e-4)))
        nbytes, wall = op.run(n)
    finally:
        op.close()
    return {"value": nbytes / wall / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} (placement, layer, channel) units of the 18x28x2 of one step "
                      f"({nbytes / 1e6:.0f} MB written), float64 NumPy oracle, one process "
                      f"per core, {wall:.1f} s wall"}


def _oracle_per_chunk(threads: int):
    """µs per chunk of the float64 oracle on the tiny GQA workload (in full) and on timed units
    of the MLA recall, sliding-window and recall-sweep workloads (extrapolated linearly to a
    whole chunk). Runs in a fresh process whose BLAS / OpenMP thread count is `threads`."""
    import workloads as wl
    from oracle import kamera_oracle as ora

    def oitem(it):
        b = lambda t: None if t is None else wl.bf16_bits(t)
        return ora.as_item(canon_k=b(it.canon_k), canon_v=b(it.canon_v), patch_u=b(it.patch_u),
                           patch_vt=b(it.patch_vt), delta=it.delta, num_tokens=it.num_tokens,
                           req=it.req, start_tok=it.start_tok, patch_m=it.patch_m,
                           patch_l0=it.patch_l0, patch_l1=it.patch_l1, delta_h=it.delta_h,
                           delta_w=it.delta_w)

    def timed(fn):  # best of two runs
        best = None
        for _ in range(2):
            t = time.perf_counter()
            fn()
            dt = time.perf_counter() - t
            best = dt if best is None else min(best, dt)
        return best

    out = {}
    # tiny GQA: the whole chunk, every layer and channel
    w = wl.config1(strong=True)
    it = oitem(w.items[0])
    units = [(l, c) for l in range(w.layout.num_layers) for c in range(2)]
    dt = timed(lambda: [ora.reuse_layer_bits(w.layout, it, l, c) for l, c in units])
    out["tiny_gqa"] = {"us_per_chunk": dt * 1e6, "sample": "the whole chunk (2 layers x K, V)"}
    # MLA recall: one unpatched and one patched layer of one chunk, x13 and x14
    w = wl.config3(n_chunks=1)
    it = oitem(w.items[0])
    t0 = timed(lambda: ora.reuse_layer_bits(w.layout, it, 0, 0))
    t1 = timed(lambda: ora.reuse_layer_bits(w.layout, it, 13, 0))
    out["mla_recall"] = {"us_per_chunk": (13 * t0 + 14 * t1) * 1e6,
                         "sample": "layers 0 and 13 of one chunk, extrapolated to 13 unpatched "
                                   "and 14 patched layers"}
    # sliding window: 64 survivor tokens of one layer, extrapolated to 576 tokens x 32 layers
    w = wl.config4(n_seq=1, layers=1)
    pool = wl.bf16_bits(w.k_pool).copy()
    pt = w.page_table.numpy()
    sp = w.spans[0]
    t2 = timed(lambda: ora.relocate(w.layout, pool, pt, sp.req, sp.start_tok, 64, sp.delta))
    out["mha_sliding_window"] = {"us_per_chunk": t2 * (576 / 64) * 32 * 1e6,
                                 "sample": "64 survivor tokens of one layer, extrapolated to "
                                           "576 tokens x 32 layers"}
    # recall sweep: K and V of one unpatched and one patched layer, x32 each
    w = wl.config5(n_req=1, recalls=1)
    unp = oitem(wl.config5_launch_items(w, 0)[0])
    pat = oitem(wl.config5_launch_items(w, 4)[0])
    t3 = timed(lambda: [ora.reuse_layer_bits(w.layout, unp, 0, c) for c in range(2)])
    t4 = timed(lambda: [ora.reuse_layer_bits(w.layout, pat, 0, c) for c in range(2)])
    out["gqa_recall_sweep"] = {"us_per_chunk": 32 * (t3 + t4) * 1e6,
                               "sample": "K and V of one unpatched and one patched layer, "
                                         "extrapolated to 32 of each"}
    return out


def _oracle_per_chunk_in(threads: int):
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = str(threads)
    import torch
    torch.set_num_threads(threads)
    return _oracle_per_chunk(threads)


def oracle_per_chunk():
    """The oracle per chunk of the other reference workloads, at 1 thread and at all threads
    (each in its own spawned process, so the thread count applies before NumPy loads)."""
    cores = os.cpu_count() or 1
    ctx = mp.get_context("spawn")
    res = {}
    for threads in (1, cores):
        with ctx.Pool(1) as pool:
            res[threads] = pool.apply(_oracle_per_chunk_in, (threads,))
    out = {"kind": "oracle", "cores": cores, "extrapolated": True,
           "unit": "us per chunk (a chunk across all its layers)"}
    for name in res[1]:
        out[name] = {"us_1_thread": res[1][name]["us_per_chunk"],
                     f"us_{cores}_threads": res[cores][name]["us_per_chunk"],
                     "sample": res[1][name]["sample"]}
    return out


def reference_arm(args, rank):
    if rank != 0:
        return
    cores = os.cpu_count() or 1
    op = OraclePool(cores)
    try:
        per_unit = op.calibrate()
        budget_s = 150.0
        per_step = max(1, int(budget_s * cores / max(per_unit, 1e-4) / (args.steps + args.warmup)))
        per_step = min(per_step, len(op.units))  # at most one whole step of the workload
        for _ in range(args.warmup):
            op.run(per_step)
        tot_b, tot_t = 0, 0.0
        for _ in range(args.steps):
            b, t = op.run(per_step)
            tot_b += b
            tot_t += t
    finally:
        op.close()
    value = tot_b / tot_t / 1e9
    w_units = 18 * 28 * 2
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot_t / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_desc(),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": f"{per_step} of the {w_units} (placement, layer, "
                                       f"channel) units per step, float64 NumPy oracle, one "
                                       f"process per core"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def config_desc(acc=None, flushed=False):
    """The workload's description; `flushed` when every timed step follows an L2 flush."""
    l2 = "inputs larger than L2: 176 MB of canonicals and a 1.06 GB pool per step"
    if flushed:
        l2 = f"flushed: a {L2Flush.NBYTES >> 20} MB write before every timed step; also " + l2
    d = {"workload": "GQA reorder, Qwen2-VL-7B-like: 28 layers, H_kv=4, head_dim=128, "
                     "theta=1e6, 3 chunks x T=1024 placed in all 6 orderings (18 placements), "
                     "rank-32 orbit patch on layers 14-27, page size 16, shuffled page table",
         "items": 18, "layers": 28, "T": 1024, "row": 512, "patch_rank": 32,
         "patched_layers": "14-27", "page_size": 16, "l2": l2}
    if acc:
        d["bytes_per_step"] = acc
    return d


# ----------------------------------------------------------------------------------------
# sharding across ranks: every rank reuses its own seeded copy of the workload (no data-path
# collective); the job time is the slowest rank's
# ----------------------------------------------------------------------------------------

def rank_seed(rank: int) -> int:
    return rank


def job_time_ms(ms: float, world: int, device=None) -> float:
    """Max over ranks of the per-step time (every rank ran the same number of steps)."""
    if world <= 1:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(written_per_rank: int, world: int, job_ms: float) -> float:
    """GB/s written by all ranks together over the slowest rank's step time."""
    return written_per_rank * world / (job_ms / 1e3) / 1e9


# ----------------------------------------------------------------------------------------
# timing: individually event-timed runs, an L2 flush between them, median and spread
# ----------------------------------------------------------------------------------------

class L2Flush:
    """A write of a buffer well above L2's 129 MB, issued between timed runs so that each
    starts with nothing of its own inputs in L2."""
    NBYTES = 512 << 20

    def __init__(self, dev):
        import torch
        self.buf = torch.empty(self.NBYTES, dtype=torch.uint8, device=dev)
        self.n = 0

    def __call__(self, stream):
        import torch
        self.n += 1
        with torch.cuda.stream(stream):
            self.buf.fill_(self.n & 0xFF)


def event_pairs(n, stream):
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    for a, b in ev:
        a.record(stream)  # creates the event handles
        b.record(stream)
    return ev


def spread(ms):
    """Median, 10th and 90th percentile (nearest rank) and mean of per-run times in ms."""
    s = sorted(ms)

    def rank(p):
        return s[min(len(s) - 1, max(0, math.ceil(p / 100 * len(s)) - 1))]
    return {"median_ms": statistics.median(s), "p10_ms": rank(10), "p90_ms": rank(90),
            "mean_ms": statistics.fmean(s), "runs": len(s)}


def kernel_fracs(kern_stats, per_kernel_bytes, peak, traffic_of=None, launches=1):
    """Per kernel: its timing spread, algorithmic bytes per step, and achieved GB/s and
    fraction of peak from the median. ``traffic_of`` maps a kernel to the workload tag of its
    recorded DRAM traffic per launch; a step of ``launches`` launches carries that many."""
    out = {}
    for name, st in kern_stats.items():
        kb = per_kernel_bytes.get(name)
        kms = st["median_ms"]
        if kb is None:  # the planning kernel: timed, its bytes are not counted
            out[name] = dict(st, ms=kms)
            continue
        gbs = kb / (kms / 1e3) / 1e9 if kms > 0 else None
        out[name] = dict(st, ms=kms, algorithmic_bytes=kb, achieved_gbs=gbs,
                         frac=gbs / peak if gbs is not None else None)
        if traffic_of and name in traffic_of:
            t = recorded_traffic(name, traffic_of[name])
            out[name]["traffic_per_launch"] = t
            out[name]["launches_per_step"] = launches
    return out


def planned(h):
    """Whether the handle's last batch call took the persistent path: its workspace (filled
    with 0xFF when it was set) then holds a plan header."""
    import torch
    ws = getattr(h, "batch_workspace", None)
    return ws is not None and int(ws[:4].view(torch.int32).item()) >= 0


def split_stats(marks_per_pass, persistent):
    """Per-kernel spreads from event quads (before, between, after planning, after) per call,
    summed over a pass's calls: the copy kernel, then the planning kernel and the persistent
    kernel, or the grid tile kernel."""
    def tot(i, j):
        return spread([sum(q[i].elapsed_time(q[j]) for q in per) for per in marks_per_pass])
    if persistent:
        return {"reuse_copy_kernel": tot(0, 1), "reuse_plan_kernel": tot(1, 2),
                "reuse_persist_kernel": tot(2, 3)}
    return {"reuse_copy_kernel": tot(0, 1), "reuse_tile_kernel": tot(1, 3)}


def time_split(h, launches, pool, st, runs, flush, stream):
    """``runs`` passes of a reuse step (one kamera_batch_reuse per launch), each after an L2
    flush, with event marks between every call's kernels (which then run one after the
    other). Returns the spread of the per-pass time of each kernel, summed over the launches."""
    import torch
    import position_independent_multimodal_gb300 as km
    marks = [[[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in launches]
             for _ in range(runs)]
    for per in marks:
        for trio in per:
            for e in trio:
                e.record(stream)
    torch.cuda.synchronize()
    for d, n, mt, mm in launches:  # warm-up pass
        km.kamera_batch_reuse(h, d, n, mt, mm, pool, st, stream)
    for per in marks:
        flush(stream)
        for (d, n, mt, mm), trio in zip(launches, per):
            km.kamera_batch_reuse_timed(h, d, n, mt, mm, pool, st, trio, stream)
    torch.cuda.synchronize()
    if int(st.item()) != 0:
        raise RuntimeError(f"device status {int(st.item())}")
    return split_stats(marks, planned(h))


def time_steps(fn, runs, flush, stream, warmup=1):
    """Spread of ``runs`` individually event-timed calls of ``fn``, an L2 flush before each."""
    import torch
    for _ in range(warmup):
        fn()
    ev = event_pairs(runs, stream)
    torch.cuda.synchronize()
    for a, b in ev:
        flush(stream)
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return spread([a.elapsed_time(b) for a, b in ev])


# ----------------------------------------------------------------------------------------
# the CUDA arm
# ----------------------------------------------------------------------------------------

def batch_handle(km, lay, n_items, dev):
    """A handle with a batch workspace for batches of up to n_items items: the library plans
    such batches on the device and runs their patched layers as a persistent kernel (it keeps
    its per-tile grid kernel for batches that do not fit that path)."""
    import torch
    h = km.create(lay)
    ws = torch.full((km.kamera_batch_workspace_bytes(h, n_items),), 0xFF, dtype=torch.uint8,
                    device=dev)
    km.kamera_set_batch_workspace(h, ws)
    return h


def kamera_arm(args, rank, world, local_rank):
    import torch
    import position_independent_multimodal_gb300 as km
    import workloads as wl

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = wl.config2(seed=rank_seed(rank), device=dev)
    lay = w.layout
    acc = accounting(w)
    h = batch_handle(km, lay, len(w.items), dev)
    k = torch.empty(lay.num_layers, w.num_slots, lay.row_k, dtype=torch.bfloat16, device=dev)
    v = torch.empty(lay.num_layers, w.num_slots, lay.row_v, dtype=torch.bfloat16, device=dev)
    pt = w.page_table.to(dev)
    pool = km.Pool(k, v, pt, w.num_slots)
    d_items = km.pack_items(w.items).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    n_items = len(w.items)
    max_m = max(it.patch_m for it in w.items)
    stream = torch.cuda.current_stream()
    n_split = max(20, min(args.steps, 1000))
    flush = L2Flush(dev)
    step_ev = event_pairs(args.steps, stream)
    # four events per split step: before the copy kernel, between it and the patched layers,
    # after the planning kernel (persistent path) and after the last kernel
    marks = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_split)]
    for trio in marks:
        for e in trio:
            e.record(stream)  # creates the event handles
    torch.cuda.synchronize()

    def step(trio=None):
        if trio is None:
            km.kamera_batch_reuse(h, d_items, n_items, 1024, max_m, pool, status, stream)
        else:
            km.kamera_batch_reuse_timed(h, d_items, n_items, 1024, max_m, pool, status, trio,
                                        stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} after warm-up")

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    clocks = ClockSampler(local_rank)
    clocks.start()
    barrier()
    torch.cuda.synchronize()
    # the step as a user runs it: the two kernels side by side (copy kernel on the library's
    # side stream, joined back before the next step); every step timed on its own, after an
    # L2 flush that the events leave out
    for a, b in step_ev:
        flush(stream)
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    barrier()
    # second figure: the same number of steps back to back, no flush between them
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        step()
    e1.record(stream)
    # per-kernel split for the roofline: the same call with event marks between its kernels,
    # which runs them one after the other on the stream, each step after an L2 flush
    for trio in marks:
        flush(stream)
        step(trio)
    torch.cuda.synchronize()
    clk = clocks.stop()
    step_stats = spread([a.elapsed_time(b) for a, b in step_ev])
    b2b_ms = e0.elapsed_time(e1) / args.steps
    persistent = planned(h)
    kern_stats = split_stats([[q] for q in marks], persistent)
    kern_ms = {k: v["median_ms"] for k, v in kern_stats.items() if k in acc["per_kernel"]}
    ms = job_time_ms(step_stats["median_ms"], world, dev)
    b2b_ms = job_time_ms(b2b_ms, world, dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the timed region")
    del flush

    e2e = None
    if not args.no_e2e:
        e2e = end_to_end(args, w, h, dev, stream)
    del k, v, pool, w
    torch.cuda.empty_cache()
    others = None
    if rank == 0 and world == 1 and not args.no_other_workloads:
        others = other_workloads(dev)

    cpu = cpu_chunks = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.cpu_seconds)
        cpu_chunks = oracle_per_chunk()

    if rank != 0:
        return
    peak, src = measured_peak()
    s = ms / 1e3
    achieved = acc["algorithmic"] / s / 1e9
    dom = max(kern_ms, key=kern_ms.get)
    kernels = kernel_fracs(kern_stats, acc["per_kernel"], peak)
    line = {
        "metric": METRIC,
        "value": whole_job_gbs(acc["written"], world, ms),
        "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "step_timing": dict(step_stats, back_to_back_mean_ms=b2b_ms,
                            protocol=(f"{args.steps} steps each timed by its own pair of events, "
                                      f"an L2 flush (a {L2Flush.NBYTES >> 20} MB write) before "
                                      f"each and outside the events; ms_per_step and value are "
                                      f"the median; back_to_back_mean_ms is the mean of "
                                      f"{args.steps} further steps run back to back with no "
                                      f"flush")),
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_desc(acc, flushed=True),
        "chunks_per_s": n_items * world / s,
        "us_per_chunk": ms * 1e3 / n_items,
        "gb_s_moved": achieved * world,
        "frac_hbm_peak": achieved / peak,
        "roofline": {"bound": "hbm", "achieved": kernels[dom]["achieved_gbs"], "peak": peak,
                     "unit": "GB/s", "frac": kernels[dom]["frac"],
                     "traffic": recorded_traffic(dom),
                     "kernel": dom, "algorithmic_bytes_per_launch": acc["per_kernel"][dom],
                     "launch_ms": kern_ms[dom],
                     "peak_source": (f"{src} (MEASURED_PEAKS.json hbm_gbs)" if src == "measured"
                                     else "fallback 6.8 TB/s")},
        "kernels": kernels,
        "gpu_launches": (3 if persistent else 2) * args.steps,
        "kernel_split": (f"per-kernel medians (p10, p90) of {len(marks)} further steps, each "
                         f"after an L2 flush, with event marks between the kernels (run one "
                         f"after the other); the headline step runs the copy kernel beside the "
                         f"patched layers' kernels; frac from the median"
                         + ("; the patched layers take the planning kernel (one CTA: groups, "
                            "task rows, CTA ranges; its time is reported, its bytes are not "
                            "counted) and the persistent kernel, the roofline's kernel"
                            if persistent else "")),
        "clocks": clk,
    }
    if e2e:
        line["e2e"] = e2e
    if others:
        line["other_workloads"] = others
    if cpu:
        line["cpu_baseline"] = cpu
    if cpu_chunks:
        line["cpu_baseline_per_chunk"] = cpu_chunks
    print(json.dumps(line), flush=True)


OTHER_WORKLOADS = ("tiny_gqa_one_chunk", "patch_readd_in_place_18_placements",
                   "decode_attention_reorder_pool",
                   "mrope_reorder_18_placements", "reanchor_18_placements", "mla_recall_64_chunks",
                   "mla_recall_one_chunk",
                   "mha_sliding_window_448_survivors", "gqa_recall_sweep_1024_items",
                   "form_patch_84_deficits")


def other_workloads(dev, only=None, survivors_seqs=64, mla_chunks=64, sweep_requests=256):
    """Brief timings of the in-place switch, decode attention over the written pool, M-RoPE
    reorder, re-anchoring, MLA recall, sliding-window survival, recall-sweep and
    patch-forming workloads (each a parity-tested configuration of its own); reported beside
    the main line. ``only`` names one of them to run alone."""
    import torch
    import position_independent_multimodal_gb300 as km
    import workloads as wl

    peak, _ = measured_peak()
    out = {}

    def want(name):
        return only is None or only == name

    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()

    def reuse_calls(w, launches, runs=20, split=False):
        """Median (spread) of ``runs`` individually timed steps, one kamera_batch_reuse per
        launch, an L2 flush before each; with ``split``, also the per-kernel spread."""
        lay = w.layout
        h = batch_handle(km, lay, max(len(items) for items in launches), dev)
        k = torch.empty(lay.num_layers, w.num_slots, lay.row_k, dtype=torch.bfloat16, device=dev)
        v = (torch.empty(lay.num_layers, w.num_slots, lay.row_v, dtype=torch.bfloat16,
                         device=dev) if lay.kind == wl.GQA else None)
        pool = km.Pool(k, v, w.page_table.to(dev), w.num_slots)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        packed = [(km.pack_items(items).to(dev), len(items),
                   max(it.num_tokens for it in items), max(it.patch_m for it in items))
                  for items in launches]

        def call():
            for d, n, mt, mm in packed:
                km.kamera_batch_reuse(h, d, n, mt, mm, pool, st, stream)
        step = time_steps(call, runs, flush, stream)
        kern = time_split(h, packed, pool, st, runs, flush, stream) if split else None
        if int(st.item()) != 0:
            raise RuntimeError(f"device status {int(st.item())}")
        return step, kern

    if want("patch_readd_in_place_18_placements") or want("decode_attention_reorder_pool"):
        # reversible switch: the patch re-added in place on the cached rows of the 18 reorder
        # placements (their patched layers), alternately added and removed
        w = wl.config2(device=dev)
        lay = w.layout
        h = km.create(lay)
        k = torch.empty(lay.num_layers, w.num_slots, lay.row_k, dtype=torch.bfloat16, device=dev)
        v = torch.empty_like(k)
        pool = km.Pool(k, v, w.page_table.to(dev), w.num_slots)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        d_items = km.pack_items(w.items).to(dev)
        km.kamera_batch_reuse(h, d_items, len(w.items), 1024, 32, pool, st)
        flips = [1]

        def readd():
            sign = flips[0]
            flips[0] = -sign
            km.kamera_batch_patch_inplace(h, d_items, len(w.items), 1024, 32, pool, sign, st,
                                          stream)
        step = time_steps(readd, 20, flush, stream, warmup=4)
        ms = step["median_ms"]
        if int(st.item()) != 0:
            raise RuntimeError(f"device status {int(st.item())}")
        rows = sum(it.num_tokens * (it.patch_l1 - it.patch_l0) for it in w.items)
        moved = rows * (lay.row_k + lay.row_v) * 2 * 2 + \
            sum((it.patch_u.numel() + it.patch_vt.numel()) * 2 for it in w.items[:3])
        out["patch_readd_in_place_18_placements"] = {
            "workload": "GQA reorder pool (28 layers, H_kv=4 x 128): rank-32 patch re-added in place "
                        "on layers 14-27 of all 18 placements (one batched call), alternately +1 "
                        "and -1",
            "ms_per_step": ms, "timing": step, "gb_s_moved": moved / ms / 1e6,
            "frac_hbm_peak": moved / ms / 1e6 / peak}

        # consumer check: decode attention of one query token per head (Qwen2-VL-7B: 28 query
        # heads over the 4 KV heads) over the six 3072-token requests of that pool, every layer
        hq, ctx = 28, 3 * 1024
        reqs = int(w.page_table.shape[0])
        g = torch.Generator(device=dev)
        g.manual_seed(5)
        q = torch.randn(reqs, hq, lay.head_dim, generator=g, device=dev).to(torch.bfloat16)
        ctx_len = torch.full((reqs,), ctx, dtype=torch.int32, device=dev)
        o_buf = torch.empty(reqs, hq, lay.head_dim, device=dev)
        lse = torch.empty(reqs, hq, device=dev)
        ws = torch.empty(km.kamera_decode_attention_workspace(h, reqs, hq, ctx), dtype=torch.uint8,
                         device=dev)

        def attend_all_layers():
            for layer in range(lay.num_layers):
                km.kamera_decode_attention(h, pool, layer, q, ctx_len, ctx, lay.head_dim ** -0.5,
                                           o_buf, lse, ws, st)
        # a decode step runs its per-layer calls from a CUDA graph: capture the 28 calls once and
        # time the replays (the calls are made once before capture, which sets up the kernels)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            attend_all_layers()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            attend_all_layers()
        step = time_steps(graph.replay, 20, flush, stream, warmup=3)
        ms = step["median_ms"]
        if int(st.item()) != 0:
            raise RuntimeError(f"device status {int(st.item())}")
        kv_bytes = reqs * ctx * lay.num_layers * (lay.row_k + lay.row_v) * 2
        out["decode_attention_reorder_pool"] = {
            "workload": "decode attention over the reorder pool: 6 requests x 3072 tokens, 28 query "
                        "heads over 4 KV heads x 128, all 28 layers (one call per layer, replayed "
                        "from a CUDA graph)",
            "ms_per_step": ms, "timing": step, "gb_s_read": kv_bytes / ms / 1e6,
            "frac_hbm_peak": kv_bytes / ms / 1e6 / peak}
        del w, k, v, pool, q, ws, o_buf, graph
        torch.cuda.empty_cache()

    if want("mrope_reorder_18_placements"):
        w = wl.config2_mrope(device=dev)
        acc = accounting(w)
        step, _ = reuse_calls(w, [w.items])
        ms = step["median_ms"]
        out["mrope_reorder_18_placements"] = {
            "workload": "the GQA reorder step with Qwen2.5-VL M-RoPE (16|24|24 pairs over t, h, w; "
                        "t moved by j*1024, h and w by j*16 at ordering position j)",
            "ms_per_call": ms, "timing": step, "gb_s_written": acc["written"] / ms / 1e6,
            "frac_hbm_peak": acc["algorithmic"] / ms / 1e6 / peak}
        del w
        torch.cuda.empty_cache()

    if want("reanchor_18_placements"):
        # QV-PIC-style re-anchoring: 18 placements of three unrotated 1024-token images, every
        # layer, per-token (t, h, w) positions
        w = wl.config_reanchor(device=dev)
        lay = w.layout
        h = km.create(lay)
        k = torch.empty(lay.num_layers, w.num_slots, lay.row_k, dtype=torch.bfloat16, device=dev)
        v = torch.empty_like(k)
        pool = km.Pool(k, v, w.page_table.to(dev), w.num_slots)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        d_items = km.pack_anchor_items(w.items).to(dev)
        step = time_steps(lambda: km.kamera_reanchor(h, d_items, len(w.items), 1024, pool, st,
                                                     stream), 20, flush, stream, warmup=3)
        ms = step["median_ms"]
        if int(st.item()) != 0:
            raise RuntimeError(f"device status {int(st.item())}")
        written = sum(it.num_tokens for it in w.items) * lay.num_layers * (lay.row_k + lay.row_v) * 2
        distinct = {it.chunk_id: it for it in w.items}.values()
        read = sum(it.num_tokens for it in distinct) * lay.num_layers * (lay.row_k + lay.row_v) * 2 \
            + sum(it.positions.numel() * 8 for it in w.items)
        out["reanchor_18_placements"] = {
            "workload": "QV-PIC-style re-anchoring: three 32 x 32-token images stored before rotation "
                        "(Qwen2.5-VL layout, 28 layers, H_kv=4 x 128, M-RoPE 16|24|24) placed in all "
                        "6 orderings, every layer, per-token (t, h, w) positions",
            "ms_per_call": ms, "timing": step, "gb_s_written": written / ms / 1e6,
            "frac_hbm_peak": (written + read) / ms / 1e6 / peak}
        del w, k, v, pool, d_items
        torch.cuda.empty_cache()

    if want("tiny_gqa_one_chunk"):
        # the correctness-sized workload: one 256-token chunk, 2 layers, one kamera_reuse call
        # (launch- and latency-bound at this size)
        w = wl.config1(device=dev, strong=True)
        acc = accounting(w)
        lay = w.layout
        h = km.create(lay)
        k = torch.empty(lay.num_layers, w.num_slots, lay.row_k, dtype=torch.bfloat16, device=dev)
        pool = km.Pool(k, torch.empty_like(k), w.page_table.to(dev), w.num_slots)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        it = w.items[0]
        step = time_steps(lambda: km.kamera_reuse(h, it, pool, st, stream), 200, flush, stream,
                          warmup=20)
        ms = step["median_ms"]
        if int(st.item()) != 0:
            raise RuntimeError(f"device status {int(st.item())}")
        out["tiny_gqa_one_chunk"] = {
            "workload": "GQA 2 layers, H_kv=2 x 64, one chunk T=256 relocated by delta=1000, "
                        "m=8 patch on both layers (one kamera_reuse call)",
            "us_per_call": ms * 1e3, "timing": step, "gb_s_written": acc["written"] / ms / 1e6,
            "frac_hbm_peak": acc["algorithmic"] / ms / 1e6 / peak,
            "chunks_per_s": 1 / ms * 1e3}
        del w, k, pool
        torch.cuda.empty_cache()

    if want("mla_recall_64_chunks"):
        w = wl.config3(device=dev, n_chunks=mla_chunks)
        acc = accounting(w)
        step, kern = reuse_calls(w, [w.items], split=True)
        ms = step["median_ms"]
        out["mla_recall_64_chunks"] = {
            "workload": f"MLA (DeepSeek-V2-Lite-shaped) 27 layers, c_KV 512 + k_pe 64, "
                        f"{mla_chunks} chunks T=1024, delta in [-32768, 32768], m=32 on layers "
                        f"13-26",
            "ms_per_call": ms, "timing": step, "gb_s_written": acc["written"] / ms / 1e6,
            "frac_hbm_peak": acc["algorithmic"] / ms / 1e6 / peak,
            "chunks_per_s": len(w.items) / ms * 1e3,
            "kernels": kernel_fracs(kern, acc["per_kernel"], peak,
                                    {"reuse_tile_kernel": "mla_recall"} if mla_chunks == 64
                                    else None)}
        del w
        torch.cuda.empty_cache()

    if want("mla_recall_one_chunk"):
        # the recall as the paper states it: one T=1024 chunk at a random offset, one
        # kamera_reuse call (batch 1; the two kernels side by side)
        w = wl.config3(device=dev, n_chunks=1)
        acc = accounting(w)
        lay = w.layout
        h = km.create(lay)
        k = torch.empty(lay.num_layers, w.num_slots, lay.row_k, dtype=torch.bfloat16, device=dev)
        pool = km.Pool(k, None, w.page_table.to(dev), w.num_slots)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        it = w.items[0]
        step = time_steps(lambda: km.kamera_reuse(h, it, pool, st, stream), 200, flush, stream,
                          warmup=20)
        if int(st.item()) != 0:
            raise RuntimeError(f"device status {int(st.item())}")
        ms = step["median_ms"]
        out["mla_recall_one_chunk"] = {
            "workload": f"MLA (DeepSeek-V2-Lite-shaped) 27 layers, c_KV 512 + k_pe 64, one chunk "
                        f"T=1024 at delta={it.delta}, m=32 on layers 13-26, one kamera_reuse "
                        f"call",
            "us_per_call": ms * 1e3, "timing": step,
            "gb_s_written": acc["written"] / ms / 1e6,
            "frac_hbm_peak": acc["algorithmic"] / ms / 1e6 / peak,
            "chunks_per_s": 1 / ms * 1e3}
        del w, k, pool
        torch.cuda.empty_cache()

    if want("mha_sliding_window_448_survivors"):
        w = wl.config4(device=dev, n_seq=survivors_seqs)
        h = km.create(w.layout)
        vd = torch.zeros(1, 1, 8, dtype=torch.bfloat16, device=dev)
        pool = km.Pool(w.k_pool, vd, w.page_table.to(dev), w.num_slots)
        st = torch.zeros(1, dtype=torch.int32, device=dev)

        def reloc():
            for sp in w.spans:
                km.kamera_relocate(h, pool, sp.req, sp.start_tok, sp.num_tokens, sp.delta, st,
                                   stream)
        step = time_steps(reloc, 20, flush, stream)
        ms = step["median_ms"]
        moved = sum(sp.num_tokens for sp in w.spans) * w.layout.num_layers * w.layout.row_k * 2 * 2
        n_seq = len(w.spans)
        pool_gb = w.k_pool.numel() * 2 / 1e9
        out["mha_sliding_window_448_survivors"] = {
            "workload": f"MHA 32 layers x 32 heads x 128, {n_seq} sequences x 7 survivor chunks of "
                        f"576 tokens re-rotated in place by delta=-576 (K pool {pool_gb:.0f} GB)",
            "ms_per_step": ms, "timing": step, "gb_s_written": moved / 2 / ms / 1e6,
            "frac_hbm_peak": moved / ms / 1e6 / peak,
            "chunks_per_s": 7 * n_seq / ms * 1e3}
        del w, pool
        torch.cuda.empty_cache()

    if want("gqa_recall_sweep_1024_items"):
        w = wl.config5(device=dev, n_req=sweep_requests)
        n_items = len(w.items)
        launches = [wl.config5_launch_items(w, g) for g in range(8)]
        step, kern = reuse_calls(w, launches, split=True)
        ms = step["median_ms"]
        accs = [accounting(w, items) for items in launches]
        written = sum(a["written"] for a in accs)
        alg = sum(a["algorithmic"] for a in accs)
        per_kernel = {name: sum(a["per_kernel"][name] for a in accs)
                      for name in accs[0]["per_kernel"]}
        out["gqa_recall_sweep_1024_items"] = {
            "workload": f"GQA 64 layers (8 launches of 8-layer slices), H_kv=8 x 128, "
                        f"{sweep_requests} requests x 4 recalls T=1024, delta in [0, 131072), "
                        f"m=64 on layers 32-63",
            "ms_per_step": ms, "timing": step, "gb_s_written": written / ms / 1e6,
            "frac_hbm_peak": alg / ms / 1e6 / peak, "chunks_per_s": n_items / ms * 1e3,
            "kernels": kernel_fracs(kern, per_kernel, peak,
                                    {"reuse_tile_kernel": "recall_sweep"}
                                    if sweep_requests == 256 else None, launches=4)}
        del w, launches
        torch.cuda.empty_cache()

    if want("form_patch_84_deficits"):
        # patch forming: the 84 deficits of the reorder workload's patched layers (3 chunks x 14
        # layers x K and V), T = 1024 tokens x W = 512, top m = 32 from a k = 40 sketch with one
        # power iteration, written into the patch store layout
        n, T, W, k, q, m = 84, 1024, 512, 40, 1, 32
        delta, omega = wl.deficit_problems(n, T, W, k=k, rank=64, decay=0.9, noise=1e-2, seed=0,
                                           device=dev)
        u = torch.empty(n, T, m, dtype=torch.bfloat16, device=dev)
        vt = torch.empty(n, m, W, dtype=torch.bfloat16, device=dev)
        sig = torch.empty(n, m, dtype=torch.float32, device=dev)
        ws = torch.empty(km.kamera_form_patch_workspace(n, T, W, k), dtype=torch.uint8, device=dev)

        def form():
            km.kamera_form_patch(delta, omega, k, q, m, u, vt, sig, ws, num_problems=n, T=T, W=W,
                                 ld=W, delta_stride=T * W, omega_stride=0, u_stride=T * m,
                                 vt_stride=m * W)
        step = time_steps(form, 20, flush, stream, warmup=2)
        ms = step["median_ms"]
        # algorithmic float32 flops: the (2 + 2q) products with Δ, 12·M·k² per CholeskyQR3 on M
        # rows, and U·Σ = Q·Ũ_m (the Jacobi sweeps are not counted)
        flops = n * ((2 + 2 * q) * 2 * T * W * k + 12 * k * k * ((1 + q) * T + q * W) +
                     2 * T * k * m)
        out["form_patch_84_deficits"] = {
            "workload": "patch forming: 84 float32 deficits 1024 x 512 (the reorder workload's "
                        "patched layers), top 32 of a 40-column sketch, 1 power iteration",
            "ms_per_call": ms, "timing": step, "deficits_per_s": n / ms * 1e3,
            "gflop_s": flops / ms / 1e6,
            "delta_gb_s": (2 + 2 * q) * n * T * W * 4 / ms / 1e6}
        del delta, omega, u, vt, sig, ws
        torch.cuda.empty_cache()

    return out


def end_to_end(args, w, h, dev, stream):
    """Same metric through the C-ABI with host buffers: every step copies the canonical and
    patch stores, the items and the page table from pinned host memory (a KV store kept in
    host memory), runs the batch into the device pool, where attention reads it, and reads the
    step's result back: the call's device status word.

    Steps are pipelined the way a serving loop would run them: each step's input copies are
    spread over four copy streams into one of two device buffer sets, so step i + 1's copies
    overlap step i's kernels; a set is refilled only after the kernels that read it finished."""
    import torch
    import position_independent_multimodal_gb300 as km
    import workloads as wl

    lay = w.layout
    n_sets, n_copy = 2, 4
    host, seen = [], {}
    for t in [x for it in w.items for x in (it.canon_k, it.canon_v, it.patch_u, it.patch_vt)]:
        if t is None or t.data_ptr() in seen:
            continue
        hb = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        hb.copy_(t)
        seen[t.data_ptr()] = len(host)
        host.append(hb)
    sets = []
    for _ in range(n_sets):
        dbs = [torch.empty_like(hb, device=dev) for hb in host]
        items = [wl.Item(**{**it.__dict__,
                            "canon_k": dbs[seen[it.canon_k.data_ptr()]],
                            "canon_v": dbs[seen[it.canon_v.data_ptr()]],
                            "patch_u": None if it.patch_u is None else
                            dbs[seen[it.patch_u.data_ptr()]],
                            "patch_vt": None if it.patch_vt is None else
                            dbs[seen[it.patch_vt.data_ptr()]]}) for it in w.items]
        h_items = km.pack_items(items).pin_memory()
        sets.append({"dbs": dbs, "h_items": h_items,
                     "d_items": torch.empty_like(h_items, device=dev),
                     "d_pt": torch.empty(w.page_table.shape, dtype=w.page_table.dtype,
                                         device=dev),
                     "done": torch.cuda.Event()})
    h_pt = w.page_table.pin_memory()
    k = torch.empty(lay.num_layers, w.num_slots, lay.row_k, dtype=torch.bfloat16, device=dev)
    v = torch.empty_like(k)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    h_status = torch.zeros(1, dtype=torch.int32, pin_memory=True)
    max_m = max(it.patch_m for it in w.items)
    n_items = len(w.items)
    copy_streams = [torch.cuda.Stream(device=dev) for _ in range(n_copy)]
    h2d = sum(hb.numel() * hb.element_size() for hb in host) + \
        sets[0]["h_items"].numel() + h_pt.numel() * 4
    d2h = h_status.numel() * 4
    count = [0]

    def step():
        cur = sets[count[0] % n_sets]
        count[0] += 1
        pieces = [(db, hb) for db, hb in zip(cur["dbs"], host)] + \
            [(cur["d_items"], cur["h_items"]), (cur["d_pt"], h_pt)]
        joined = []
        for j, cs in enumerate(copy_streams):
            cs.wait_event(cur["done"])  # the kernels that last read this set are finished
            with torch.cuda.stream(cs):
                for db, hb in pieces[j::n_copy]:
                    db.copy_(hb, non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(cs)
            joined.append(ev)
        for ev in joined:
            stream.wait_event(ev)
        pool = km.Pool(k, v, cur["d_pt"], w.num_slots)
        km.kamera_batch_reuse(h, cur["d_items"], n_items, 1024, max_m, pool, status, stream)
        cur["done"].record(stream)
        h_status.copy_(status, non_blocking=True)

    for _ in range(2 * n_sets):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.e2e_steps
    if int(h_status.item()) != 0:
        raise RuntimeError(f"device status {int(h_status.item())}")
    written = sum(lay.num_layers * it.num_tokens * (lay.row_k + lay.row_v) * 2
                  for it in w.items)
    return {"value": written / (ms / 1e3) / 1e9, "unit": "GB/s", "ms_per_step": ms,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "pipeline": f"{n_copy} copy streams, {n_sets} input buffer sets"}


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        reference_arm(args, rank)
        return
    if args.workload is not None:
        import torch
        print(json.dumps(other_workloads(torch.device("cuda", local_rank), only=args.workload,
                                         survivors_seqs=args.survivors_seqs,
                                         mla_chunks=args.mla_chunks,
                                         sweep_requests=args.sweep_requests)))
        return
    if world > 1:
        import torch
        torch.distributed.init_process_group(backend="nccl")
    kamera_arm(args, rank, world, local_rank)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
