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
    return ap.parse_args()


# ----------------------------------------------------------------------------------------
# workload accounting
# ----------------------------------------------------------------------------------------

def accounting(w):
    """Algorithmic bytes of one step of a reuse workload (bf16 = 2 bytes)."""
    lay = w.layout
    row = lay.row_k + lay.row_v
    written = sum(lay.num_layers * it.num_tokens * row * 2 for it in w.items)
    seen, canon = set(), 0
    for it in w.items:
        key = it.canon_k.data_ptr()
        if key not in seen:
            seen.add(key)
            canon += lay.num_layers * it.num_tokens * row * 2
    seen, patch = set(), 0
    for it in w.items:
        if it.patch_u is None:
            continue
        key = it.patch_u.data_ptr()
        if key not in seen:
            seen.add(key)
            patch += (it.patch_u.numel() + it.patch_vt.numel()) * 2
    naive_canon = written
    meta = 64 * len(w.items) + w.page_table.numel() * 4
    return dict(written=written, canon_distinct=canon, canon_naive=naive_canon, patch=patch,
                meta=meta, algorithmic=written + canon + patch + meta)


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
                         patch_l1=it.patch_l1) for it in w.items]
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


def config_desc(acc=None):
    d = {"workload": "GQA reorder, Qwen2-VL-7B-like: 28 layers, H_kv=4, head_dim=128, "
                     "theta=1e6, 3 chunks x T=1024 placed in all 6 orderings (18 placements), "
                     "rank-32 orbit patch on layers 14-27, page size 16, shuffled page table",
         "items": 18, "layers": 28, "T": 1024, "row": 512, "patch_rank": 32,
         "patched_layers": "14-27", "page_size": 16,
         "l2": "inputs larger than L2: 176 MB of canonicals and a 1.06 GB pool per step"}
    if acc:
        d["bytes_per_step"] = acc
    return d


# ----------------------------------------------------------------------------------------
# the CUDA arm
# ----------------------------------------------------------------------------------------

def kamera_arm(args, rank, world, local_rank):
    import torch
    import position_independent_multimodal_gb300 as km
    import workloads as wl

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = wl.config2(seed=rank, device=dev)
    lay = w.layout
    acc = accounting(w)
    h = km.create(lay)
    k = torch.empty(lay.num_layers, w.num_slots, lay.row_k, dtype=torch.bfloat16, device=dev)
    v = torch.empty(lay.num_layers, w.num_slots, lay.row_v, dtype=torch.bfloat16, device=dev)
    pt = w.page_table.to(dev)
    pool = km.Pool(k, v, pt, w.num_slots)
    d_items = km.pack_items(w.items).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    n_items = len(w.items)
    max_m = max(it.patch_m for it in w.items)
    stream = torch.cuda.current_stream()

    def step():
        km.kamera_batch_reuse(h, d_items, n_items, 1024, max_m, pool, status, stream)

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
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / args.steps
    if world > 1:
        t = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the timed region")

    e2e = None
    if not args.no_e2e:
        e2e = end_to_end(args, w, h, dev, stream)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        del w
        cpu = cpu_baseline(args.cpu_seconds)

    if rank != 0:
        return
    peak, src = measured_peak()
    s = ms / 1e3
    achieved = acc["algorithmic"] / s / 1e9
    line = {
        "metric": METRIC,
        "value": acc["written"] * world / s / 1e9,
        "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_desc(acc),
        "chunks_per_s": n_items * world / s,
        "us_per_chunk": ms * 1e3 / n_items,
        "gb_s_moved": achieved * world,
        "frac_hbm_peak": achieved / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)" if src == "measured"
                     else "fallback 6.8 TB/s",
                     "kernel": "reuse_stream_kernel",
                     "algorithmic_bytes_per_launch": acc["algorithmic"]},
        "gpu_launches": args.steps,
        "clocks": clk,
    }
    if e2e:
        line["e2e"] = e2e
    if cpu:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)


def end_to_end(args, w, h, dev, stream):
    """Same metric through the C-ABI with host buffers: every step copies the canonical and
    patch stores, the items and the page table from pinned host memory, runs the batch and
    reads the written pool back."""
    import torch
    import position_independent_multimodal_gb300 as km
    import workloads as wl

    lay = w.layout
    host, dev_bufs, seen = [], {}, {}
    for t in [x for it in w.items for x in (it.canon_k, it.canon_v, it.patch_u, it.patch_vt)]:
        if t is None or t.data_ptr() in seen:
            continue
        hb = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        hb.copy_(t)
        db = torch.empty_like(t)
        seen[t.data_ptr()] = db
        host.append((hb, db))
    items = [wl.Item(**{**it.__dict__,
                        "canon_k": seen[it.canon_k.data_ptr()],
                        "canon_v": seen[it.canon_v.data_ptr()],
                        "patch_u": None if it.patch_u is None else seen[it.patch_u.data_ptr()],
                        "patch_vt": None if it.patch_vt is None else
                        seen[it.patch_vt.data_ptr()]}) for it in w.items]
    h_items = km.pack_items(items).pin_memory()
    d_items = torch.empty_like(h_items, device=dev)
    h_pt = w.page_table.pin_memory()
    d_pt = torch.empty_like(h_pt, device=dev)
    k = torch.empty(lay.num_layers, w.num_slots, lay.row_k, dtype=torch.bfloat16, device=dev)
    v = torch.empty_like(k)
    hk = torch.empty(k.shape, dtype=k.dtype, pin_memory=True)
    hv = torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
    pool = km.Pool(k, v, d_pt, w.num_slots)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    max_m = max(it.patch_m for it in w.items)
    h2d = sum(hb.numel() * hb.element_size() for hb, _ in host) + h_items.numel() + \
        h_pt.numel() * 4
    d2h = (hk.numel() + hv.numel()) * 2

    def step():
        for hb, db in host:
            db.copy_(hb, non_blocking=True)
        d_items.copy_(h_items, non_blocking=True)
        d_pt.copy_(h_pt, non_blocking=True)
        km.kamera_batch_reuse(h, d_items, len(items), 1024, max_m, pool, status, stream)
        hk.copy_(k, non_blocking=True)
        hv.copy_(v, non_blocking=True)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.e2e_steps
    written = sum(lay.num_layers * it.num_tokens * (lay.row_k + lay.row_v) * 2 for it in items)
    return {"value": written / (ms / 1e3) / 1e9, "unit": "GB/s", "ms_per_step": ms,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        reference_arm(args, rank)
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
