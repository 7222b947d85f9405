#!/usr/bin/env python
"""Benchmark of the sparse-attention indexer top-k on one GB300.

One step = one pass of the hot path over its synthetic batch:
  * topk_transform on the packed-extend prefill chunk (2 requests x 8192
    rows on a 70000-token KV, scores [16384, 140000] fp32, page_size 1).

The JSON line follows the repository's bench contract: `value` is rows/s
with inputs resident in HBM; `e2e` repeats the step through the C ABI with
host-resident inputs (pinned host -> device copies and the device -> host
read of the slots inside the timed region); `roofline` is for the dominant
kernel; `cpu_baseline` times the CPU oracle on a bounded sample of the same
workload. `--impl reference` times only the oracle (the reference arm).
"""

from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "topk rows/s & HBM GB/s (% peak); fused score+topk keys/s (% roofline)"
UNIT = "rows/s"
K = 512
WORKLOAD = "packed-extend prefill top-k: 2 req x 8192 rows, KV 70000, scores [16384,140000] fp32, k=512, page_size=1"


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1900.0)), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [ln for ln in (out or "").splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- workload
def build_inputs(pinned: bool, new_tokens: int = 8192):
    import torch

    import workloads as W

    row_starts, seq_lens, r2b, width = W.packed_extend_meta(new_tokens=new_tokens)
    rows = int(seq_lens.size)
    host = torch.empty((rows, width), dtype=torch.float32, pin_memory=pinned)
    hn = host.numpy()
    chunk = 1024
    for r0 in range(0, rows, chunk):
        W.fill_rows(hn[r0:r0 + chunk], r0, 3, row_starts, seq_lens, fill=0.0)
    pt = W.page_table_perm(3, (2, 70000))
    meta = dict(row_starts=row_starts, seq_lens=seq_lens, row_to_batch=r2b, page_tables=pt, width=width, rows=rows)
    return host, meta


def algorithmic_bytes(meta) -> float:
    keys = float(meta["seq_lens"].astype(np.int64).sum())
    # scores read once + page-table rows + metadata + slots written
    return keys * 4 + meta["page_tables"].nbytes + meta["rows"] * (3 * 4 + K * 4)


# --------------------------------------------------------------------------- oracle
def oracle_sample(meta, budget_s: float = 15.0, max_rows: int = 4000):
    """Time the CPU oracle (single-threaded numpy sort) on a row sample."""
    import workloads as W
    from oracle.topk import topk_transform as oracle_topk

    rows = meta["rows"]
    sample = np.linspace(0, rows - 1, max_rows).astype(np.int64)
    done = 0
    t_total = 0.0
    for i in sample:
        n = int(meta["seq_lens"][i])
        w = W.packed_extend_window(3, int(i), n)
        b = int(meta["row_to_batch"][i])
        t0 = time.perf_counter()
        oracle_topk(w[None, :], np.array([n]), meta["page_tables"][[b]], 1, K)
        t_total += time.perf_counter() - t0
        done += 1
        if t_total > budget_s:
            break
    return done / t_total, done, t_total


def run_reference(args):
    rank, world, _ = _dist()
    if rank != 0:
        return
    import workloads as W

    row_starts, seq_lens, r2b, width = W.packed_extend_meta()
    meta = dict(row_starts=row_starts, seq_lens=seq_lens, row_to_batch=r2b,
                page_tables=W.page_table_perm(3, (2, 70000)), width=width, rows=int(seq_lens.size))
    budget = max(2.0, 120.0 / max(1, args.steps + args.warmup))
    vals = []
    for s in range(args.warmup + args.steps):
        v, n, t = oracle_sample(meta, budget_s=budget, max_rows=400)
        if s >= args.warmup:
            vals.append(v)
    value = float(np.median(vals))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 16384 / value * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": {"workload": WORKLOAD},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"rows spread over the 16384-row chunk, about {budget:.0f} s of sorting per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- GPU arm
def run_gpu(args):
    import torch

    rank, world, local = _dist()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import sparse_attention_indexer_top_gb300 as sai

    sai.load()
    hbm_peak, _, peak_kind = _peaks()

    host, meta = build_inputs(pinned=True, new_tokens=args.new_tokens)
    rows, width = meta["rows"], meta["width"]
    scores = torch.empty((rows, width), dtype=torch.float32, device=dev)
    scores.copy_(host, non_blocking=False)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    seq_lens, row_starts, r2b, pt = t(meta["seq_lens"]), t(meta["row_starts"]), t(meta["row_to_batch"]), t(meta["page_tables"])
    out_slots = torch.empty((rows, K), dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step():
        sai.topk_transform(scores, seq_lens, pt, row_starts=row_starts, row_to_batch=r2b, out_slots=out_slots,
                           stream=stream)

    launches_per_step = 1
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    assert sai.device_status() == 0

    # timed region: inputs (4.3 GB of windows) exceed L2, so no flush is needed
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t0 = time.perf_counter()
        for a, b in evs:
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    per = [a.elapsed_time(b) for a, b in evs]
    ms = float(np.mean(per))
    if world > 1:
        tt = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
        ms = float(tt.item())
    value = rows * world / (ms * 1e-3)
    alg = algorithmic_bytes(meta)
    achieved = alg / (ms * 1e-3) / 1e9
    keys = float(meta["seq_lens"].astype(np.int64).sum())

    # end to end: pinned host scores -> device, kernel, slots -> host
    e2e_steps = 0 if args.no_e2e else max(1, min(3, args.steps))
    host_out = torch.empty((rows, K), dtype=torch.int32, pin_memory=True)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(e2e_steps):
            scores.copy_(host, non_blocking=True)
            step()
            host_out.copy_(out_slots, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / max(1, e2e_steps)
    h2d = host.numel() * 4
    d2h = rows * K * 4

    cpu = None
    if rank == 0 and not args.no_cpu:
        v, n, tt = oracle_sample(meta)
        cpu = {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{n} rows spread over the chunk ({tt:.1f} s of single-threaded stable sorts)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "rows": rows, "keys_per_step": keys, "k": K,
                       "l2": "inputs larger than L2 (4.3 GB of score windows per step)",
                       "keys_per_s": keys * world / (ms * 1e-3), "hbm_gbs": achieved},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "traffic": None, "peak_kind": peak_kind,
                         "kernel": "topk_stream_kernel"},
            "e2e": None if args.no_e2e else {"value": rows / (e2e_ms * 1e-3), "unit": UNIT,
                                             "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk.summary(),
            "cpu_baseline": cpu,
            "wall_s_timed": wall,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end timing")
    ap.add_argument("--new-tokens", type=int, default=8192,
                    help="query rows per request (8192 = the full packed-extend chunk; smaller for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
