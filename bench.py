#!/usr/bin/env python
"""Benchmark of the sparse-attention indexer top-k on one GB300.

One step = one pass of the whole hot path, each part over its synthetic
batch:
  * topk_transform on the packed-extend prefill chunk (2 requests x 8192
    rows on a 70000-token KV, scores [16384, 140000] fp32, page_size 1);
  * fused FP8 index score + top-512 for decode (64 rows, 64 heads x 128,
    seq_lens U[4096, 32768], 128-token blocks);
  * fused FP8 index score + top-512 for prefill (4096 causal rows on a
    32768-token KV, grouped by 4).

The JSON line follows the repository's bench contract: `value` is query
rows per second over the whole step with inputs resident in HBM; `e2e`
repeats the step through the C ABI with host-resident inputs (pinned host ->
device copies of every input and the device -> host read of every output
inside the timed region); `roofline` is for the kernel that takes the most
time, `config.paths` gives every part's own numbers; `cpu_baseline` times
the CPU oracle on a bounded row sample of each part. `--impl reference`
times only the oracle (the reference arm).
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
WORKLOAD = ("indexer hot path step: packed-extend top-k (16384 rows, KV 70000, fp32 [16384,140000], page_size 1) "
            "+ fused FP8 score+top-k decode (64 rows, 64x128 heads, U[4096,32768] keys) "
            "+ fused FP8 score+top-k prefill (4096 causal rows, KV 32768, groups of 4); k=512")
PATHS = ("topk_packed_extend", "fused_decode", "fused_prefill")


def _peaks():
    """(HBM GB/s, dense bf16 TFLOP/s burst, provenance)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1900.0)), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


FP8_OVER_BF16 = 2.0  # nominal dense fp8 / bf16 tensor ratio (4.5 / 2.25 PFLOP/s), used only if the GEMM fails


def measure_fp8_peak(dev, n: int = 8192, reps: int = 10):
    """Dense e4m3 x e4m3 -> bf16 GEMM throughput (TFLOP/s) of this GPU: a
    cuBLASLt GEMM through torch._scaled_mm on n^3 (2 n^3 flops), best of
    `reps` launches timed with CUDA events after 3 warm-ups. Returns
    (TFLOP/s, note) or (None, why) when the GEMM is unavailable."""
    import torch

    try:
        g = torch.Generator(device=dev).manual_seed(7)
        a = torch.randn((n, n), device=dev, generator=g).to(torch.float8_e4m3fn)
        b = torch.randn((n, n), device=dev, generator=g).to(torch.float8_e4m3fn)
        one = torch.ones((), device=dev, dtype=torch.float32)

        def run():
            return torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)

        for _ in range(3):
            run()
        torch.cuda.synchronize(dev)
        best = float("inf")
        for _ in range(reps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            run()
            e1.record()
            torch.cuda.synchronize(dev)
            best = min(best, e0.elapsed_time(e1))
        del a, b
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12, f"torch._scaled_mm e4m3 {n}^3, best of {reps} ({best:.3f} ms)"
    except Exception as exc:  # no fp8 GEMM in this torch build
        return None, f"fp8 GEMM unavailable ({type(exc).__name__}: {exc})"

# DRAM bytes (read + write) per key, from one ncu capture of each kernel as
# it stands (one pass, at full size; summaries under profiles/, by kernel
# and workload): top-k stream on the 16384 packed-extend rows, 4336.33 MB +
# 0.23 MB per launch for 1079.8 M keys; fused prefill on 4096 rows, 39.10 MB
# + 0.06 MB for 125.8 M keys; fused decode on 64 rows, 159.08 MB + 1.45 MB
# for 1.19 M keys; the bf16-cache kernels on the same shapes, 76.88 MB +
# 2.23 MB (prefill) and 312.57 MB + 2.37 MB (decode). Traffic grows with the
# keys streamed. Set an entry to None whenever its kernel changes until it
# is re-captured.
TRAFFIC_BYTES_PER_KEY = {
    "topk_packed_extend": (21681633536 + 1127424) / 5 / 1079779328,
    "fused_prefill": (195485952 + 288768) / 5 / 125831168,
    "fused_decode": (795407616 + 7244544) / 5 / 1190814,
    "fused_prefill_bf16": (384384256 + 11137792) / 5 / 125831168,
    "fused_decode_bf16": (1562842624 + 11865856) / 5 / 1190814,
}


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def _max_over_ranks(x: float, world: int, device) -> float:
    """The largest x over the ranks: the job's time is its slowest rank's."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _job_rate(rows_per_rank: int, world: int, ms: float) -> float:
    """Whole-job rows/s: every rank runs its own replica of the step (weak
    scaling, no data-path collective), the job takes `ms` per step."""
    return rows_per_rank * world / (ms * 1e-3)


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
def _bind_host_to_gpu(local: int) -> str:
    """Run this process on the CPUs next to the GPU, so that the host buffers
    of the end-to-end timing are allocated (first touch) in that CPU's memory
    and copied over its own link rather than across sockets. Returns a note
    for the JSON line."""
    try:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        idx = vis.split(",")[local] if vis else str(local)
        bus = subprocess.run(["nvidia-smi", "--query-gpu=pci.bus_id", "--format=csv,noheader", "-i", idx],
                             capture_output=True, text=True, timeout=20).stdout.strip().lower()
        dom, b, rest = bus.split(":")
        path = f"/sys/bus/pci/devices/{dom[-4:]}:{b}:{rest}/local_cpulist"
        with open(path) as f:
            spec = f.read().strip()
        cpus = set()
        for part in spec.split(","):
            if "-" in part:
                lo, hi = part.split("-")
                cpus.update(range(int(lo), int(hi) + 1))
            elif part:
                cpus.add(int(part))
        cpus &= os.sched_getaffinity(0)
        if not cpus:
            return "host affinity unchanged (no local CPUs listed)"
        os.sched_setaffinity(0, cpus)
        return f"host threads on the GPU's {len(cpus)} local CPUs"
    except Exception as exc:  # no sysfs entry, other platforms
        return f"host affinity unchanged ({type(exc).__name__})"


class Part:
    """One part of the step: host (pinned) inputs, device copies, outputs."""

    def __init__(self, name):
        self.name = name
        self.host = {}      # name -> pinned host tensor
        self.dev = {}       # name -> device tensor
        self.out = {}       # name -> device output tensor
        self.rows = 0
        self.keys = 0.0
        self.bytes = 0.0    # algorithmic HBM bytes per launch (each input byte once)
        self.l2_bytes = 0.0  # bytes the kernels stream, re-reads served by L2 included
        self.flops = 0.0    # algorithmic tensor flops per launch
        self.launches = 0
        self.meta = {}
        self.uploads = None  # [(device view, pinned host tensor)]; None: every host tensor to its device copy

    def upload_pairs(self):
        """The host-to-device copies of this part's inputs for one step."""
        if self.uploads is not None:
            return self.uploads
        return [(self.dev[k], t) for k, t in self.host.items()]


def _pin(a):
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.pin_memory()


def build_topk_part(dev, new_tokens: int, name: str = "topk_packed_extend"):
    import torch

    import workloads as W

    part = Part(name)
    row_starts, seq_lens, r2b, width = W.packed_extend_meta(new_tokens=new_tokens)
    rows = int(seq_lens.size)
    reqs = int(r2b.max()) + 1
    per_req = width // reqs  # columns of the shared buffer one request's windows lie in
    # Host side: each request's [rows of the request, its columns] block,
    # pinned and contiguous; the rest of the shared buffer is never read.
    blocks = [torch.empty((new_tokens, per_req), dtype=torch.float32, pin_memory=True) for _ in range(reqs)]
    chunk = 1024
    tmp = np.empty((chunk, width), dtype=np.float32)
    for r0 in range(0, rows, chunk):
        n = min(chunk, rows - r0)
        W.fill_rows(tmp[:n], r0, 3, row_starts, seq_lens, fill=0.0)
        for q in range(reqs):  # rows r0 .. r0+n-1 of request q, if any
            a, b = max(r0, q * new_tokens), min(r0 + n, (q + 1) * new_tokens)
            if a < b:
                blocks[q].numpy()[a - q * new_tokens:b - q * new_tokens] = tmp[a - r0:b - r0, q * per_req:(q + 1) * per_req]
    pt = W.page_table_perm(3, (2, 70000))
    part.host = {"seq_lens": _pin(seq_lens), "row_starts": _pin(row_starts), "row_to_batch": _pin(r2b),
                 "page_tables": _pin(pt)}
    part.dev = {k: v.to(dev) for k, v in part.host.items()}
    scores = torch.zeros((rows, width), dtype=torch.float32, device=dev)
    views = [scores[q * new_tokens:(q + 1) * new_tokens, q * per_req:(q + 1) * per_req] for q in range(reqs)]
    for v, h in zip(views, blocks):
        v.copy_(h)
    part.dev["scores"] = scores
    part.uploads = [(part.dev[k], t) for k, t in part.host.items()] + list(zip(views, blocks))
    import sparse_attention_indexer_top_gb300 as sai

    ws = sai.topk_transform_workspace(rows, width)
    part.out = {"slots": torch.empty((rows, K), dtype=torch.int32, device=dev),
                "workspace": torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)}
    if name == "topk_blocks":  # the same call also writes each row's 128-token block list
        part.out["blocks"] = torch.empty((rows, K), dtype=torch.int32, device=dev)
        part.out["counts"] = torch.empty((rows,), dtype=torch.int32, device=dev)
    part.rows = rows
    part.keys = float(seq_lens.astype(np.int64).sum())
    part.bytes = part.keys * 4 + pt.nbytes + rows * (3 * 4 + K * 4)
    if name == "topk_blocks":
        part.bytes += rows * (K * 4 + 4)
    part.launches = 1
    part.meta = dict(row_starts=row_starts, seq_lens=seq_lens, row_to_batch=r2b, page_tables=pt, width=width)
    return part


def build_fused_part(dev, name: str, inp, group_rows: int):
    import torch

    part = Part(name)
    arrays = {"q": inp.q, "w": inp.w, "kcache": inp.kcache, "kscale": inp.kscale,
              "block_table": inp.block_table, "seq_lens": inp.seq_lens}
    if inp.row_to_batch is not None:
        arrays["row_to_batch"] = inp.row_to_batch
    part.host = {k: _pin(v) for k, v in arrays.items()}
    if inp.dtype == "bf16":  # uint16 bit patterns, handed over as torch.bfloat16
        for k in ("q", "kcache"):
            part.host[k] = _pin(arrays[k].view(np.int16)).view(torch.bfloat16)
    part.dev = {k: v.to(dev) for k, v in part.host.items()}
    rows = inp.rows
    part.out = {"slots": torch.empty((rows, K), dtype=torch.int32, device=dev),
                "indices": torch.empty((rows, K), dtype=torch.int32, device=dev),
                "scores": torch.empty((rows, K), dtype=torch.float32, device=dev)}
    import sparse_attention_indexer_top_gb300 as sai

    max_len = int(inp.seq_lens.max())
    ws = sai.index_score_topk_workspace(rows, max_len, group_rows)
    part.out["workspace"] = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
    part.rows = rows
    n = inp.seq_lens.astype(np.int64)
    part.keys = float(n.sum())
    h, d = inp.heads, inp.dim
    # each key's row (fp8 or bf16) + its scale, read once per row group; q, w;
    # block ids; outputs
    groups = -(-rows // group_rows)
    key_bytes = d * inp.kcache.itemsize + 4  # a key row and its scale
    # keys streamed by the kernel: once per row group (L2 serves the re-reads
    # of a request's keys by its other groups)
    key_reads = float(sum(int(n[g * group_rows:(g + 1) * group_rows].max()) for g in range(groups)))
    # distinct keys, read once from HBM: per block-table row, its longest row
    batch = np.arange(rows) if inp.row_to_batch is None else inp.row_to_batch
    key_unique = float(sum(int(n[batch == b].max()) for b in np.unique(batch)))
    fixed = inp.q.nbytes + inp.w.nbytes + rows * K * 12
    part.bytes = key_unique * (key_bytes + 4 / 128) + fixed
    part.l2_bytes = key_reads * (key_bytes + 4 / 128) + fixed
    part.flops = part.keys * h * d * 2.0
    part.launches = 2
    part.meta = dict(inp=inp, group_rows=group_rows, max_len=max_len)
    return part


def build_topk_decode_part(dev):
    """The decode-layout top-k: 128 rows, seq_lens U[8192, 32768], bf16-rounded
    N(0,1) scores in a [128, 32768] buffer (ties certain), 128-token pages
    (slot = block*128 + idx%128). Rows of up to 32768 scores: one CTA each.
    Not part of the default step (it is launch-latency bound)."""
    import torch

    import workloads as W

    inp = W.decode_topk()
    part = Part("topk_decode")
    part.host = {"scores": _pin(inp.scores), "seq_lens": _pin(inp.seq_lens), "page_tables": _pin(inp.page_tables)}
    part.dev = {k: v.to(dev) for k, v in part.host.items()}
    import sparse_attention_indexer_top_gb300 as sai

    rows = int(inp.seq_lens.size)
    ws = sai.topk_transform_workspace(rows, inp.scores.shape[1])
    part.out = {"slots": torch.empty((rows, K), dtype=torch.int32, device=dev),
                "workspace": torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)}
    part.rows = rows
    part.keys = float(inp.seq_lens.astype(np.int64).sum())
    part.bytes = part.keys * 4 + rows * (4 + K * 4 + K * 4)  # scores, lens, slots, <= k table reads
    part.launches = 2
    part.meta = dict(inp=inp)
    return part


def build_per_head_part(dev):
    """Per-index-head top-k on the fused decode workload (64 rows, 64 heads x
    128 e4m3, U[4096, 32768] keys): 4096 (row, head) selections. Not part of
    the default step (a variant). Bytes: the key stream and the outputs (a
    single-pass kernel's traffic); the library's two-stage design also writes
    and reads a [4096, 32768] fp32 score buffer."""
    import torch

    import workloads as W

    inp = W.fused_decode()
    part = build_fused_part(dev, "per_head_decode", inp, 1)
    rows = inp.rows
    import sparse_attention_indexer_top_gb300 as sai

    max_len = int(inp.seq_lens.max())
    part.out = {"slots": torch.empty((rows, 64, K), dtype=torch.int32, device=dev),
                "indices": torch.empty((rows, 64, K), dtype=torch.int32, device=dev)}
    ws = sai.index_score_topk_per_head_workspace(rows, max_len)
    part.out["workspace"] = torch.empty(max(ws, 256), dtype=torch.uint8, device=dev)
    n = inp.seq_lens.astype(np.int64)
    part.bytes = float(n.sum()) * (inp.dim + 4) + inp.q.nbytes + inp.w.nbytes + rows * 64 * K * 8
    part.launches = 3
    return part


def build_sparse_blocks_part(dev):
    """Per-row block lists of a packed-extend-sized top-k output: 16384 rows
    of 512 token slots of a 140000-slot pool (page_size 1), 128-token blocks.
    Not part of the default step (a follow-on of the top-k)."""
    import torch

    rng = np.random.default_rng(6)
    rows = 16384
    slots = rng.integers(0, 140000, size=(rows, K)).astype(np.int32)
    part = Part("sparse_blocks")
    part.host = {"slots": _pin(slots)}
    part.dev = {k: v.to(dev) for k, v in part.host.items()}
    part.out = {"blocks": torch.empty((rows, K), dtype=torch.int32, device=dev),
                "counts": torch.empty((rows,), dtype=torch.int32, device=dev)}
    part.rows = rows
    part.keys = float(rows * K)
    part.bytes = rows * K * 4 * 2 + rows * 4
    part.launches = 1
    part.meta = dict(slots=slots)
    return part


def build_parts(dev, args):
    import workloads as W

    parts = []
    if "topk_packed_extend" in args.paths:
        parts.append(build_topk_part(dev, args.new_tokens))
    if "topk_blocks" in args.paths:
        parts.append(build_topk_part(dev, args.new_tokens, "topk_blocks"))
    if "fused_decode" in args.paths:
        parts.append(build_fused_part(dev, "fused_decode", W.fused_decode(), 1))
    if "fused_prefill" in args.paths:
        parts.append(build_fused_part(dev, "fused_prefill", W.fused_prefill(rows=args.prefill_rows), 4))
    if "fused_decode_bf16" in args.paths:
        parts.append(build_fused_part(dev, "fused_decode_bf16", W.fused_decode(dtype="bf16"), 1))
    if "fused_prefill_bf16" in args.paths:
        parts.append(build_fused_part(dev, "fused_prefill_bf16", W.fused_prefill(rows=args.prefill_rows, dtype="bf16"),
                                      4))
    if "sparse_blocks" in args.paths:
        parts.append(build_sparse_blocks_part(dev))
    if "per_head_decode" in args.paths:
        parts.append(build_per_head_part(dev))
    if "topk_decode" in args.paths:
        parts.append(build_topk_decode_part(dev))
    return parts


def launch_part(part, stream):
    import sparse_attention_indexer_top_gb300 as sai

    d, o = part.dev, part.out
    if part.name == "sparse_blocks":
        sai.sparse_blocks(d["slots"], 128, out_blocks=o["blocks"], out_counts=o["counts"], stream=stream)
    elif part.name == "per_head_decode":
        sai.index_score_topk_per_head(d["q"], d["w"], d["kcache"], d["kscale"], d["block_table"], d["seq_lens"],
                                      max_seq_len=part.meta["max_len"], row_to_batch=d.get("row_to_batch"),
                                      out_slots=o["slots"], out_indices=o["indices"], workspace=o["workspace"],
                                      stream=stream)
    elif part.name == "topk_decode":
        sai.topk_transform(d["scores"], d["seq_lens"], d["page_tables"], page_size=128, out_slots=o["slots"],
                           workspace=o["workspace"], stream=stream)
    elif part.name == "topk_packed_extend":
        sai.topk_transform(d["scores"], d["seq_lens"], d["page_tables"], row_starts=d["row_starts"],
                           row_to_batch=d["row_to_batch"], out_slots=o["slots"], workspace=o["workspace"],
                           stream=stream)
    elif part.name == "topk_blocks":
        sai.topk_transform(d["scores"], d["seq_lens"], d["page_tables"], row_starts=d["row_starts"],
                           row_to_batch=d["row_to_batch"], out_slots=o["slots"], block_size=128,
                           out_blocks=o["blocks"], out_counts=o["counts"], workspace=o["workspace"], stream=stream)
    else:
        sai.index_score_topk(d["q"], d["w"], d["kcache"], d["kscale"], d["block_table"], d["seq_lens"],
                             max_seq_len=part.meta["max_len"], row_to_batch=d.get("row_to_batch"),
                             group_rows=part.meta["group_rows"], out_slots=o["slots"], out_indices=o["indices"],
                             out_scores=o["scores"], workspace=o["workspace"], stream=stream)


# --------------------------------------------------------------------------- oracle
# The CPU oracle, timed on the host cores: a pool of worker processes (spawn,
# one per core), each running the oracle on its share of a part's rows until
# its time budget is spent. Only the oracle calls are timed; loading the
# inputs (memory-mapped .npy files written by the parent) and regenerating a
# top-k window from its seed are not. A part's rate is the rows all workers
# finished divided by the longest worker's oracle time (they run at once).
_ORACLE_INPUTS = {}


def _oracle_warm(_):
    import oracle.blocks  # noqa: F401
    import oracle.score  # noqa: F401
    import oracle.topk  # noqa: F401
    import workloads  # noqa: F401

    return os.getpid()


def _oracle_inputs(spec):
    key = spec.get("folder") or spec["kind"]
    if key not in _ORACLE_INPUTS:
        import workloads as W

        arr = {}
        if "folder" in spec:
            for f in os.listdir(spec["folder"]):
                arr[f[:-4]] = np.load(os.path.join(spec["folder"], f), mmap_mode="r")
        if spec["kind"] == "fused":
            r2b = arr.get("row_to_batch")
            arr = W.FusedInputs(arr["q"], arr["w"], arr["kcache"], arr.get("kscale"), arr["block_table"],
                                np.asarray(arr["seq_lens"]), None if r2b is None else np.asarray(r2b),
                                dtype=spec["dtype"])
        _ORACLE_INPUTS[key] = arr
    return _ORACLE_INPUTS[key]


def _oracle_rows(task):
    """Worker: the oracle on `rows` of one part until `budget` seconds of
    oracle time are spent. Returns (rows done, oracle seconds)."""
    import workloads as W
    from oracle.blocks import sparse_blocks as oracle_blocks
    from oracle.score import index_score_topk as oracle_fused
    from oracle.score import index_score_topk_per_head
    from oracle.topk import topk_transform as oracle_topk

    name, spec, rows, budget = task
    data = _oracle_inputs(spec)
    done, spent = 0, 0.0
    for i in rows:
        i = int(i)
        if name in ("topk_packed_extend", "topk_blocks"):
            n = int(spec["seq_lens"][i])
            w = W.packed_extend_window(3, i, n)
            t0 = time.perf_counter()
            sl, _ = oracle_topk(w[None, :], np.array([n]), spec["page_tables"][[int(spec["row_to_batch"][i])]], 1, K)
            if name == "topk_blocks":
                oracle_blocks(sl, 128)
        elif name == "topk_decode":
            n = int(data["seq_lens"][i])
            t0 = time.perf_counter()
            oracle_topk(np.asarray(data["scores"][i:i + 1, :n]), np.array([n]), data["page_tables"][i:i + 1], 128, K)
        elif name == "sparse_blocks":  # 64 rows per item
            t0 = time.perf_counter()
            oracle_blocks(np.asarray(data["slots"][64 * i:64 * i + 64]), 128)
        elif name == "per_head_decode":
            t0 = time.perf_counter()
            index_score_topk_per_head(data, rows=[i])
        else:
            t0 = time.perf_counter()
            oracle_fused(data, rows=[i])
        spent += time.perf_counter() - t0
        done += 64 if name == "sparse_blocks" else 1
        if spent > budget:
            break
    return done, spent


def _oracle_specs(parts_meta, folder):
    """Per part: (name, rows of the step, worker input spec, item order)."""
    specs = []
    for name, nrows, meta in parts_meta:
        if name in ("topk_packed_extend", "topk_blocks"):
            spec = dict(kind="packed", seq_lens=meta["seq_lens"], row_to_batch=meta["row_to_batch"],
                        page_tables=meta["page_tables"])
            items = np.arange(nrows)
        else:
            sub = os.path.join(folder, name)
            os.makedirs(sub)
            if name == "sparse_blocks":
                arrays, spec = {"slots": meta["slots"]}, dict(kind="blocks")
                items = np.arange(nrows // 64)
            elif name == "topk_decode":
                inp = meta["inp"]
                arrays = {"scores": inp.scores, "seq_lens": inp.seq_lens, "page_tables": inp.page_tables}
                spec, items = dict(kind="topk"), np.arange(nrows)
            else:
                inp = meta["inp"]
                arrays = {f: getattr(inp, f) for f in ("q", "w", "kcache", "kscale", "block_table", "seq_lens",
                                                       "row_to_batch")}
                spec, items = dict(kind="fused", dtype=inp.dtype), np.arange(nrows)
            for f, a in arrays.items():
                if a is not None:
                    np.save(os.path.join(sub, f + ".npy"), np.ascontiguousarray(a))
            spec["folder"] = sub
        # spread each worker's items over the whole part (row lengths vary along it)
        rng = np.random.default_rng(11)
        specs.append((name, nrows, spec, rng.permutation(items)))
    return specs


class OraclePool:
    """The oracle's worker pool over the host cores (spawn start method: a
    process forked after CUDA was used can hang)."""

    def __init__(self, parts_meta, workers=None):
        import multiprocessing as mp
        import tempfile

        for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[v] = "1"  # one BLAS thread per worker process
        self.workers = workers or len(os.sched_getaffinity(0))
        self._tmp = tempfile.TemporaryDirectory()
        self.specs = _oracle_specs(parts_meta, self._tmp.name)
        self.pool = mp.get_context("spawn").Pool(self.workers)
        self.pool.map(_oracle_warm, range(self.workers))

    def close(self):
        self.pool.close()
        self.pool.join()
        self._tmp.cleanup()

    def step_rate(self, budget_s):
        """Rows/s of the oracle over the step's row mix (all workers), the
        same for one core, and a note on the sample."""
        per_step, per_step_1, rows, notes = 0.0, 0.0, 0, []
        budget = budget_s / max(len(self.specs), 1)
        for name, nrows, spec, items in self.specs:
            tasks = [(name, spec, items[w::self.workers], budget) for w in range(self.workers)]
            res = self.pool.map(_oracle_rows, tasks)
            done = sum(r[0] for r in res)
            longest = max(r[1] for r in res)
            total = sum(r[1] for r in res)
            per_step += nrows * longest / max(done, 1)
            per_step_1 += nrows * total / max(done, 1)
            rows += nrows
            notes.append(f"{name}: {done} of {nrows} rows in {longest:.1f} s on {self.workers} processes "
                         f"({total:.1f} s of oracle time)")
        return rows / per_step, rows / per_step_1, "; ".join(notes)


def _parts_meta_for_reference(args):
    import workloads as W

    metas = []
    if "topk_packed_extend" in args.paths:
        row_starts, seq_lens, r2b, width = W.packed_extend_meta(new_tokens=args.new_tokens)
        metas.append(("topk_packed_extend", int(seq_lens.size),
                      dict(row_starts=row_starts, seq_lens=seq_lens, row_to_batch=r2b,
                           page_tables=W.page_table_perm(3, (2, 70000)))))
    if "fused_decode" in args.paths:
        inp = W.fused_decode()
        metas.append(("fused_decode", inp.rows, dict(inp=inp)))
    if "fused_prefill" in args.paths:
        inp = W.fused_prefill(rows=args.prefill_rows)
        metas.append(("fused_prefill", inp.rows, dict(inp=inp)))
    for dt_name, make in (("fused_decode_bf16", lambda: W.fused_decode(dtype="bf16")),
                          ("fused_prefill_bf16", lambda: W.fused_prefill(rows=args.prefill_rows, dtype="bf16"))):
        if dt_name in args.paths:
            inp = make()
            metas.append((dt_name, inp.rows, dict(inp=inp)))
    return metas


def run_reference(args):
    rank, world, _ = _dist()
    if rank != 0:
        return
    pool = OraclePool(_parts_meta_for_reference(args))
    budget = max(3.0, 150.0 / max(1, args.steps + args.warmup))
    vals, note, one = [], "", 0.0
    try:
        for s in range(args.warmup + args.steps):
            v, one, note = pool.step_rate(budget)
            if s >= args.warmup:
                vals.append(v)
    finally:
        pool.close()
    value = float(np.median(vals))
    rows = sum(m[1] for m in pool.specs)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": rows / value * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": {"workload": WORKLOAD},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": pool.workers, "kind": "oracle",
                             "one_core_value": one,
                             "sample": (f"per step, a bounded row sample of each part (about {budget:.0f} s of wall "
                                        f"time over {pool.workers} worker processes); ms_per_step is extrapolated "
                                        f"from the sample's rate to the whole step; last step: {note}")},
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
    hbm_peak, bf16_peak, peak_kind = _peaks()
    fp8_peak, fp8_note = measure_fp8_peak(dev)
    if fp8_peak is not None:
        fp8_kind = f"measured fp8 burst on this GPU: {fp8_note}"
    else:
        fp8_peak = bf16_peak * FP8_OVER_BF16
        fp8_kind = f"{peak_kind} bf16 burst x {FP8_OVER_BF16} (nominal fp8/bf16; {fp8_note})"

    host_note = _bind_host_to_gpu(local)
    parts = build_parts(dev, args)
    stream = torch.cuda.Stream(device=dev)

    def step():
        for part in parts:
            launch_part(part, stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    assert sai.device_status() == 0, "a kernel flagged its inputs"

    # timed region
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in parts]
          for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # L2 flush before every timed step (outside the step's events): a write of
    # twice the L2 size, so no part finds its inputs cached from the last step
    l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0)) or (128 << 20)
    flush = torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev)
    with ClockSampler(local) as clk:
        t0 = time.perf_counter()
        for s in range(args.steps):
            with torch.cuda.stream(stream):
                flush.fill_(s & 0xFF)
            for j, part in enumerate(parts):
                ev[s][j][0].record(stream)
                launch_part(part, stream)
                ev[s][j][1].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    # medians over the timed steps
    part_ms = [float(np.median([ev[s][j][0].elapsed_time(ev[s][j][1]) for s in range(args.steps)]))
               for j in range(len(parts))]
    ms = float(np.median([ev[s][0][0].elapsed_time(ev[s][-1][1]) for s in range(args.steps)]))
    ms = _max_over_ranks(ms, world, dev)
    rows = sum(p.rows for p in parts)
    value = _job_rate(rows, world, ms)

    paths = {}
    for part, pm in zip(parts, part_ms):
        entry = {"ms": pm, "rows_per_s": part.rows / (pm * 1e-3), "keys_per_s": part.keys / (pm * 1e-3),
                 "hbm_gbs": part.bytes / (pm * 1e-3) / 1e9, "hbm_frac": part.bytes / (pm * 1e-3) / 1e9 / hbm_peak}
        if part.l2_bytes > part.bytes:  # re-reads of a request's keys, served by L2
            entry["l2_gbs"] = part.l2_bytes / (pm * 1e-3) / 1e9
        if part.flops:
            entry["tflops"] = part.flops / (pm * 1e-3) / 1e12
            if part.name.endswith("_bf16"):
                entry["bf16_frac"] = entry["tflops"] / bf16_peak
            else:
                entry["fp8_frac"] = entry["tflops"] / fp8_peak
        paths[part.name] = entry
    if "topk_blocks" in paths and "topk_packed_extend" in paths:
        added = paths["topk_blocks"]["ms"] - paths["topk_packed_extend"]["ms"]
        entry = {"added_ms_in_topk": added}
        if "sparse_blocks" in paths:
            entry["separate_pass_ms"] = paths["sparse_blocks"]["ms"]
        paths["block_lists"] = entry
    # Report-only parts (default: the decode-layout top-k, the latency-bound
    # serving shape): timed after the step with their own events and an L2
    # flush before each launch, not part of the step or its rate.
    report = [n for n in args.report if n not in args.paths]
    if report:
        rparts = build_parts(dev, argparse.Namespace(**{**vars(args), "paths": report}))
        for part in rparts:
            with torch.cuda.stream(stream):
                for _ in range(args.warmup):
                    launch_part(part, stream)
            torch.cuda.synchronize()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
            for e0, e1 in evs:
                with torch.cuda.stream(stream):
                    flush.fill_(1)
                e0.record(stream)
                launch_part(part, stream)
                e1.record(stream)
            torch.cuda.synchronize()
            pm = float(np.median([e0.elapsed_time(e1) for e0, e1 in evs]))
            paths[part.name] = {"ms": pm, "rows_per_s": part.rows / (pm * 1e-3), "keys_per_s": part.keys / (pm * 1e-3),
                                "hbm_gbs": part.bytes / (pm * 1e-3) / 1e9,
                                "hbm_frac": part.bytes / (pm * 1e-3) / 1e9 / hbm_peak, "in_step": False}
        assert sai.device_status() == 0, "a kernel flagged its inputs"
    # the dominant kernel's roofline
    top = int(np.argmax(part_ms))
    tp, tm = parts[top], part_ms[top]
    if tp.name == "fused_prefill":
        roof = {"bound": "tensor", "achieved": tp.flops / (tm * 1e-3) / 1e12, "peak": fp8_peak, "unit": "TFLOP/s",
                "peak_kind": fp8_kind}
    elif tp.name == "fused_prefill_bf16":
        roof = {"bound": "tensor", "achieved": tp.flops / (tm * 1e-3) / 1e12, "peak": bf16_peak, "unit": "TFLOP/s",
                "peak_kind": f"{peak_kind} bf16 burst"}
    else:
        roof = {"bound": "hbm", "achieved": tp.bytes / (tm * 1e-3) / 1e9, "peak": hbm_peak, "unit": "GB/s",
                "peak_kind": peak_kind}
    roof["frac"] = roof["achieved"] / roof["peak"]
    per_key = TRAFFIC_BYTES_PER_KEY.get(tp.name)
    roof["traffic"] = None if per_key is None else per_key * tp.keys
    roof["kernel"] = tp.name

    # end to end: every input copied from pinned host memory, every output read back
    e2e = None
    if not args.no_e2e:
        outs_host = {(p.name, k): torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
                     for p in parts for k, v in p.out.items() if k != "workspace"}
        h2d = sum(t.numel() * t.element_size() for p in parts for _, t in p.upload_pairs())
        d2h = sum(t.numel() * t.element_size() for t in outs_host.values())
        # Steps are pipelined over two streams: a step's large uploads (the
        # top-k score blocks, the decode key cache) go on a copy stream as soon
        # as the previous step's calls that read them are done, overlapping
        # that step's remaining calls and read-back; the small uploads, every
        # call and the read-back stay on the compute stream. Two untimed steps
        # first (the first uploads also allocate the staging buffers of the
        # strided copies), then the time of n steps from an idle start.
        copy_stream = torch.cuda.Stream(device=dev)
        big = {id(p): [(d, t) for d, t in p.upload_pairs() if t.numel() * t.element_size() >= (64 << 20)]
               for p in parts}
        small = {id(p): [(d, t) for d, t in p.upload_pairs() if t.numel() * t.element_size() < (64 << 20)]
                 for p in parts}
        last_big = [p for p in parts if big[id(p)]][-1] if any(big[id(p)] for p in parts) else parts[-1]
        n_e2e = max(1, min(5, args.steps))
        n_warm = max(2, min(args.warmup, 5))
        read_done = torch.cuda.Event()  # the last step's calls that read a large upload are done
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)

        def e2e_step():
            copy_stream.wait_event(read_done)
            with torch.cuda.stream(copy_stream):
                for p in parts:
                    for dst, t in big[id(p)]:
                        dst.copy_(t, non_blocking=True)
            uploaded = torch.cuda.Event()
            uploaded.record(copy_stream)
            with torch.cuda.stream(stream):
                for p in parts:
                    for dst, t in small[id(p)]:
                        dst.copy_(t, non_blocking=True)
                stream.wait_event(uploaded)
                for p in parts:
                    launch_part(p, stream)
                    if p is last_big:  # every call that reads a large upload is issued
                        read_done.record(stream)
                for p in parts:
                    for k, v in p.out.items():
                        if k != "workspace":
                            outs_host[(p.name, k)].copy_(v, non_blocking=True)

        read_done.record(stream)
        for _ in range(n_warm):
            e2e_step()
        torch.cuda.synchronize()
        e0.record(stream)
        copy_stream.wait_event(e0)
        for _ in range(n_e2e):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / n_e2e
        e2e = {"value": rows / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    cpu = None
    if rank == 0 and not args.no_cpu:
        pool = OraclePool([(p.name, p.rows, p.meta) for p in parts])
        try:
            v, one, note = pool.step_rate(20.0)
        finally:
            pool.close()
        cpu = {"value": v, "unit": UNIT, "cores": pool.workers, "kind": "oracle", "one_core_value": one,
               "sample": f"a bounded row sample of each part (about 20 s of wall time), rate extrapolated to the "
                         f"step's rows: {note}"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32 (top-k), e4m3 x e4m3 -> f32 (fused scores)", "data": "synthetic",
            "config": {"workload": WORKLOAD, "rows_per_step": rows, "k": K,
                       "l2": "flushed before every timed step (write of 2x L2); step inputs 4.5 GB", "host": host_note, "paths": paths},
            "roofline": roof,
            "e2e": e2e,
            "gpu_launches": sum(p.launches for p in parts) * args.steps,
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
    ap.add_argument("--paths", default=",".join(PATHS), help="comma-separated parts of the step")
    ap.add_argument("--report", default="topk_decode",
                    help="comma-separated parts timed after the step, outside it (reported in config.paths)")
    ap.add_argument("--new-tokens", type=int, default=8192,
                    help="query rows per request of the packed-extend part (8192 = full chunk)")
    ap.add_argument("--prefill-rows", type=int, default=4096, help="query rows of the fused prefill part")
    args = ap.parse_args()
    args.paths = [p for p in args.paths.split(",") if p]
    args.report = [p for p in args.report.split(",") if p]
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
