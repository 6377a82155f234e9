"""Benchmark: decode top-2048 sparse-attention indexer on GB300.

One step = one pass of the decode hot path over the decode-batch workload
(32 requests, next_n 1, seq_lens uniform in [2048, 32768], 64 heads x 128,
fp8 e4m3 paged index cache, top-2048): row expansion + q quantisation +
paged gather + tensor-core scoring + causal mask + top-k, through the C ABI.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line. ``value`` is indexed keys/s (sum over token rows of the
keys each row scores) over all ranks, device-timed with CUDA events around a
CUDA graph of K steps (inputs resident in HBM, cold L2: every step reads a
different copy of the index cache, the copies together several times L2).
``e2e`` is the same metric with pinned host buffers copied in and the indices
copied out every step. ``--impl reference`` times the CPU oracle on the host
cores instead (bounded sample per step). Multi-GPU runs are replicas: every
rank runs its own batch (weak scaling), no collective on the data path.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "indexed keys/sec for decode top-2048; % of HBM roofline (1×GB300)"
WORKLOAD = "decode"
WORKLOAD_DESC = ("decode batch: 32 requests, next_n 1, seq_lens uniform in [2048, 32768], "
                 "64 index heads x head_dim 128, bf16 q, fp8 e4m3 paged index-K (page 64, "
                 "fp32 per-token scale), random block table, top-2048")
PAGE_KEY_BYTES = 132  # 128 fp8 values + 4-byte scale per key
MX_KEY_BYTES = 68     # 64 bytes of packed e2m1 values + 4 ue8m0 block scales per key


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--record-counters", metavar="NCU_REPORT",
                    help="store the DRAM and tensor-pipe counters of the one score/select "
                         "launch in this ncu report as --workload's entry of "
                         "profiles/score_select_counters.json, then exit")
    ap.add_argument("--no-extra-configs", action="store_true",
                    help="measure only --workload (by default the decode-batch run also "
                         "measures the long-context and MTP configurations)")
    ap.add_argument("--seed", type=int, default=0x5EED)
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_seed(base: int, rank: int) -> int:
    """Each replica draws its own batch."""
    return base + 1000 * rank


def max_over_ranks(values, world: int, device="cpu"):
    """Element-wise max of a list of floats over all ranks (identity for one rank).
    The reduction runs on `device` (a CUDA device under NCCL, the CPU under gloo)."""
    if world == 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def whole_job_rate(units_per_rank_step: int, steps: int, world: int, ms: float) -> float:
    """Units all ranks processed per second, timed by the slowest rank (ms)."""
    return units_per_rank_step * steps * world / (ms / 1e3)


WORKLOAD_DESCS = {
    "decode": WORKLOAD_DESC,
    "mtp": ("MTP decode: 64 requests, next_n 2, decode_lens from {1, 2}, seq_lens uniform in "
            "[4096, 65536], 64 index heads x 128, fp8 e4m3 paged index-K, top-2048"),
    "long": ("long context: 128 requests, next_n 1, seq_len 131072, 1% heavy-tail keys, "
             "64 index heads x 128, fp8 e4m3 paged index-K, top-2048"),
    "tiny": ("tiny decode: 4 requests, next_n 1, seq_lens {1000, 2048, 3000, 4096}, "
             "64 index heads x 128, fp8 e4m3 paged index-K, top-2048"),
    "decode_mxfp4": ("decode batch with MXFP4 index keys: 32 requests, next_n 1, seq_lens "
                     "uniform in [2048, 32768], 64 index heads x 128, 68-byte e2m1 + ue8m0 keys, "
                     "top-2048"),
    "long_mxfp4": ("long context with MXFP4 index keys: 128 requests, next_n 1, seq_len 131072, "
                   "64 index heads x 128, 68-byte e2m1 + ue8m0 keys, top-2048"),
    "long_blocks": ("long context (128 x 131072 keys, 1% heavy-tail), block selection: the "
                    "decode logits, then per row the 32 best 64-token blocks by their largest "
                    "logit plus the first and the last 4 blocks"),
    "dcp_long": ("long context (128 x 131072 keys, 1% heavy-tail) key-sharded over 2 decode-"
                 "context-parallel ranks in runs of 1 token, the ranks run one after the other "
                 "on one GPU: per rank top-2048 with logits over its 65536 keys per row, then "
                 "the merge of the ranks' candidates"),
}


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 20):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 f"-i", str(self.gpu), "-lms", str(self.period)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self._t.join(timeout=2)

    def summary(self, min_mhz_load: float = 500.0):
        sms, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm, smax = float(f[1]), float(f[2])
            except ValueError:
                continue
            sms.append(sm)
            mx.append(smax)
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        loaded = [s for s in sms if s >= min_mhz_load] or sms
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sms)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def measured_peak_gbs():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def kernel_code_hash(root: str) -> str:
    """First 16 hex digits of the sha256 of the score/select and split-row
    selection kernels' code (score_select.cu, row_select.cu, common.cuh,
    internal.h without comments or whitespace)."""
    import hashlib
    import re
    csrc = os.path.join(root, "sparse_attention_indexer_block_gb300", "csrc")
    h = hashlib.sha256()
    for name in ("score_select.cu", "row_select.cu", "common.cuh", "internal.h"):
        with open(os.path.join(csrc, name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def profiled_counters(workload: str):
    """The ncu counters of one score/select launch and the split-row selection
    launch after it on `workload` (DRAM bytes read + written, tensor-pipe
    activity of the score kernel), from profiles/score_select_counters.json, or
    None when they were taken on other kernel sources (or not at all)."""
    try:
        with open(os.path.join(ROOT, "profiles", "score_select_counters.json")) as f:
            entry = json.load(f).get(workload)
    except (OSError, ValueError):
        return None
    if not entry or entry.get("source_sha256_16") != kernel_code_hash(ROOT):
        return None
    return entry


def measured_peak_fp8_tflops():
    """Dense fp8 tensor peak: the measured bf16 burst figure x 2 (the nominal
    fp8:bf16 ratio), or the fallback 1.9 PFLOP/s bf16 x 2."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return 2.0 * float(json.load(f)["bf16_tflops"]), "measured bf16 burst x 2"
    except (OSError, KeyError, ValueError):
        return 3800.0, "fallback 1.9 PFLOP/s bf16 x 2"


def run_prefill(args, rank, world, local):
    """Prefill indexer (4 requests x 8192 causal queries, top-2048 per query)
    through indexer_prefill_topk, M*N logits-budget chunking included. The
    score is a dense fp8 contraction (64 heads x 128 per key and query), so the
    roofline is the fp8 tensor peak."""
    import torch

    import synth
    import sparse_attention_indexer_block_gb300 as saib
    from sparse_attention_indexer_block_gb300 import build as libbuild

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    libbuild.build()
    saib.load()
    d = synth.make_prefill("prefill", seed=rank_seed(args.seed, rank), device=dev)
    sl = d.seq_lens.cpu().numpy().astype(np.int64)
    ql = d.query_lens.cpu().numpy().astype(np.int64)
    # keys scored per step: query i of a request sees seq_len - query_len + i + 1 keys
    keys_per_step = int(sum(((L - n) * n + n * (n + 1) // 2) for L, n in zip(sl, ql)))
    flops_per_step = keys_per_step * 64 * 128 * 2
    k = d.topk
    out = torch.empty((int(ql.sum()), k), dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    chunks = saib.indexer_plan_prefill_chunks(sl, ql, 40 * 8192, 512 << 20)
    ws_n = saib.indexer_prefill_workspace_bytes(sl, ql, k, 40 * 8192, 512 << 20)
    ws = torch.empty(max(ws_n, 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(dev)

    def step():
        saib.indexer_prefill_topk(d.q, d.w, d.cache, d.block_table, d.seq_lens, d.query_start_loc,
                                  sl, ql, k, out_idx=out, workspace=ws, dev_error=err,
                                  stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            step()
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())} during warm-up")
    K = args.steps
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for _ in range(K):
                step()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_soak = time.time()
        with torch.cuda.stream(stream):
            while time.time() - t_soak < 1.0:
                g.replay()
                stream.synchronize()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
    ms = max_over_ranks([e0.elapsed_time(e1)], world, dev)[0]
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())} in the timed region")
    peak, peak_src = measured_peak_fp8_tflops()
    tflops = flops_per_step * K / (ms / 1e3) / 1e12
    if rank == 0:
        line = {"metric": "indexed keys/sec for prefill top-2048 (fp8 tensor roofline)",
                "value": whole_job_rate(keys_per_step, K, world, ms), "unit": "keys/s",
                "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": ms / K,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "fp8_e4m3 (fp32 accumulate)", "data": "synthetic",
                "config": {"workload": "prefill: 4 requests x 8192 queries causally over 8192 "
                                       "keys, 64 heads x 128, top-2048, 512 MiB logits budget",
                           "keys_per_step": keys_per_step, "flops_per_step": flops_per_step,
                           "timing": "CUDA events around a CUDA graph of K calls (whole path)",
                           "parallelism": f"replicas x{world}"},
                "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": peak,
                             "unit": "TFLOP/s", "frac": round(tflops / peak, 4),
                             "traffic": None, "peak_source": peak_src,
                             "scope": "whole prefill call (prep + score/select, all chunks)"},
                "clocks": clk.summary(), "gpu_launches": 2 * len(chunks) * K}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_insert(args, rank, world, local):
    """Index-key cache insert (the step that fills the cache the indexer
    reads): 1 Mi new tokens of bf16 keys quantised per token and written to
    their slots (pages in random order, tokens of a page contiguous, as a
    prefill's new tokens land). HBM-bound: 256 B of keys + 8 B of slot read
    and 132 B written per token."""
    import torch

    import sparse_attention_indexer_block_gb300 as saib
    from sparse_attention_indexer_block_gb300 import build as libbuild

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    libbuild.build()
    saib.load()
    T = 1 << 20
    g = torch.Generator(device=dev).manual_seed(rank_seed(args.seed, rank))
    pages = T // 64
    n_copies = 2  # alternate two input/output sets so no step finds its data in L2
    ks = [torch.randn((T, 128), generator=g, device=dev).to(torch.bfloat16)
          for _ in range(n_copies)]
    perm = torch.randperm(pages, generator=g, device=dev)
    slots = (perm.repeat_interleave(64) * 64 + torch.arange(T, device=dev) % 64).to(torch.int64)
    caches = [torch.zeros((pages, 8448), dtype=torch.uint8, device=dev) for _ in range(n_copies)]
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(dev)
    bytes_per_step = T * (256 + 8 + 132)

    def step(i):
        saib.indexer_insert_keys(ks[i % n_copies], slots, caches[i % n_copies], dev_error=err,
                                 stream=stream)

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            step(i)
    torch.cuda.synchronize()
    K = args.steps
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            for i in range(K):
                step(i)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            graph.replay()
            e0.record(stream)
            graph.replay()
            e1.record(stream)
        torch.cuda.synchronize()
    ms = max_over_ranks([e0.elapsed_time(e1)], world, dev)[0]
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())}")
    peak, peak_kind = measured_peak_gbs()
    gbs = bytes_per_step * K / (ms / 1e3) / 1e9
    if rank == 0:
        print(json.dumps({
            "metric": "index-key cache insert: tokens/s (HBM roofline)",
            "value": whole_job_rate(T, K, world, ms), "unit": "tokens/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": ms / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16 -> fp8_e4m3 + fp32 scale",
            "data": "synthetic",
            "config": {"workload": "insert 1 Mi tokens x 128 bf16 into a paged fp8 cache",
                       "bytes_per_step": bytes_per_step,
                       "timing": "CUDA events around a CUDA graph of K calls",
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(gbs / peak, 4), "traffic": None,
                         "peak_source": peak_kind},
            "clocks": clk.summary(), "gpu_launches": K}), flush=True)


def measure_decode(workload, seed, dev, steps, prof_steps, world, local, mx=False):
    """Device-timed decode steps on `workload` (expand + decode top-k through
    the C ABI, CUDA graphs of the K steps, every step on its own copy of the
    index cache so the copies together exceed L2 several times), the live mean
    duration of the score/select kernel (CUDA events on the launch stream) and
    the clocks sampled meanwhile. Returns a dict; the inputs for the end-to-end
    leg are in it too."""
    import torch

    import synth
    import sparse_attention_indexer_block_gb300 as saib

    if mx:  # the workload's lengths over MXFP4 keys (next_n 1)
        wl = synth.WORKLOADS[workload]
        sl = synth.draw_seq_lens(wl, seed)
        d = synth.make_decode_mxfp4_from_lens(sl, np.ones(len(sl), np.int32), 1, seed=seed,
                                              device=dev)
    else:
        d = synth.make_decode(workload, seed=seed, device=dev)
    R, G, k = d.num_reqs, d.next_n, d.topk
    seq_h = d.seq_lens.cpu().numpy().astype(np.int64)
    dl_h = d.decode_lens.cpu().numpy().astype(np.int64)
    # keys scored per step (sum of row lengths) and unique keys read
    row_lens_h = np.concatenate([[L - dd + j + 1 if j < dd else 0 for j in range(G)]
                                 for L, dd in zip(seq_h, dl_h)])
    keys_per_step = int(row_lens_h.sum())
    algo_bytes = int(seq_h.sum()) * (MX_KEY_BYTES if mx else PAGE_KEY_BYTES)

    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    cache_bytes = d.cache.numel()
    n_copies = max(2, math.ceil(3 * l2 / cache_bytes) + 1)
    caches = [d.cache] + [d.cache.clone() for _ in range(n_copies - 1)]
    ws = saib.decode_workspace(R, G, k, dev)
    out = torch.empty((R * G, k), dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(dev)

    # one step: the whole hot path from the requests' (seq_lens, decode_lens),
    # the row expansion (S1) done by the launch's first kernel
    def step(i):
        if mx:
            saib.indexer_decode_topk_mxfp4(d.q, d.w, caches[i % n_copies], d.block_table,
                                           d.seq_lens, k, out_idx=out, workspace=ws,
                                           dev_error=err, stream=stream)
            return
        saib.indexer_decode_topk_from_lens(d.q, d.w, caches[i % n_copies], d.block_table,
                                           d.seq_lens, d.decode_lens, G, k, out_idx=out,
                                           workspace=ws, dev_error=err, stream=stream)

    with torch.cuda.stream(stream):
        for i in range(3):
            step(i)
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())} during warm-up ({workload})")

    # CUDA graph of the K timed steps (replayed in pieces of at most 1000 steps)
    piece = min(steps, 1000)
    graphs = []
    done = 0
    with torch.cuda.stream(stream):
        while done < steps:
            n = min(piece, steps - done)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(done, done + n):
                    step(i)
            graphs.append(g)
            done += n
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    # soak (untimed) so the clock samples see the same load, then the timed region
    t_soak = time.time()
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            while time.time() - t_soak < 1.0:
                for g in graphs:
                    g.replay()
                stream.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for g in graphs:
                g.replay()
            e1.record(stream)
        barrier()
    ms = max_over_ranks([e0.elapsed_time(e1)], world, dev)[0]
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())} in the timed region ({workload})")

    # live per-launch duration of the score/select kernel (eager, same rotation)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(prof_steps)]
    for a, b in evs:  # torch creates the event handles on first record
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(prof_steps):
            saib.indexer_profile_events(*evs[i])
            step(i)
        saib.indexer_profile_events(None, None)
    torch.cuda.synchronize()
    kern_ms = [a.elapsed_time(b) for a, b in evs]
    kern_avg = statistics.mean(kern_ms)
    peak, peak_kind = measured_peak_gbs()
    achieved = algo_bytes / (kern_avg / 1e3) / 1e9
    counters = profiled_counters(workload + ("_mxfp4" if mx else ""))
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": counters["dram_bytes_per_launch"] if counters else None,
                "peak_source": peak_kind + " (MEASURED_PEAKS.json hbm_gbs)" if peak_kind ==
                "measured" else "fallback 6.8 TB/s",
                "traffic_source": ("ncu dram__bytes_read.sum + dram__bytes_write.sum of one "
                                   "score/select launch and its split-row selection launch "
                                   "on the same kernel sources, "
                                   "profiles/score_select_counters.json"),
                "kernel": f"score_select_kernel<{G},false,{'true' if mx else 'false'}> + "
                          "row_select_kernel (events around both launches)",
                "kernel_ms_avg": round(kern_avg, 5),
                "kernel_ms_median": round(statistics.median(kern_ms), 5),
                "kernel_launches_timed": prof_steps,
                "algorithmic_bytes_per_launch": algo_bytes}
    if counters and counters.get("tensor_pipe_pct_of_active") is not None:
        roofline["tensor_pipe_pct_of_active"] = counters["tensor_pipe_pct_of_active"]
    return {"d": d, "R": R, "G": G, "k": k, "ms": ms, "steps": steps,
            "keys_per_step": keys_per_step, "algo_bytes": algo_bytes, "roofline": roofline,
            "clocks": clk.summary(), "n_copies": n_copies, "cache_bytes": cache_bytes, "l2": l2,
            "ws": ws, "out": out, "err": err, "stream": stream,
            "row_lens_h": row_lens_h}


def measure_dcp(workload, dcp_world, interleave, seed, dev, steps, world):
    """Device-timed key-sharded decode steps: every rank's top k with logits
    on its own shard of the cache (the ranks one after the other on this GPU),
    then the merge of their candidates, all through the C ABI, in CUDA graphs.
    The shards together are the workload's cache (well above L2)."""
    import torch

    import synth
    import sparse_attention_indexer_block_gb300 as saib

    d = synth.make_decode(workload, seed=seed, device=dev)
    R, G, k = d.num_reqs, d.next_n, d.topk
    assert G == 1
    shards = synth.shard_decode(d, dcp_world, interleave, seed=seed)
    seq_h = d.seq_lens.cpu().numpy().astype(np.int64)
    keys_per_step = int(seq_h.sum())
    algo_bytes = keys_per_step * PAGE_KEY_BYTES
    ws = saib.decode_workspace(R, G, k, dev)
    cv = torch.empty((dcp_world, R, k), dtype=torch.float32, device=dev)
    ci = torch.empty((dcp_world, R, k), dtype=torch.int32, device=dev)
    out = torch.empty((R, k), dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(dev)

    def step():
        for r, (cache, bt) in enumerate(shards):
            saib.indexer_decode_topk_values(d.q, d.w, cache, bt, d.seq_lens, G, k, dcp_rank=r,
                                            dcp_world=dcp_world, dcp_interleave=interleave,
                                            out_idx=ci[r], out_val=cv[r], workspace=ws,
                                            dev_error=err, stream=stream)
        saib.indexer_dcp_merge(cv, ci, k, out_idx=out, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())} during warm-up (dcp)")
    with torch.cuda.stream(stream):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(steps):
                step()
    torch.cuda.synchronize()
    t_soak = time.time()
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        with torch.cuda.stream(stream):
            while time.time() - t_soak < 1.0:
                g.replay()
                stream.synchronize()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
    ms = max_over_ranks([e0.elapsed_time(e1)], world, dev)[0]
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())} in the timed region (dcp)")
    peak, peak_kind = measured_peak_gbs()
    gbs = algo_bytes * steps / (ms / 1e3) / 1e9
    return {"workload": WORKLOAD_DESCS["dcp_long"],
            "metric_value": whole_job_rate(keys_per_step, steps, world, ms), "unit": "keys/s",
            "ms_per_step": ms / steps, "steps": steps,
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "traffic": None,
                         "peak_source": peak_kind,
                         "kernel": "the whole step (every rank's prep, score/select, split-row "
                                   "selection and index map, then the merge), CUDA events "
                                   "around graph replays",
                         "algorithmic_bytes_per_step": algo_bytes},
            "clocks": clk.summary(), "gpu_launches": (4 * dcp_world + 1) * steps}


def measure_blocks(workload, seed, dev, steps, world):
    """Device-timed block-selection steps (the decode logits, then the block
    top-k), through the C ABI, in a CUDA graph; the index cache is well above
    L2."""
    import torch

    import synth
    import sparse_attention_indexer_block_gb300 as saib

    d = synth.make_decode(workload, seed=seed, device=dev)
    R, G, k = d.num_reqs, d.next_n, d.topk
    assert G == 1
    seq_h = d.seq_lens.cpu().numpy().astype(np.int64)
    keys_per_step = int(seq_h.sum())
    ld = int(d.block_table.shape[1]) * 64
    logits = torch.empty((R, ld), dtype=torch.float32, device=dev)
    ws = saib.decode_workspace(R, G, k, dev)
    B, K, NI, NL = 64, 32, 1, 4
    out = torch.empty((R, K + NI + NL), dtype=torch.int32, device=dev)
    cnt = torch.empty(R, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(dev)

    def step():
        saib.indexer_decode_logits(d.q, d.w, d.cache, d.block_table, d.seq_lens, 1, k,
                                   out_logits=logits, workspace=ws, dev_error=err, stream=stream)
        saib.indexer_block_topk(logits, d.seq_lens, B, K, NI, NL, out=out, cnt=cnt, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())} during warm-up (blocks)")
    with torch.cuda.stream(stream):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(steps):
                step()
    torch.cuda.synchronize()
    t_soak = time.time()
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        with torch.cuda.stream(stream):
            while time.time() - t_soak < 1.0:
                g.replay()
                stream.synchronize()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
    ms = max_over_ranks([e0.elapsed_time(e1)], world, dev)[0]
    peak, peak_kind = measured_peak_gbs()
    algo = keys_per_step * (PAGE_KEY_BYTES + 8)  # keys, logits written and read back
    gbs = algo * steps / (ms / 1e3) / 1e9
    return {"workload": WORKLOAD_DESCS["long_blocks"],
            "metric_value": whole_job_rate(keys_per_step, steps, world, ms), "unit": "keys/s",
            "ms_per_step": ms / steps, "steps": steps,
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "traffic": None, "peak_source": peak_kind,
                         "kernel": "the whole step (prep, score/select in logits mode, block "
                                   "top-k), CUDA events around graph replays",
                         "algorithmic_bytes_per_step": algo},
            "clocks": clk.summary(), "gpu_launches": 3 * steps}


def run_step_only(args, rank, world, local):
    """The block-selection or key-sharded long-context step alone (as in the
    default run's `configs`), one JSON line."""
    import torch

    import sparse_attention_indexer_block_gb300 as saib
    from sparse_attention_indexer_block_gb300 import build as libbuild

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    libbuild.build()
    saib.load()
    seed = rank_seed(args.seed, rank)
    if args.workload == "long_blocks":
        r = measure_blocks("long", seed, dev, args.steps, world)
    else:
        r = measure_dcp("long", 2, 1, seed, dev, args.steps, world)
    if rank == 0:
        print(json.dumps({"metric": METRIC, "value": r["metric_value"], "unit": "keys/s",
                          "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                          "ms_per_step": r["ms_per_step"], "higher_is_better": True,
                          "scaling": "weak", "vs_baseline": None,
                          "dtype": "fp8_e4m3 (fp32 accumulate)", "data": "synthetic",
                          "config": {"workload": r["workload"]}, "roofline": r["roofline"],
                          "clocks": r["clocks"], "gpu_launches": r["gpu_launches"]}),
              flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_ours(args, rank, world, local):
    import torch

    import sparse_attention_indexer_block_gb300 as saib
    from sparse_attention_indexer_block_gb300 import build as libbuild

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    libbuild.build()
    saib.load()

    seed = rank_seed(args.seed, rank)
    K = args.steps
    mx = args.workload.endswith("_mxfp4")
    base_wl = args.workload[:-len("_mxfp4")] if mx else args.workload
    res = measure_decode(base_wl, seed, dev, K, min(K, 400), world, local, mx=mx)
    d, R, G, k = res["d"], res["R"], res["G"], res["k"]
    ms, keys_per_step, algo_bytes = res["ms"], res["keys_per_step"], res["algo_bytes"]
    value = whole_job_rate(keys_per_step, K, world, ms)
    launches = 3 * K  # prep (with the row expansion), score/select, split-row selection
    out, ws, err, stream = res["out"], res["ws"], res["err"], res["stream"]

    # end to end: pinned host inputs in, indices out, every step
    host = {n: t.cpu().pin_memory() for n, t in
            [("q", d.q), ("w", d.w), ("cache", d.cache), ("bt", d.block_table),
             ("seq", d.seq_lens), ("dl", d.decode_lens)]}
    dbuf = {n: torch.empty_like(t, device=dev) for n, t in host.items()}
    out_h = torch.empty((R * G, k), dtype=torch.int32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * out_h.element_size()

    def e2e_step():
        for n in host:
            dbuf[n].copy_(host[n], non_blocking=True)
        if mx:
            saib.indexer_decode_topk_mxfp4(dbuf["q"], dbuf["w"], dbuf["cache"], dbuf["bt"],
                                           dbuf["seq"], k, out_idx=out, workspace=ws,
                                           dev_error=err, stream=stream)
        else:
            saib.indexer_decode_topk_from_lens(dbuf["q"], dbuf["w"], dbuf["cache"], dbuf["bt"],
                                               dbuf["seq"], dbuf["dl"], G, k, out_idx=out,
                                               workspace=ws, dev_error=err, stream=stream)
        out_h.copy_(out, non_blocking=True)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    n_e2e = max(3, min(K, 50))
    with torch.cuda.stream(stream):
        for _ in range(3):
            e2e_step()
    barrier()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        f0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        f1.record(stream)
    barrier()
    e2e_ms = max_over_ranks([f0.elapsed_time(f1) / n_e2e], world, dev)[0]
    e2e = {"value": whole_job_rate(keys_per_step, 1, world, e2e_ms), "unit": "keys/s",
           "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
           "ms_per_step": round(e2e_ms, 4), "steps": n_e2e}

    # the other decode configurations the throughput target names (long
    # context) or that share the kernel (MTP), measured the same way
    extra = {}
    if args.workload == WORKLOAD and not args.no_extra_configs:
        host = dbuf = None
        torch.cuda.empty_cache()
        for wl, steps in (("long", 100), ("mtp", 300)):
            r = measure_decode(wl, seed, dev, steps, min(steps, 100), world, local)
            extra[wl] = {"workload": WORKLOAD_DESCS[wl], "metric_value": whole_job_rate(
                r["keys_per_step"], steps, world, r["ms"]), "unit": "keys/s",
                "ms_per_step": r["ms"] / steps, "steps": steps, "roofline": r["roofline"],
                "clocks": r["clocks"], "gpu_launches": 3 * steps}
            del r
            torch.cuda.empty_cache()
        extra["dcp_long"] = measure_dcp("long", 2, 1, seed, dev, 50, world)
        torch.cuda.empty_cache()
        extra["long_blocks"] = measure_blocks("long", seed, dev, 50, world)
        torch.cuda.empty_cache()
        for wl, steps in (("decode", 400), ("long", 100)):
            r = measure_decode(wl, seed, dev, steps, min(steps, 100), world, local, mx=True)
            extra[wl + "_mxfp4"] = {
                "workload": WORKLOAD_DESCS[wl + "_mxfp4"], "metric_value": whole_job_rate(
                    r["keys_per_step"], steps, world, r["ms"]), "unit": "keys/s",
                "ms_per_step": r["ms"] / steps, "steps": steps, "roofline": r["roofline"],
                "clocks": r["clocks"], "gpu_launches": 3 * steps}
            del r
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not mx:
        cpu = cpu_baseline(d, res["row_lens_h"])

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "keys/s", "n_gpus": world, "steps": K,
                "warmup": args.warmup, "ms_per_step": ms / K, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "fp8_e4m3 (fp32 accumulate)",
                "data": "synthetic",
                "config": {"workload": WORKLOAD_DESCS.get(args.workload, args.workload),
                           "requests": R, "next_n": G, "topk": k,
                           "keys_per_step": keys_per_step,
                           "index_bytes_per_step": algo_bytes,
                           "l2": f"cold: {res['n_copies']} rotating index-cache copies "
                                 f"({res['n_copies'] * res['cache_bytes'] / 2**20:.0f} MiB > 3 x "
                                 f"L2 {res['l2'] / 2**20:.0f} MiB)",
                           "timing": "CUDA events around CUDA-graph replays of K steps",
                           "parallelism": f"replicas x{world}"},
                "roofline": res["roofline"], "cpu_baseline": cpu, "e2e": e2e,
                "clocks": res["clocks"], "gpu_launches": launches,
                "hbm_gbs_index_stream": round(algo_bytes * K / (ms / 1e3) / 1e9, 1)}
        if extra:
            line["configs"] = extra
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# the CPU oracle (baseline leg and reference arm)
# ---------------------------------------------------------------------------

def _oracle_inputs(d):
    import oracle
    import synth
    q8, _, wp = oracle.quantize_q(synth.bf16_bits(d.q), d.w.cpu().numpy())
    return (q8, wp, d.cache.cpu().numpy(), d.block_table.cpu().numpy())


def cpu_baseline(d, row_lens_h, target_s: float = 10.0):
    """The oracle as it stands on this host's cores: all rows of the workload,
    repeated while under ~target_s seconds."""
    import oracle
    q8, wp, cache, bt = _oracle_inputs(d)
    G = d.next_n
    rows = np.nonzero(row_lens_h > 0)[0]
    threads = oracle.num_threads()
    t0 = time.perf_counter()
    passes = 0
    while True:
        oracle.score_select_rows(q8, wp, cache, bt, rows, rows // G, row_lens_h[rows], d.topk,
                                 threads=threads)
        passes += 1
        if time.perf_counter() - t0 > target_s:
            break
    dt = time.perf_counter() - t0
    keys = int(row_lens_h[rows].sum()) * passes
    return {"value": keys / dt, "unit": "keys/s", "cores": threads, "kind": "oracle",
            "sample": f"whole workload ({len(rows)} token rows, {keys // passes} keys) x {passes} "
                      f"pass(es), {dt:.1f} s, {threads} threads"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    import synth
    oracle.build()
    d = synth.make_decode(args.workload, seed=args.seed, device="cpu")
    G, k = d.next_n, d.topk
    seq_h = d.seq_lens.numpy().astype(np.int64)
    dl_h = d.decode_lens.numpy().astype(np.int64)
    row_lens_h = np.concatenate([[L - dd + j + 1 if j < dd else 0 for j in range(G)]
                                 for L, dd in zip(seq_h, dl_h)])
    q8, wp, cache, bt = _oracle_inputs(d)
    threads = oracle.num_threads()
    rows_all = np.nonzero(row_lens_h > 0)[0]
    # calibrate: keys/s of the oracle on a prefix sample of every row
    cal_len = np.minimum(row_lens_h[rows_all], k + 256)
    t0 = time.perf_counter()
    oracle.score_select_rows(q8, wp, cache, bt, rows_all, rows_all // G, cal_len, k,
                             threads=threads)
    rate = cal_len.sum() / (time.perf_counter() - t0)
    budget_s = 150.0
    per_step_keys = max(64, int(rate * budget_s / (args.steps + args.warmup)))
    per_row = max(1, per_step_keys // len(rows_all))
    sample_lens = np.minimum(row_lens_h[rows_all], per_row)

    def step():
        oracle.score_select_rows(q8, wp, cache, bt, rows_all, rows_all // G, sample_lens, k,
                                 want_logits=True, threads=threads)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    keys = int(sample_lens.sum()) * args.steps
    value = keys / dt
    sample = (f"each step: up to the first {per_row} keys of each of the {len(rows_all)} token rows "
              f"({int(sample_lens.sum())} keys), scored and selected")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "keys/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD_DESCS.get(args.workload, args.workload),
                       "requests": d.num_reqs, "next_n": G,
                       "topk": k, "parallelism": "host threads"},
            "cpu_baseline": {"value": value, "unit": "keys/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "keys/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


COUNTER_METRICS = ("gpu__time_duration.sum", "dram__bytes_read.sum", "dram__bytes_write.sum",
                   "sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active")


def record_counters(report: str, workload: str):
    """Adds `workload`'s entry to profiles/score_select_counters.json from an
    ncu report of one score/select launch and the split-row selection launch
    after it on that workload (ncu -i ... --page raw --csv), keyed by the
    current kernel-code hash. DRAM bytes and times are the two launches' sums."""
    import csv
    import io
    raw = subprocess.run(["ncu", "-i", report, "--page", "raw", "--csv"], check=True,
                         capture_output=True, text=True).stdout
    rows = list(csv.reader(io.StringIO(raw)))
    hdr, units = rows[0], rows[1]
    unit = dict(zip(hdr, units))
    launches = {}
    for name in ("score_select_kernel", "row_select_kernel"):
        found = [r for r in rows[2:] if any(name in c for c in r)]
        if len(found) != 1:
            raise SystemExit(f"expected one {name} launch in {report}, found {len(found)}")
        launches[name] = dict(zip(hdr, found[0]))

    def num(vals, name, scale_to):
        v = float(vals[name].replace(",", ""))
        u = unit.get(name, "")
        mult = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1e3, "MB": 1e6,
                "GB": 1e9, "nsecond": 1e-9, "usecond": 1e-6, "msecond": 1e-3, "second": 1,
                "ns": 1e-9, "us": 1e-6, "ms": 1e-3, "%": 1, "": 1}[u]
        return v * mult / scale_to

    def total(name, scale_to):
        return sum(num(v, name, scale_to) for v in launches.values())
    score = launches["score_select_kernel"]
    entry = {"source_sha256_16": kernel_code_hash(ROOT),
             "kernel": next(c for c in score.values() if "score_select_kernel" in c),
             "dram_bytes_read": int(total("dram__bytes_read.sum", 1)),
             "dram_bytes_write": int(total("dram__bytes_write.sum", 1)),
             "gpu_time_us_cold_serialised": round(total("gpu__time_duration.sum", 1e-6), 2),
             "row_select_gpu_time_us_cold_serialised": round(
                 num(launches["row_select_kernel"], "gpu__time_duration.sum", 1e-6), 2)}
    entry["dram_bytes_per_launch"] = entry["dram_bytes_read"] + entry["dram_bytes_write"]
    tp = "sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active"
    entry["tensor_pipe_pct_of_active"] = round(num(score, tp, 1), 2) if tp in score else None
    path = os.path.join(ROOT, "profiles", "score_select_counters.json")
    try:
        with open(path) as f:
            data = json.load(f)
    except (OSError, ValueError):
        data = {}
    data[workload] = entry
    with open(path, "w") as f:
        json.dump(data, f, indent=1, sort_keys=True)
        f.write("\n")
    print(json.dumps({workload: entry}))


def main():
    args = parse()
    if args.record_counters:
        record_counters(args.record_counters, args.workload)
        return
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
    elif args.workload == "prefill":
        run_prefill(args, rank, world, local)
    elif args.workload == "insert":
        run_insert(args, rank, world, local)
    elif args.workload in ("long_blocks", "dcp_long"):
        run_step_only(args, rank, world, local)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
