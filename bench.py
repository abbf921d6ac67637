"""Benchmark of the decode-step paged-KV attention path (append -> split-K decode -> combine).

Default workload: the long-context GQA decode (28 layers, 16 query heads / 8 KV heads of 128,
batch 8 x 32 768 tokens, 16-slot pages, 1 % outlier keys), the largest single-GPU workload and
one of the two the 70 % HBM-roofline target is set on.  One step runs the whole path for every
layer; the step is captured once as a CUDA graph with programmatic dependent launch and replayed.
The same JSON line also carries the other workloads (mixed serving, ragged batch, single stream,
sliding window), each timed the same way under the same clock sampling (`extra_workloads`).

Prints one JSON line.  `--impl reference` times the fp64 CPU oracle on the host cores instead.
Multi-GPU runs (torchrun) are independent replicas: the path has no exchange step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from pkv_inputs import workloads as W  # noqa: E402

METRIC = "decode-attention KV GB/s & % of GB300 HBM roofline; attention µs/step/layer"
DEFAULT_CONFIG = 4
DEFAULT_EXTRA = "5,3,2,6"  # the other workloads, timed after the headline one
FALLBACK_HBM_GBS = 6800.0
# ncu summaries of the headline kernel (per workload id): per-launch DRAM bytes and the hash of the
# kernel sources they were taken from
PROFILE_SUMMARY = {
    2: os.path.join(ROOT, "profiles", "decode_kernel_phi3_b1_ctx4096.md"),
    4: os.path.join(ROOT, "profiles", "decode_kernel_gqa16x8_d128_b8_ctx32768.md"),
}
# the decode kernel's sources, in the order their bytes are hashed for the profile summary
DECODE_SOURCES = [os.path.join(ROOT, "paged_kv_decode_pkv_gb300", "csrc", f) for f in
                  ("decode_partial.cu", "merge.cuh", "ptx.cuh", "rope.cuh", "pkv_internal.h")]


def decode_sources_sha256() -> str:
    """sha256 of the decode kernel's code: its sources without blank and whole-line // comment
    lines (a comment edit does not change the kernel)."""
    h = hashlib.sha256()
    for f in DECODE_SOURCES:
        with open(f, "rb") as fh:
            for line in fh.read().splitlines():
                t = line.strip()
                if t and not t.startswith(b"//"):
                    h.update(line + b"\n")
    return h.hexdigest()


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG, choices=sorted(W.CONFIGS))
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="bound of the CPU-baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    # smaller variants of a workload, for profiler captures of the same kernels
    ap.add_argument("--layers", type=int, default=0, help="override the number of layers")
    ap.add_argument("--batch", type=int, default=0, help="override the batch size")
    ap.add_argument("--pool-pages", type=int, default=0, help="override the pool size in pages")
    ap.add_argument("--extra", default=DEFAULT_EXTRA,
                    help="comma-separated workload ids timed after the headline one ('' for none)")
    ap.add_argument("--int8", action="store_true",
                    help="int8 KV cache (PKV_OPT_INT8_KV): the history is appended through the library's "
                         "quantizing append; bytes are the int8 blocks read")
    return ap.parse_args()


def workload(args) -> W.Config:
    cfg = W.CONFIGS[args.config]
    changes = {}
    if args.layers:
        changes["layers"] = args.layers
    if args.batch:
        changes["batch"] = args.batch
        changes["chunk_seqs"] = min(cfg.chunk_seqs, args.batch)
    if args.pool_pages:
        changes["pool_pages"] = args.pool_pages
    return W.scaled(cfg, **changes) if changes else cfg


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def ncu_traffic(cid: int):
    """Per-launch DRAM bytes of the decode kernel on workload `cid` from the committed ncu summary,
    or None when there is none or the kernel source changed since the counters were taken."""
    if cid not in PROFILE_SUMMARY:
        return None
    try:
        text = open(PROFILE_SUMMARY[cid]).read()
        src = decode_sources_sha256()
        m_hash = re.search(r"kernel sources sha256:\s*([0-9a-f]{64})", text)
        m_val = re.search(r"dram bytes per launch:\s*([0-9]+)", text)
        if m_hash and m_val and m_hash.group(1) == src:
            return int(m_val.group(1))
    except OSError:
        pass
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"pkv_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return None
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v.lower() == "active"})
        loaded = [r for r in rows if r[2] > 0.25 * max(x[2] for x in rows)] or rows
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------------------------------------
# ranks: one per GPU, each on its own batch of the workload (weak scaling, no collective on the data path)


def rank_seed(cfg: W.Config, rank: int) -> int:
    """Seed of rank r's batch: rank 0 runs the standard workload, the others distinct batches of it."""
    return W.SEED_BASE + cfg.cid + 7919 * rank


def reduce_max(x: float, world: int, device=None) -> float:
    """Maximum of a per-rank value over all ranks (a no-op on one rank)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------------------------
# CPU oracle timing (test infrastructure: the oracle is never on the product path)


def oracle_sample(step: W.Step, seconds: float, max_layers: int):
    """Time the oracle (append + attention) layer by layer on the host cores until `seconds` of
    oracle work or `max_layers` layers; returns (GB/s, threads, description)."""
    import oracle

    from tests import harness as H

    # bound the sample to one sequence when a layer is larger than the long-context GQA layer
    # (1.07 GB, timed whole)
    seqs = list(range(step.batch))
    if step.kv_bytes() > 1.2e9:
        seqs = [int(np.argmax(step.seq_len))]
    sub = W.substep(step, seqs) if len(seqs) < step.batch else step
    done_bytes, done_time, layers = 0, 0.0, 0
    for layer in range(max_layers):
        pool = W.host_pool_pages(sub, layer, np.arange(sub.num_pages))
        q, k, v = W.new_qkv(step, layer, rows=W.token_rows(step, seqs))
        g = H.geometry(sub)
        t0 = time.perf_counter()
        q_out = oracle.append(g, q, k, v, sub.pos_map, sub.append_indptr, sub.page_indptr, sub.page_indices, pool)
        oracle.attention(g, pool, q_out[H.query_rows(sub)], sub.page_indptr, sub.page_indices, sub.last_page_len,
                         window=step.cfg.window, sinks=oracle_sinks(step, layer))
        done_time += time.perf_counter() - t0
        done_bytes += sub.kv_bytes()
        layers += 1
        if done_time >= seconds:
            break
    what = (f"{layers} layer(s) x {len(seqs)} of {step.batch} sequence(s) of {step.cfg.name}: fp64 append + "
            f"unsplit attention, {done_bytes / 1e9:.3f} GB of KV")
    return done_bytes / done_time / 1e9, oracle.threads(), what


def oracle_sinks(step: W.Step, layer: int):
    return W.sink_logits(step, layer).astype(np.float64) if step.cfg.sinks else None


def reference_sample(step: W.Step, budget_bytes: float = 2e9):
    """The bounded sample the oracle arm times per step: the whole step when its KV fits the
    budget, else one layer, else the longest sequence of one layer."""
    cfg = step.cfg
    if step.kv_bytes() * cfg.layers <= budget_bytes:
        return list(range(cfg.layers)), list(range(step.batch))
    if step.kv_bytes() <= budget_bytes:
        return [0], list(range(step.batch))
    return [0], [int(np.argmax(step.seq_len))]


def run_reference(args):
    """The oracle arm: fp64 CPU oracle on the host cores, same metric and unit."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle

    from tests import harness as H

    cfg = workload(args)
    step = W.make_step(cfg)
    layers, seqs = reference_sample(step)
    sub = W.substep(step, seqs) if len(seqs) < step.batch else step
    g = H.geometry(sub)
    rows = W.token_rows(step, seqs)
    inputs = [(W.host_pool_pages(sub, l, np.arange(sub.num_pages)), *W.new_qkv(step, l, rows=rows)) for l in layers]
    sinks = [oracle_sinks(step, l) for l in layers]
    times = []
    for i in range(args.warmup + args.steps):
        pools = [x[0].copy() for x in inputs]
        t0 = time.perf_counter()
        for pool, (_, q, k, v), sk in zip(pools, inputs, sinks):
            q_out = oracle.append(g, q, k, v, sub.pos_map, sub.append_indptr, sub.page_indptr, sub.page_indices,
                                  pool)
            oracle.attention(g, pool, q_out[H.query_rows(sub)], sub.page_indptr, sub.page_indices,
                             sub.last_page_len, window=cfg.window, sinks=sk)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    t = statistics.mean(times)
    sample_bytes = sub.kv_bytes() * len(layers)
    value = sample_bytes / t / 1e9
    sample = (f"each step: {len(layers)} of {cfg.layers} layer(s) x {len(seqs)} of {step.batch} sequence(s) of "
              f"{cfg.name} ({sample_bytes / 1e6:.1f} MB KV): fp64 append + unsplit attention")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg.name},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# ------------------------------------------------------------------------------------------------


def prefill_measure(cfg, step, cache, layers, tabs, q_out, stream, time_graph, dev):
    """Chunked-prefill attention of every appended token (pkv_prefill_attention), one launch per
    layer in a CUDA graph, on workloads whose sequences append several tokens.  Tensor-bound at
    long contexts: flops = 4 * Hq * head_dim * sum over tokens of the positions each attends to."""
    import torch

    if int(step.new_tokens.max()) <= 1:
        return None
    # the sequences that appended a chunk (the others are decode steps, served by the decode kernel)
    seqs = np.flatnonzero(step.new_tokens > 1)
    ai = np.concatenate([[0], np.cumsum(step.new_tokens[seqs])]).astype(np.int32)
    rows = np.concatenate([np.arange(step.append_indptr[s], step.append_indptr[s + 1]) for s in seqs])
    pi = np.concatenate([[0], np.cumsum(np.diff(step.page_indptr)[seqs])]).astype(np.int32)
    px = np.concatenate([step.page_indices[step.page_indptr[s]:step.page_indptr[s + 1]] for s in seqs])
    sub = {"append_indptr": ai, "pos_map": step.pos_map[rows], "page_indptr": pi, "page_indices": px,
           "last_page_len": step.last_page_len[seqs]}
    sub = {k: torch.from_numpy(np.ascontiguousarray(v, dtype=np.int32)).to(dev) for k, v in sub.items()}
    rows_d = torch.from_numpy(rows.astype(np.int64)).to(dev)
    qs = [q_out[l].index_select(0, rows_d) for l in layers]
    T = int(rows.size)
    outs = [torch.empty((T, cfg.hq, cfg.head_dim), dtype=torch.float16, device=dev) for _ in layers]
    lses = [torch.empty((T, cfg.hq), dtype=torch.float32, device=dev) for _ in layers]

    def run():
        for l in layers:
            cache.prefill_attention(l, qs[l], sub["append_indptr"], sub["pos_map"], sub["page_indptr"],
                                    sub["page_indices"], sub["last_page_len"], out=outs[l], lse=lses[l])

    with torch.cuda.stream(stream):
        run()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        run()
    torch.cuda.synchronize()
    ms = time_graph(g)
    seen = step.pos_map[rows].astype(np.int64) + 1
    if cfg.window:
        seen = np.minimum(seen, cfg.window)
    flops = 4.0 * cfg.hq * cfg.head_dim * float(seen.sum())
    tflops = flops * cfg.layers / (ms * 1e-3) / 1e12
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, kind = float(json.load(f)["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    except Exception:
        peak, kind = 1900.0, "fallback"
    return {"value": tflops, "unit": "TFLOP/s", "bound": "tensor", "peak": peak, "frac": tflops / peak,
            "peak_source": kind + "; fp16 mma runs at the bf16 rate", "us_per_layer": ms * 1e3 / cfg.layers,
            "flops_per_layer": flops, "tokens": T, "sequences": int(seqs.size),
            "step": "per layer: pkv_prefill_attention over the sequences that appended a chunk (every chunk "
                    "token, causal; tcgen05.mma with tensor-memory accumulators)"}


def qkv_measure(args, cfg, step, cache, layers, tabs, q_out, counters, po, pl, outs, lses, total_pages, stream,
                time_graph, dev):
    """The Q4F16_1 QKV projection fused with RoPE and the KV append (pkv_qkv_append_rope), one
    launch per layer in a CUDA graph, each layer with its own weights; and the same followed by
    the merged decode (the attention segment of the pages' decode loop).  Weight bytes per layer:
    packed nibbles, fp16 scales and the inputs; HBM-bound."""
    import torch

    import paged_kv_decode_pkv_gb300 as pkv

    hidden = W.qkv_hidden(cfg)
    if hidden > 4096 or hidden % 32 or step.num_tokens > 256:
        return None  # a large token count makes the projection a GEMM, which this kernel is not
    ws = []
    for l in layers:
        w, sc = W.qkv_weights(step, l)
        x = W.hidden_states(step, l)
        ws.append((torch.from_numpy(x).view(torch.float16).to(dev), torch.from_numpy(w.view(np.int32)).to(dev),
                   torch.from_numpy(sc).view(torch.float16).to(dev)))
    use_q_indptr = int(step.new_tokens.max()) > 1

    def proj_step():
        for l in layers:
            x, w, sc = ws[l]
            cache.qkv_append_rope(l, x, w, sc, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"],
                                  tabs["page_indices"], q_out=q_out[l])

    def proj_decode_step():
        for l in layers:
            x, w, sc = ws[l]
            cache.qkv_append_rope(l, x, w, sc, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"],
                                  tabs["page_indices"], q_out=q_out[l])
            cache.decode_attention_merged(l, q_out[l], tabs["page_indptr"], tabs["page_indices"],
                                          tabs["last_page_len"], step.max_pages_per_seq, counters,
                                          q_indptr=tabs["append_indptr"] if use_q_indptr else None,
                                          total_pages=total_pages, partial_o=po, partial_lse=pl, out=outs[l],
                                          lse=lses[l])

    with torch.cuda.stream(stream):
        proj_decode_step()
    torch.cuda.synchronize()
    code, flags = cache.check_status(stream)
    if code != 0:
        raise RuntimeError(f"device status after the projection: {pkv.status_string(code)} flags {flags:#x}")
    g1, g2 = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g1, stream=stream):
        proj_step()
    with torch.cuda.graph(g2, stream=stream):
        proj_decode_step()
    torch.cuda.synchronize()
    proj_ms = time_graph(g1)
    both_ms = time_graph(g2)
    n_rows = (cfg.hq + 2 * cfg.hkv) * cfg.head_dim
    wbytes = n_rows * hidden // 2 + n_rows * (hidden // 32) * 2 + step.num_tokens * hidden * 2
    peak, _ = measured_peaks()
    per_layer_us = proj_ms * 1e3 / cfg.layers
    gbs = wbytes * cfg.layers / (proj_ms * 1e-3) / 1e9
    # the projection alone (pkv_qkv_project) for several token counts over every layer's weights: one
    # token on CUDA cores, several on tensor cores (mma.sync)
    sweep = {}
    gen = torch.Generator(device=dev)
    gen.manual_seed(step.seed)
    for T in (1, 8, 16, 32):
        xs = [(torch.randn((T, hidden), generator=gen, device=dev) * 0.5).to(torch.float16) for _ in layers]
        ys = [torch.empty((T, n_rows), dtype=torch.float16, device=dev) for _ in layers]

        def proj_only():
            for l in layers:
                cache.qkv_project(xs[l], ws[l][1], ws[l][2], y=ys[l])

        with torch.cuda.stream(stream):
            proj_only()
        torch.cuda.synchronize()
        g3 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g3, stream=stream):
            proj_only()
        torch.cuda.synchronize()
        ms_t = time_graph(g3)
        tb = n_rows * hidden // 2 + n_rows * (hidden // 32) * 2 + T * hidden * 2
        sweep[str(T)] = {"us_per_layer": ms_t * 1e3 / cfg.layers,
                         "gbs": tb * cfg.layers / (ms_t * 1e-3) / 1e9,
                         "tflops": 2.0 * T * n_rows * hidden * cfg.layers / (ms_t * 1e-3) / 1e12}
    return {"value": gbs, "unit": "GB/s", "bytes_per_layer": wbytes, "us_per_layer": per_layer_us,
            "roofline_frac": gbs / peak, "hidden": hidden, "rows": n_rows,
            "step": "per layer: pkv_qkv_append_rope (Q4F16_1 projection + RoPE + append, one launch)",
            "with_decode_us_per_layer": both_ms * 1e3 / cfg.layers,
            "with_decode": "per layer: pkv_qkv_append_rope + pkv_decode_attention_merged",
            "project_tokens": sweep,
            "project_tokens_step": "per layer: pkv_qkv_project of T tokens (one token: CUDA cores; several: mma.sync)"}


def kv_bytes_layer(step: W.Step, int8: bool) -> int:
    """Algorithmic KV bytes one layer's decode reads: fp16 K and V, or (int8 cache) the int8 codes
    and the fp32 scale of every attended slot."""
    if not int8:
        return step.kv_bytes()
    cfg = step.cfg
    seen = np.minimum(step.seq_len, cfg.window) if cfg.window > 0 else step.seq_len
    return int(seen.sum()) * cfg.hkv * 2 * (cfg.head_dim + 4)


def int8_pools(step: W.Step, cfg, layers, dev):
    """int8 pools, one per entry of `layers` (workload layer ids), whose history (every position
    but the step's new tokens) went through the library's quantizing append: seeded raw k and v
    rows of that layer appended sequence by sequence."""
    import torch

    import paged_kv_decode_pkv_gb300 as pkv
    from pkv_inputs import dev_fill_range, key

    blk = 16 * cfg.head_dim + 64
    pools = [torch.zeros((step.num_pages, 2, cfg.hkv, blk), dtype=torch.uint8, device=dev) for _ in layers]
    builder = pkv.Cache(len(layers), step.num_pages, cfg.hq, cfg.hkv, cfg.head_dim, step.max_position, cfg.theta,
                        pools=pools, options=pkv.OPT_INT8_KV)
    pi = torch.from_numpy(step.page_indptr.astype(np.int32)).to(dev)
    px = torch.from_numpy(step.page_indices.astype(np.int32)).to(dev)
    cached = (step.seq_len - step.new_tokens).astype(np.int64)
    for slot, l in enumerate(layers):
        for s in range(step.batch):
            n = int(cached[s])
            if n <= 0:
                continue
            rows = n * cfg.hkv * cfg.head_dim
            k = torch.empty(rows, dtype=torch.float16, device=dev)
            v = torch.empty(rows, dtype=torch.float16, device=dev)
            seed = step.seed + 1000003 * (l + 1)
            dev_fill_range(k.data_ptr(), rows, key(seed, 2 * s), 0, cfg.value_scale)
            dev_fill_range(v.data_ptr(), rows, key(seed, 2 * s + 1), 0, cfg.value_scale)
            q = torch.zeros((n, cfg.hq, cfg.head_dim), dtype=torch.float16, device=dev)
            seq_pi = torch.tensor([0, int(step.page_indptr[s + 1] - step.page_indptr[s])], dtype=torch.int32,
                                  device=dev)
            seq_px = px[int(step.page_indptr[s]):int(step.page_indptr[s + 1])].contiguous()
            pos = torch.arange(n, dtype=torch.int32, device=dev)
            ai = torch.tensor([0, n], dtype=torch.int32, device=dev)
            builder.append_rope(slot, q, k.view(n, cfg.hkv, cfg.head_dim), v.view(n, cfg.hkv, cfg.head_dim), pos,
                                ai, seq_pi, seq_px)
    torch.cuda.synchronize()
    code, flags = builder.check_status()
    if code != 0:
        raise RuntimeError(f"int8 history append: status {code} flags {flags:#x}")
    del builder, pi
    return pools


def staged(arrays, dev):
    """One pinned host buffer and one device buffer holding `arrays` at 256-byte aligned offsets;
    returns (host, device, device views with each array's shape and dtype: fp16 for uint16 bits)."""
    import torch

    offs, pos = [], 0
    for a in arrays:
        pos = (pos + 255) & ~255
        offs.append(pos)
        pos += a.nbytes
    host = torch.empty(max(pos, 1), dtype=torch.uint8).pin_memory()
    hnp = host.numpy()
    for a, o in zip(arrays, offs):
        hnp[o:o + a.nbytes] = np.ascontiguousarray(a).view(np.uint8).reshape(-1)
    devbuf = host.to(dev)
    kinds = {np.dtype(np.int32): torch.int32, np.dtype(np.uint16): torch.float16, np.dtype(np.float32): torch.float32}
    views = [devbuf[o:o + a.nbytes].view(kinds[a.dtype]).view(a.shape) for a, o in zip(arrays, offs)]
    return host, devbuf, views


def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    cfg = workload(args)
    line = measure_headline(args, cfg, world, rank, local, dev)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()  # the headline workload's pools are released before the next ones
    extra = [] if args.int8 else [int(x) for x in args.extra.split(",") if x.strip()]
    if extra:
        line["extra_workloads"] = {}
        for cid in extra:
            res = measure_extra(args, W.CONFIGS[cid], world, rank, local, dev)
            line["extra_workloads"][res["workload"]] = res
            torch.cuda.synchronize()
            torch.cuda.empty_cache()
    if rank == 0 and not args.no_cpu_baseline:
        step = W.make_step(cfg, rank_seed(cfg, rank))
        gbs, threads, what = oracle_sample(step, args.cpu_seconds, cfg.layers)
        line["cpu_baseline"] = {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": what}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def measure_extra(args, cfg, world, rank, local, dev):
    """Another workload timed like the headline one: its whole step (every layer, the headline
    layer step per layer) captured as one CUDA graph with programmatic dependent launch and early
    page copies, replayed K times after W warm-up replays, with the clocks sampled meanwhile.
    Inputs resident in HBM; every step reads more KV than the L2 holds."""
    import torch

    import paged_kv_decode_pkv_gb300 as pkv

    step = W.make_step(cfg, rank_seed(cfg, rank))
    layers = list(range(cfg.layers))
    pools = [W.device_pool(step, l) for l in layers]
    windows = [cfg.window] * cfg.layers if cfg.window else None
    sinks = [torch.from_numpy(W.sink_logits(step, l)).to(dev) for l in layers] if cfg.sinks else None
    cache = pkv.Cache(cfg.layers, step.num_pages, cfg.hq, cfg.hkv, cfg.head_dim, step.max_position, cfg.theta,
                      pools=pools, options=pkv.OPT_PDL | pkv.OPT_EARLY_PAGES, windows=windows, sinks=sinks)
    B, T = step.batch, step.num_tokens
    total_pages = int(step.page_indptr[-1])
    S, chunk = cache.plan_decode(B, step.max_pages_per_seq, total_pages)
    tabs = {k: torch.from_numpy(np.ascontiguousarray(getattr(step, k), dtype=np.int32)).to(dev) for k in
            ("pos_map", "append_indptr", "page_indptr", "page_indices", "last_page_len")}
    qkv = []
    for l in layers:
        q, k, v = W.new_qkv(step, l)
        qkv.append(tuple(torch.from_numpy(x).view(torch.float16).to(dev) for x in (q, k, v)))
    q_out = [torch.empty((T, cfg.hq, cfg.head_dim), dtype=torch.float16, device=dev) for _ in layers]
    po = torch.empty((B, cfg.hq, S, cfg.head_dim), dtype=torch.float32, device=dev)
    pl = torch.empty((B, cfg.hq, S), dtype=torch.float32, device=dev)
    outs = [torch.empty((B, cfg.hq, cfg.head_dim), dtype=torch.float16, device=dev) for _ in layers]
    lses = [torch.empty((B, cfg.hq), dtype=torch.float32, device=dev) for _ in layers]
    counters = torch.zeros(B * cfg.hkv, dtype=torch.int32, device=dev)

    def step_fn():
        for l in layers:
            q, k, v = qkv[l]
            cache.append_decode_attention(l, q, k, v, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"],
                                          tabs["page_indices"], tabs["last_page_len"], step.max_pages_per_seq,
                                          counters, total_pages=total_pages, q_out=q_out[l], partial_o=po,
                                          partial_lse=pl, out=outs[l], lse=lses[l])

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        step_fn()
    torch.cuda.synchronize()
    code, flags = cache.check_status(stream)
    if code != 0:
        raise RuntimeError(f"{cfg.name}: device status {pkv.status_string(code)} flags {flags:#x}")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step_fn()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def time_graph(g):
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                g.replay()
            ev0.record()
            for _ in range(args.steps):
                g.replay()
            ev1.record()
        torch.cuda.synchronize()
        return reduce_max(ev0.elapsed_time(ev1) / args.steps, world, dev)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        step_ms = time_graph(graph)
    code, flags = cache.check_status(stream)
    if code != 0:
        raise RuntimeError(f"{cfg.name}: device status after the timed region {pkv.status_string(code)} "
                           f"flags {flags:#x}")
    peak, _ = measured_peaks()
    kv_step = step.kv_bytes() * cfg.layers
    value = world * kv_step / (step_ms * 1e-3) / 1e9
    one_launch = T == B
    res = {"workload": cfg.name, "value": value, "unit": "GB/s", "frac": value / world / peak,
           "ms_per_step": step_ms, "us_per_layer": step_ms * 1e3 / cfg.layers, "layers": cfg.layers, "batch": B,
           "kv_bytes_per_step": kv_step, "splits": S,
           "step": "per layer: pkv_append_decode_attention (" +
                   ("1 launch)" if one_launch else "2 launches for chunked appends: append, merged decode)"),
           **({"window": cfg.window} if cfg.window else {}),
           "clocks": clocks.summary()}
    pf = prefill_measure(cfg, step, cache, layers, tabs, q_out, stream, time_graph, dev)
    if pf is not None:
        res["prefill"] = pf
    return res


def measure_headline(args, cfg, world, rank, local, dev):
    """The headline workload: the JSON line's value, roofline, e2e, launch layouts, and the fused
    QKV projection and chunked prefill where the workload has them."""
    import torch
    import torch.distributed as dist

    import paged_kv_decode_pkv_gb300 as pkv

    step = W.make_step(cfg, rank_seed(cfg, rank))
    layers = list(range(cfg.layers))
    pools = int8_pools(step, cfg, layers, dev) if args.int8 else [W.device_pool(step, l) for l in layers]
    # layer variants of the workload: sliding window and attention sinks
    windows = [cfg.window] * cfg.layers if cfg.window else None
    sinks = [torch.from_numpy(W.sink_logits(step, l)).to(dev) for l in layers] if cfg.sinks else None
    cache = pkv.Cache(cfg.layers, step.num_pages, cfg.hq, cfg.hkv, cfg.head_dim, step.max_position, cfg.theta,
                      pools=pools, options=pkv.OPT_PDL | pkv.OPT_EARLY_PAGES | (pkv.OPT_INT8_KV if args.int8 else 0),
                      windows=windows, sinks=sinks)
    B, T = step.batch, step.num_tokens
    total_pages = int(step.page_indptr[-1])
    S, chunk = cache.plan_decode(B, step.max_pages_per_seq, total_pages)

    # The step's inputs (page tables and every layer's new q, k, v) live in one pinned host buffer and
    # one device buffer of the same layout, so the end-to-end step moves them with one copy; the
    # outputs (every layer's out and lse) likewise come back with one copy.
    in_arrays = [np.ascontiguousarray(getattr(step, k), dtype=np.int32) for k in
                 ("pos_map", "append_indptr", "page_indptr", "page_indices", "last_page_len")]
    for l in layers:
        in_arrays += [np.ascontiguousarray(x) for x in W.new_qkv(step, l)]
    in_host, in_dev, in_views = staged(in_arrays, dev)
    tabs = dict(zip(("pos_map", "append_indptr", "page_indptr", "page_indices", "last_page_len"), in_views[:5]))
    qkv = [tuple(in_views[5 + 3 * l + i] for i in range(3)) for l in layers]
    use_q_indptr = int(step.new_tokens.max()) > 1
    q_out = [torch.empty((T, cfg.hq, cfg.head_dim), dtype=torch.float16, device=dev) for _ in layers]
    po = torch.empty((B, cfg.hq, S, cfg.head_dim), dtype=torch.float32, device=dev)
    pl = torch.empty((B, cfg.hq, S), dtype=torch.float32, device=dev)
    out_arrays = []
    for _ in layers:
        out_arrays += [np.zeros((B, cfg.hq, cfg.head_dim), dtype=np.uint16), np.zeros((B, cfg.hq), dtype=np.float32)]
    out_host, out_dev, out_views = staged(out_arrays, dev)
    outs = [out_views[2 * l] for l in layers]
    lses = [out_views[2 * l + 1] for l in layers]

    counters = torch.zeros(B * cfg.hkv, dtype=torch.int32, device=dev)

    # one new token per sequence: pkv_append_decode_attention is a single launch (two on an int8 cache)
    one_launch = T == B and not args.int8

    def layer_chain_fused(l):
        """append, split-K decode and combine in one launch (two for chunked appends)"""
        q, k, v = qkv[l]
        cache.append_decode_attention(l, q, k, v, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"],
                                      tabs["page_indices"], tabs["last_page_len"], step.max_pages_per_seq,
                                      counters, total_pages=total_pages, q_out=q_out[l], partial_o=po,
                                      partial_lse=pl, out=outs[l], lse=lses[l])

    def layer_chain(l):
        """append -> split-K decode with the combine merged into the same launch (two launches)"""
        q, k, v = qkv[l]
        cache.append_rope(l, q, k, v, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"],
                          tabs["page_indices"], q_out=q_out[l])
        cache.decode_attention_merged(l, q_out[l], tabs["page_indptr"], tabs["page_indices"], tabs["last_page_len"],
                                      step.max_pages_per_seq, counters,
                                      q_indptr=tabs["append_indptr"] if use_q_indptr else None,
                                      total_pages=total_pages, partial_o=po, partial_lse=pl, out=outs[l],
                                      lse=lses[l])

    def layer_chain_separate(l):
        """append -> split-K decode -> combine, three launches"""
        q, k, v = qkv[l]
        cache.append_rope(l, q, k, v, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"],
                          tabs["page_indices"], q_out=q_out[l])
        cache.decode_attention(l, q_out[l], tabs["page_indptr"], tabs["page_indices"], tabs["last_page_len"],
                               step.max_pages_per_seq, q_indptr=tabs["append_indptr"] if use_q_indptr else None,
                               total_pages=total_pages, partial_o=po, partial_lse=pl)
        cache.combine(po, pl, out=outs[l], lse=lses[l], sinks=None if sinks is None else sinks[l])

    def step_fn():
        for l in layers:
            layer_chain(l)

    def step_fn_separate():
        for l in layers:
            layer_chain_separate(l)

    def step_fn_fused():
        for l in layers:
            layer_chain_fused(l)

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        step_fn()
        step_fn_fused()
    torch.cuda.synchronize()
    code, flags = cache.check_status(stream)
    if code != 0:
        raise RuntimeError(f"device status {pkv.status_string(code)} flags {flags:#x}")
    # The two- and three-launch layouts write the pools through the append kernel, after which the
    # next one-launch step of each layer runs without early page copies; they are captured first,
    # and one eager one-launch step runs before the headline graph is captured.
    graph_two = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_two, stream=stream):
        step_fn()
    graph_sep = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_sep, stream=stream):
        step_fn_separate()
    with torch.cuda.stream(stream):
        step_fn_fused()
    graph = torch.cuda.CUDAGraph()  # the headline step: pkv_append_decode_attention per layer
    with torch.cuda.graph(graph, stream=stream):
        step_fn_fused()
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            dist.barrier()

    def max_over_ranks(x):
        return reduce_max(x, world, dev)

    # ---- timed region: K graph replays ----------------------------------------------------------
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    torch.cuda.synchronize()
    barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            ev0.record()
            for _ in range(args.steps):
                graph.replay()
            ev1.record()
        torch.cuda.synchronize()
    barrier()
    step_ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps)
    # the same step as two launches per layer (append; decode with the merge) and as three
    # (append, decode, combine), for reference
    def time_graph(g):
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                g.replay()
            ev0.record()
            for _ in range(args.steps):
                g.replay()
            ev1.record()
        torch.cuda.synchronize()
        return max_over_ranks(ev0.elapsed_time(ev1) / args.steps)

    step_sep_ms = time_graph(graph_sep)
    step_two_ms = time_graph(graph_two)
    code, flags = cache.check_status(stream)
    if code != 0:
        raise RuntimeError(f"device status after the timed region: {pkv.status_string(code)} flags {flags:#x}")
    kv_step = kv_bytes_layer(step, args.int8) * cfg.layers
    value = world * kv_step / (step_ms * 1e-3) / 1e9

    # ---- per-kernel durations: events around each layer's decode launch on the launching stream ----
    # A second handle over the same pools launches without programmatic dependent launch, so each
    # kernel runs alone between its events; a GPU sleep in front of every step keeps the launches
    # queued so that the events time the device, not the host's launch rate.  The kernel is the
    # headline step's: the one-launch decode (append, split-K decode and merge); with chunked
    # appends, the merged decode after the append launch.
    plain = pkv.Cache(cfg.layers, step.num_pages, cfg.hq, cfg.hkv, cfg.head_dim, step.max_position, cfg.theta,
                      pools=pools, options=pkv.OPT_INT8_KV if args.int8 else 0, windows=windows, sinks=sinks)

    def layer_chain_plain(l, events):
        q, k, v = qkv[l]
        if one_launch:
            events[0].record()
            plain.append_decode_attention(l, q, k, v, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"],
                                          tabs["page_indices"], tabs["last_page_len"], step.max_pages_per_seq,
                                          counters, total_pages=total_pages, q_out=q_out[l], partial_o=po,
                                          partial_lse=pl, out=outs[l], lse=lses[l])
            events[1].record()
            return
        plain.append_rope(l, q, k, v, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"],
                          tabs["page_indices"], q_out=q_out[l])
        events[0].record()
        plain.decode_attention_merged(l, q_out[l], tabs["page_indptr"], tabs["page_indices"], tabs["last_page_len"],
                                      step.max_pages_per_seq, counters,
                                      q_indptr=tabs["append_indptr"] if use_q_indptr else None,
                                      total_pages=total_pages, partial_o=po, partial_lse=pl, out=outs[l],
                                      lse=lses[l])
        events[1].record()

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps * cfg.layers)]
    sleep_cycles = int(2e9 * max(0.02, 0.002 * cfg.layers))
    with torch.cuda.stream(stream):
        i = 0
        for _ in range(args.steps):
            torch.cuda._sleep(sleep_cycles)
            for l in layers:
                layer_chain_plain(l, ev[i])
                i += 1
    torch.cuda.synchronize()
    dec_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    kv_layer = kv_bytes_layer(step, args.int8)
    # With one launch per layer the timed region is nothing but this kernel, launched back to back
    # (programmatic dependent launch overlaps each prologue with the previous launch), so its
    # average launch duration there is the step time over the launches.  With chunked appends the
    # step also runs the append kernel, and the isolated launches give the decode kernel's time.
    launch_ms = step_ms / cfg.layers if one_launch else dec_ms
    achieved = kv_layer / (launch_ms * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()
    overridden = bool(args.batch or args.pool_pages or args.int8)
    traffic = None if overridden else ncu_traffic(cfg.cid)

    # ---- end to end through the API with host buffers ------------------------------------------
    h2d = sum(a.nbytes for a in in_arrays)
    d2h = sum(a.nbytes for a in out_arrays)

    def e2e_step():
        in_dev.copy_(in_host, non_blocking=True)     # page tables and every layer's q, k, v
        for l in layers:
            layer_chain_fused(l)
        out_host.copy_(out_dev, non_blocking=True)   # every layer's out and lse

    e2e_graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        e2e_step()
    torch.cuda.synchronize()
    with torch.cuda.graph(e2e_graph, stream=stream):
        e2e_step()
    torch.cuda.synchronize()

    def timed_e2e(fn):
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                fn()
                stream.synchronize()
        barrier()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for _ in range(args.steps):
                fn()
                stream.synchronize()  # the step's result is on the host
        barrier()
        return max_over_ranks((time.perf_counter() - t0) / args.steps)

    # ---- the pages' fused QKV dispatch: Q4F16_1 projection + RoPE + append, then the decode -----
    prefill = None if args.int8 else prefill_measure(cfg, step, cache, layers, tabs, q_out, stream, time_graph, dev)
    qkv_proj = None if args.int8 else qkv_measure(args, cfg, step, cache, layers, tabs, q_out, counters, po, pl, outs, lses, total_pages,
                           stream, time_graph, dev)

    e2e_s = timed_e2e(e2e_graph.replay)
    e2e_eager_s = timed_e2e(e2e_step)
    code, flags = cache.check_status(stream)
    if code != 0:
        raise RuntimeError(f"device status after the e2e region: {pkv.status_string(code)} flags {flags:#x}")

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8 KV codes, f16 queries, f32 accumulate" if args.int8 else "f16 data, f32 accumulate", "data": "synthetic",
        "config": {"workload": cfg.name, "layers": cfg.layers, "batch": B, "q_heads": cfg.hq,
                   "kv_heads": cfg.hkv, "head_dim": cfg.head_dim, "page_size": 16,
                   "context_tokens": int(step.seq_len.sum()), "kv_bytes_per_step": kv_step,
                   "splits": S, "chunk_pages": chunk,
                   **({"window": cfg.window} if cfg.window else {}),
                   **({"kv_cache": "int8 blocks (codes + fp32 scale per slot); bytes are those read",
                       "fp16_equivalent_kv_bytes_per_step": step.kv_bytes() * cfg.layers} if args.int8 else {}),
                   **({"attention_sinks": "per layer and query head"} if cfg.sinks else {}),
                   "l2": f"inputs larger than L2: {kv_step / 1e9:.2f} GB of KV per step",
                   "launch": "CUDA graph of the step, programmatic dependent launch, early page copies",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "hbm_roofline_frac_step": value / world / peak,
        "attention_us_per_step_per_layer": launch_ms * 1e3,
        "step_us_per_layer": step_ms * 1e3 / cfg.layers,
        "step": "per layer: pkv_append_decode_attention (" +
                ("1 launch: append, split-K decode and merge)" if one_launch else
                 "2 launches on an int8 cache: the quantizing append, then split-K decode with the merge)"
                 if args.int8 else
                 "2 launches for chunked appends: append, then split-K decode with the merge)"),
        "two_kernels": {"value": world * kv_step / (step_two_ms * 1e-3) / 1e9, "ms_per_step": step_two_ms,
                        "step": "per layer: pkv_append_rope + pkv_decode_attention_merged"},
        "separate_kernels": {"value": world * kv_step / (step_sep_ms * 1e-3) / 1e9, "ms_per_step": step_sep_ms,
                             "step": "per layer: pkv_append_rope + pkv_decode_attention + pkv_combine"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "decode_kernel, one-launch step (append, split-K decode, merge)" if one_launch
                     else "decode_kernel (merged combine)",
                     "algorithmic_bytes_per_launch": kv_layer, "avg_launch_us": launch_ms * 1e3,
                     "launch_timing": "timed region (step time / launches)" if one_launch else
                     "isolated launches (events around each, no programmatic dependent launch)",
                     "isolated_launch_us": dec_ms * 1e3,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, burst copy)"},
        "e2e": {"value": world * kv_step / e2e_s / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3,
                "mode": "CUDA graph of one host-to-device copy of the step's inputs, the API calls and one "
                        "device-to-host copy of every layer's out and lse",
                "eager_value": world * kv_step / e2e_eager_s / 1e9, "eager_ms_per_step": e2e_eager_s * 1e3},
        "gpu_launches": args.steps * cfg.layers * (1 if one_launch else 2),
        "qkv_projection": qkv_proj,
        **({"prefill": prefill} if prefill is not None else {}),
        "clocks": clocks.summary(),
    }
    return line


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
