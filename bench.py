#!/usr/bin/env python3
"""Benchmark of the DSA sparse-MLA prefill hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-modes]

Headline workload: DeepSeek-V3.2 shard, per-token sparse prefill of one
16384-token causal chunk over 16384 latent rows, H = 32, D_QK = 576, D_V = 512,
top-2048 locality indices (synthetic, seeded).  One step = one call of the
per-token kernel over the whole chunk; the L2 is flushed (256 MiB write)
between timed steps and only the kernel is inside the CUDA events.

Prints ONE JSON line (rank 0).  ``value`` is whole-job query-tokens/s.  The
``modes`` object times the other forms on their own workloads (grouped:
union build + grouped kernel; NoPE layout per-token and grouped; masked MHA:
key mask + masked kernel).  ``--impl reference`` times the fp64 CPU oracle
(the only reference this method has here) on a bounded sample instead.
Under torchrun every rank runs its own chunk (weak scaling, no collective on
the data path); time is the max over ranks.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse prefill query-tokens/s & useful TFLOP/s per GB300; % of HBM / bf16 peak"
HEADLINE = "v32_h32_16k"
FLUSH_BYTES = 256 << 20


# ----------------------------------------------------------------------------
# environment
# ----------------------------------------------------------------------------
_T0 = time.time()


def log(msg):
    """Progress to stderr (the JSON line is the only stdout output)."""
    print(f"[bench {time.time() - _T0:7.1f}s] {msg}", file=sys.stderr, flush=True)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "dsa_sparse_mla_prefill_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_key, src_hash, launch_units):
    """DRAM bytes per launch from a committed ncu summary, scaled to this
    launch by units processed; None if absent or the kernel changed since."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel_key)
    if not d or d.get("source_hash") != src_hash:
        return None
    return d["dram_bytes_per_unit"] * launch_units


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        for ts, line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), parts[4:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        t0, t1 = (self.marks[0], self.marks[-1]) if len(self.marks) >= 2 else (rows[0][0], rows[-1][0])
        inwin = [r for r in rows if t0 <= r[0] <= t1] or rows
        names = ["active_mask", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in inwin:
            for n, v in zip(names[1:], r[3][1:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[1] for r in inwin), "sm_max_mhz": max(r[2] for r in inwin),
                "reasons": sorted(reasons), "samples": len(inwin)}


# ----------------------------------------------------------------------------
# multi-GPU: independent replicas (weak scaling), max-over-ranks timing
# ----------------------------------------------------------------------------
def rank_workload(w, rank):
    """Every rank processes its own chunk of the same shape (its own seed):
    the per-token path has no exchange step, so ranks share nothing."""
    from dataclasses import replace
    return w if rank == 0 else replace(w, seed=w.seed + 1000 * rank)


def max_over_ranks(x, dist=None, device=None):
    """Max of a per-rank float over all ranks (identity without a process group)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, world, ms_max):
    """Whole-job units/s: every rank's units over the slowest rank's time."""
    return world * units_per_rank / (ms_max / 1e3)


# ----------------------------------------------------------------------------
# workloads and algorithmic work
# ----------------------------------------------------------------------------
def sparse_work(w, idx, row_bytes=None):
    """Valid (token, key) pairs and algorithmic bytes / useful FLOPs of the per-token form
    (row_bytes: bytes gathered per selected row, the bf16 row unless given)."""
    pairs = int((idx[:, :w.k] >= 0).sum())
    row = w.d_qk * 2 if row_bytes is None else row_bytes
    bytes_ = pairs * row + w.T * w.H * w.d_qk * 2 + w.T * w.H * w.d_v * 2 + w.T * w.ld * 4 + w.T * w.H * 4
    flops = 2.0 * w.H * pairs * (w.d_qk + w.d_v)
    return pairs, bytes_, flops


def to_dev(x, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(dev)


def timed_steps(fn, steps, warmup, stream, flush=None):
    """Runs fn() warmup + steps times; per-step CUDA events around fn only;
    flush (untimed) before each step.  Returns list of ms."""
    import torch
    for _ in range(warmup):
        if flush is not None:
            flush()
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        if flush is not None:
            flush()
        ev[i][0].record(stream)
        fn()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


# ----------------------------------------------------------------------------
# CPU baseline: the oracle as it stands, on a bounded sample, spawn pool
# ----------------------------------------------------------------------------
def _oracle_worker(args):
    """Runs the oracle over this worker's tokens, 16 per call, until its time
    budget is spent.  Returns (tokens done, seconds)."""
    q, kv, idx, k, scale, d_qk, d_v, budget = args
    from oracle.dsa_oracle import sparse_prefill
    t0 = time.perf_counter()
    done = 0
    for s in range(0, q.shape[0], 16):
        sparse_prefill(q[s:s + 16], kv, idx[s:s + 16], k, scale, d_qk, d_v)
        done += min(16, q.shape[0] - s)
        if time.perf_counter() - t0 > budget:
            break
    return done, time.perf_counter() - t0


def cpu_baseline(w, x, budget_s=12.0, pool=None, cores=None):
    """Times oracle.sparse_prefill, as it stands, on the host cores: each of
    ``cores`` spawn workers (one BLAS thread each) takes a disjoint random
    sample of the workload's tokens and works through it until ``budget_s``
    seconds have passed.  Throughput = tokens done / slowest worker's time."""
    cores = cores or os.cpu_count() or 1
    rng = np.random.default_rng(7)
    toks = rng.permutation(w.T)
    chunks = [np.sort(c) for c in np.array_split(toks, cores) if len(c)]
    tasks = [(x.q[c], x.kv, x.idx[c], w.k, w.scale, w.d_qk, w.d_v, budget_s) for c in chunks]
    own = pool is None
    if own:
        pool = oracle_pool(cores)
    res = pool.map(_oracle_worker, tasks)
    if own:
        pool.close()
        pool.join()
    n = sum(r[0] for r in res)
    wall = max(r[1] for r in res)
    return {"value": n / wall, "unit": "query-tokens/s", "cores": len(tasks), "kind": "oracle",
            "sample": f"{n} of {w.T} tokens of {w.name} (random, seeded), fp64 numpy oracle in batches of 16, "
                      f"{len(tasks)} spawn workers x 1 BLAS thread, {wall:.1f} s",
            "seconds": wall}


def _noop(_):
    return 0


def _single_thread_blas():
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"


def oracle_pool(cores):
    """Spawn pool whose workers start with one BLAS thread each (the variables
    are set while the children are created, before they import numpy)."""
    saved = {v: os.environ.get(v) for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")}
    _single_thread_blas()
    try:
        pool = mp.get_context("spawn").Pool(cores)
        pool.map(_noop, range(cores))
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    return pool


# ----------------------------------------------------------------------------
# modes: the other forms on their own workloads
# ----------------------------------------------------------------------------
def run_modes(dev, stream, peaks, steps, warmup, flush, only=None):
    """Times the other forms on their own workloads (``only``: a subset of the names)."""
    import torch
    import dsa_sparse_mla_prefill_gb300 as dsa
    from synth import WORKLOADS, make_masked_inputs, make_sparse_inputs
    out = {}
    steps = max(3, min(steps, 10))

    def sparse_block(name, grouped=True, per_token=True, w=None):
        w = WORKLOADS[name] if w is None else w
        log(f"mode {name}")
        x = make_sparse_inputs(w)
        q, kv = to_dev(x.q, dev), to_dev(x.kv, dev)
        idx = torch.from_numpy(x.idx).to(dev)
        pairs, abytes, flops = sparse_work(w, x.idx)
        res = {"T": w.T, "N": w.N, "H": w.H, "d_qk": w.d_qk, "k": w.k, "ld": w.ld}
        if per_token:
            o = torch.empty((w.T, w.H, 512), dtype=torch.bfloat16, device=dev)
            l = torch.empty((w.T, w.H), dtype=torch.float32, device=dev)
            ms = statistics.median(timed_steps(lambda: dsa.dsa_sparse_prefill(q, kv, idx, w.k, w.scale, out=o,
                                                                               lse=l), steps, warmup, stream, flush))
            res["per_token"] = {"ms": ms, "query_tokens_per_s": w.T / ms * 1e3,
                                "useful_tflops": flops / ms / 1e9, "logical_gbs": abytes / ms / 1e6,
                                "hbm_frac_logical": abytes / ms / 1e6 / peaks["hbm_gbs"]}
            # DRAM bytes from a committed ncu capture of this workload (scaled
            # by tokens; none if the kernel changed since)
            if w.H == 32 and w.d_qk == 576:
                traffic = profiled_traffic("sparse_prefill_" + w.name, kernel_source_hash(
                    ["sparse_prefill.cu", "dsa_device.cuh"]), w.T)
                if traffic:
                    res["per_token"].update(dram_bytes=traffic, dram_gbs=traffic / ms / 1e6,
                                            dram_frac=traffic / ms / 1e6 / peaks["hbm_gbs"])
        if grouped:
            G = w.G
            upad = dsa.dsa_union_pad(G, w.k, 128)
            ng = dsa.dsa_num_groups(x.cu_seqlens_q, w.T, G)
            u = torch.empty((ng, upad), dtype=torch.int32, device=dev)
            ul = torch.empty((ng,), dtype=torch.int32, device=dev)
            m = torch.empty((ng, upad), dtype=torch.uint8, device=dev)
            ub = lambda: dsa.dsa_union_build(idx, w.k, G, w.N, cu_seqlens_q=x.cu_seqlens_q, union_pad=upad,
                                             out=(u, ul, m))
            ms_u = statistics.median(timed_steps(ub, steps, warmup, stream, flush))
            ub_bytes = w.T * w.ld * 4 + ng * upad * 5 + ng * 4
            res["union_build"] = {"ms": ms_u, "ms_per_16k_tokens": ms_u * 16384 / w.T,
                                  "gbs": ub_bytes / ms_u / 1e6, "hbm_frac": ub_bytes / ms_u / 1e6 / peaks["hbm_gbs"]}
            ulen = ul.cpu().numpy().astype(np.int64)
            res["union_mean"] = float(ulen.mean())
            o = torch.empty((w.T, w.H, 512), dtype=torch.bfloat16, device=dev)
            l = torch.empty((w.T, w.H), dtype=torch.float32, device=dev)
            try:
                gfn = lambda: dsa.dsa_grouped_prefill(q, kv, u, ul, m, G, w.scale, cu_seqlens_q=x.cu_seqlens_q,
                                                      out=o, lse=l)
                gfn()
                ms_g = statistics.median(timed_steps(gfn, steps, warmup, stream, flush))
                uflops = 2.0 * 128 * float(ulen.sum()) * (w.d_qk + w.d_v)
                res["grouped"] = {"ms": ms_g, "with_union_build_ms": ms_g + ms_u,
                                  "query_tokens_per_s": w.T / ms_g * 1e3,
                                  "union_plus_useful_tflops": uflops / ms_g / 1e9,
                                  "useful_tflops": flops / ms_g / 1e9,
                                  "tensor_frac": uflops / ms_g / 1e9 / peaks["bf16_tflops"],
                                  "gathered_gb": float(ulen.sum()) * w.d_qk * 2 / 1e9}
            except dsa.DSAError as e:
                res["grouped"] = {"unavailable": str(e)}
        return res

    def want(name):
        return only is None or name in only

    for name in ("grouped_21k_of_32k", "nope_2x8192"):
        if want(name):
            out[name] = sparse_block(name)
            torch.cuda.empty_cache()
    # the headline shard at the tail of a 131072-row context: the 151 MB
    # latent table does not fit in the L2 (per-token form only)
    if want("v32_h32_16k_of_128k"):
        out["v32_h32_16k_of_128k"] = sparse_block("v32_h32_16k_of_128k", grouped=False)
        torch.cuda.empty_cache()
    # the headline workload in grouped form (H = 32: G = 4 tokens per group)
    if want("v32_h32_16k_grouped"):
        out["v32_h32_16k_grouped"] = sparse_block("v32_h32_16k", per_token=False)
        torch.cuda.empty_cache()
    # wide-union stress variant of the grouped workload: every token draws its
    # replacements independently, so the 8-token unions grow
    if want("grouped_21k_of_32k_wide"):
        wide = dataclasses.replace(WORKLOADS["grouped_21k_of_32k"], name="grouped_21k_of_32k_wide",
                                   index_gen="locality_wide")
        out["grouped_21k_of_32k_wide"] = sparse_block("grouped_21k_of_32k_wide", w=wide)
        torch.cuda.empty_cache()
    # the headline workload over an FP8 KV cache: the cache is written once
    # (quantize); a step is either the per-token kernel reading the FP8 rows
    # directly, or a dequantize to bf16 followed by the bf16 per-token kernel
    if want("v32_h32_16k_fp8kv"):
        w = WORKLOADS["v32_h32_16k"]
        log("mode v32_h32_16k_fp8kv")
        x = make_sparse_inputs(w)
        q, kv = to_dev(x.q, dev), to_dev(x.kv, dev)
        idx = torch.from_numpy(x.idx).to(dev)
        fp8 = torch.empty((w.N, dsa.dsa_kv_fp8_row_bytes(64)), dtype=torch.uint8, device=dev)
        deq = torch.empty((w.N, w.d_qk), dtype=torch.bfloat16, device=dev)
        o = torch.empty((w.T, w.H, 512), dtype=torch.bfloat16, device=dev)
        l = torch.empty((w.T, w.H), dtype=torch.float32, device=dev)
        ms_q = statistics.median(timed_steps(lambda: dsa.dsa_kv_fp8_quantize(kv, 64, out=fp8), steps, warmup,
                                             stream, flush))
        ms_d = statistics.median(timed_steps(lambda: dsa.dsa_kv_fp8_dequantize(fp8, 64, out=deq), steps, warmup,
                                             stream, flush))
        def fp8_step():
            dsa.dsa_kv_fp8_dequantize(fp8, 64, out=deq)
            dsa.dsa_sparse_prefill(q, deq, idx, w.k, w.scale, out=o, lse=l)
        ms_s = statistics.median(timed_steps(fp8_step, steps, warmup, stream, flush))
        ms_f = statistics.median(timed_steps(lambda: dsa.dsa_sparse_prefill_fp8(q, fp8, idx, w.k, w.scale, out=o,
                                                                                 lse=l), steps, warmup, stream, flush))
        rb = dsa.dsa_kv_fp8_row_bytes(64)
        qbytes = w.N * (w.d_qk * 2 + rb)
        dbytes = w.N * (rb + w.d_qk * 2)
        _, fbytes, fflops = sparse_work(w, x.idx, row_bytes=rb)
        out["v32_h32_16k_fp8kv"] = {
            "cache_bytes": w.N * rb, "cache_bytes_bf16": w.N * w.d_qk * 2,
            "quantize": {"ms": ms_q, "gbs": qbytes / ms_q / 1e6, "hbm_frac": qbytes / ms_q / 1e6 / peaks["hbm_gbs"]},
            "dequantize": {"ms": ms_d, "gbs": dbytes / ms_d / 1e6, "hbm_frac": dbytes / ms_d / 1e6 / peaks["hbm_gbs"]},
            "dequantize_plus_per_token": {"ms": ms_s, "query_tokens_per_s": w.T / ms_s * 1e3},
            "per_token_fp8": {"ms": ms_f, "query_tokens_per_s": w.T / ms_f * 1e3,
                              "algorithmic_bytes": fbytes, "row_bytes": rb, "logical_gbs": fbytes / ms_f / 1e6,
                              "hbm_frac_logical": fbytes / ms_f / 1e6 / peaks["hbm_gbs"],
                              "useful_tflops": fflops / ms_f / 1e9}}
        del q, kv, idx, fp8, deq, o, l
        torch.cuda.empty_cache()

    # masked dense MHA: DeepSeek-V3.2 geometry (contiguous per-head q/k/v),
    # then the GLM NoPE and GLM-5 geometries with k and v read as views of one
    # per-head projection output and the RoPE key columns shared
    def masked_block(name):
        w = WORKLOADS[name]
        log(f"mode {name}")
        x = make_masked_inputs(w)
        words = (max(w.kv_lens) + 31) // 32
        words = (words + 3) // 4 * 4
        idx = torch.from_numpy(x.idx).to(dev)
        km = torch.empty((w.T, words), dtype=torch.int32, device=dev)
        kfn = lambda: dsa.dsa_topk_to_key_mask(idx, w.k, words, cu_seqlens_q=x.cu_seqlens_q,
                                               cu_seqlens_kv=x.cu_seqlens_kv, out=km)
        ms_k = statistics.median(timed_steps(kfn, steps, warmup, stream, flush))
        res = {"T": w.T, "H": w.H, "d_qk": w.d_qk, "d_rope": w.d_rope, "d_v": w.d_v, "key_mask": {"ms": ms_k}}
        try:
            q = to_dev(x.q, dev)
            o = torch.empty((w.T, w.H, w.d_v), dtype=torch.bfloat16, device=dev)
            l = torch.empty((w.T, w.H), dtype=torch.float32, device=dev)
            if w.split_kv:
                dn = w.d_qk - w.d_rope
                kvp = to_dev(x.kvp, dev)
                k_pe = to_dev(x.k_pe, dev) if x.k_pe is not None else None
                k, v = kvp[..., :dn], kvp[..., dn:]
                mfn = lambda: dsa.dsa_masked_mha_prefill_strided(q, k, v, km, w.scale, k_pe=k_pe,
                                                                 cu_seqlens_q=x.cu_seqlens_q,
                                                                 cu_seqlens_kv=x.cu_seqlens_kv, out=o, lse=l)
            else:
                k, v = to_dev(x.k, dev), to_dev(x.v, dev)
                mfn = lambda: dsa.dsa_masked_mha_prefill(q, k, v, km, w.scale, cu_seqlens_q=x.cu_seqlens_q,
                                                         cu_seqlens_kv=x.cu_seqlens_kv, out=o, lse=l)
            mfn()
            ms_m = statistics.median(timed_steps(mfn, steps, warmup, stream, flush))
            pairs = int((x.idx[:, :w.k] >= 0).sum())
            useful = 2.0 * w.H * pairs * (w.d_qk + w.d_v)
            causal = sum(2.0 * w.H * (n * (n + 1) / 2) * (w.d_qk + w.d_v) for n in w.q_lens)
            res["masked"] = {"ms": ms_m, "query_tokens_per_s": w.T / ms_m * 1e3,
                             "useful_tflops": useful / ms_m / 1e9, "dense_causal_tflops": causal / ms_m / 1e9,
                             "tensor_frac_dense_causal": causal / ms_m / 1e9 / peaks["bf16_tflops"]}
        except dsa.DSAError as e:
            res["masked"] = {"unavailable": str(e)}
        return res

    for name in ("masked_2x8192", "masked_nope_2x8192", "masked_glm5_2x8192"):
        if want(name):
            out[name] = masked_block(name)
            torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------------------------
# arms
# ----------------------------------------------------------------------------
def headline_config(w, x, world):
    """The workload description both arms print (same keys, same values)."""
    return {"workload": w.name, "T": w.T, "N": w.N, "H": w.H, "d_qk": w.d_qk, "d_v": w.d_v, "k": w.k,
            "ld": w.ld, "index_gen": "locality (8-token blocks, 2048 base + 352-position shared pool)",
            "valid_pairs": int((x.idx[:, :w.k] >= 0).sum()),
            "l2": "flushed before every timed step (256 MiB write, outside the events)",
            "parallelism": f"replica per GPU x{world}"}


def run_ours(args):
    import torch
    import torch.distributed as dist
    import dsa_sparse_mla_prefill_gb300 as dsa
    from synth import WORKLOADS, make_sparse_inputs

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks = measured_peaks()
    w = rank_workload(WORKLOADS[HEADLINE], rank)

    # CPU baseline pool first (spawn), before heavy GPU work
    pool = None
    cores = os.cpu_count() or 1
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        pool = oracle_pool(cores)

    log(f"generating {w.name}")
    x = make_sparse_inputs(w)
    pairs, abytes, flops = sparse_work(w, x.idx)
    log("inputs ready")
    q, kv = to_dev(x.q, dev), to_dev(x.kv, dev)
    idx = torch.from_numpy(x.idx).to(dev)
    out = torch.empty((w.T, w.H, w.d_v), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.T, w.H), dtype=torch.float32, device=dev)
    flush_buf = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush = lambda: flush_buf.zero_()
    stream = torch.cuda.current_stream(dev)
    step = lambda: dsa.dsa_sparse_prefill(q, kv, idx, w.k, w.scale, out=out, lse=lse)

    # one untimed step first: the device error counters must be clean (no
    # out-of-range index, no bounded wait that ran out) before anything is timed
    step()
    torch.cuda.synchronize()
    st, counts = dsa.dsa_last_device_error()
    if st != 0:
        raise RuntimeError(f"device error counters after the first step: {counts}")

    log("first step ok; timing")
    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        flush()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks.mark()
    clocks.stop()
    ms = [a.elapsed_time(b) for a, b in ev]
    ms_step = max_over_ranks(sum(ms) / len(ms), dist, dev)
    value = job_throughput(w.T, world, ms_step)
    # beside the cold-L2 headline: the same steps back to back (no flush), L2 as the previous step left it
    hot_ms = max_over_ranks(statistics.mean(timed_steps(step, args.steps, 1, stream, None)), dist, dev)

    log(f"timed: {ms_step:.3f} ms/step")
    # end-to-end through host buffers: every step the host call copies q, kv
    # and the indices in from pinned host memory and out and lse back, in
    # chunks whose copies overlap the kernel (dsa_sparse_prefill_host)
    hq = torch.from_numpy(np.ascontiguousarray(x.q).view(np.int16)).view(torch.bfloat16).pin_memory()
    hkv = torch.from_numpy(np.ascontiguousarray(x.kv).view(np.int16)).view(torch.bfloat16).pin_memory()
    hidx = torch.from_numpy(x.idx).pin_memory()
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    hlse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    del q, idx
    torch.cuda.empty_cache()
    chunk = args.e2e_chunk
    # streamed form: a workspace that holds every token (sized with chunk_tokens
    # >= T), one kernel launch, the copies in chunks of at most `chunk` tokens
    ws = torch.empty(dsa.dsa_sparse_prefill_host_workspace(w.T, w.N, w.d_qk, w.H, w.d_qk, w.ld, w.T, True),
                     dtype=torch.uint8, device=dev)

    def e2e_step():
        dsa.dsa_sparse_prefill_host(hq, hkv, hidx, w.k, w.scale, hout, hlse, ws, chunk_tokens=chunk, stream=stream)

    e2e_steps = max(3, min(args.steps, 20))
    e2e_ms = statistics.mean(timed_steps(e2e_step, e2e_steps, min(args.warmup, 3), stream, flush))
    del ws
    # the ring form beside it: three chunk buffer sets, one kernel launch per chunk
    ws_ring = torch.empty(dsa.dsa_sparse_prefill_host_workspace(w.T, w.N, w.d_qk, w.H, w.d_qk, w.ld, chunk, True),
                          dtype=torch.uint8, device=dev)

    def ring_step():
        dsa.dsa_sparse_prefill_host(hq, hkv, hidx, w.k, w.scale, hout, hlse, ws_ring, chunk_tokens=chunk,
                                    stream=stream)

    ring_ms = max_over_ranks(statistics.mean(timed_steps(ring_step, e2e_steps, min(args.warmup, 3), stream, flush)),
                             dist, dev)
    del ws_ring
    h2d = hq.numel() * 2 + hkv.numel() * 2 + hidx.numel() * 4
    d2h = hout.numel() * 2 + hlse.numel() * 4
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)
    # the copy engines alone on the same pinned buffers: one host -> device copy
    # of q and one device -> host copy of out per step (what bounds the e2e step
    # when the kernel is shorter than its copies)
    dq = torch.empty(hq.shape, dtype=hq.dtype, device=dev)
    dout = torch.empty(hout.shape, dtype=hout.dtype, device=dev)
    h2d_ms = statistics.median(timed_steps(lambda: dq.copy_(hq, non_blocking=True), 5, 2, stream))
    d2h_ms = statistics.median(timed_steps(lambda: hout.copy_(dout, non_blocking=True), 5, 2, stream))
    h2d_gbs = hq.numel() * 2 / h2d_ms / 1e6
    d2h_gbs = hout.numel() * 2 / d2h_ms / 1e6
    del dq, dout

    log(f"e2e: {e2e_ms:.3f} ms/step")
    src_hash = kernel_source_hash(["sparse_prefill.cu", "dsa_device.cuh"])
    traffic = profiled_traffic("sparse_prefill_" + HEADLINE, src_hash, w.T)
    achieved = abytes / (ms_step / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "query-tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": headline_config(w, x, world),
        "useful_tflops": world * flops / (ms_step / 1e3) / 1e12,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                     "basis": "logical bytes: every selected row once per token (the form's defining re-gather) "
                              "+ q, out, indices, lse, over the kernel time; the 18.9 MB KV table stays in the "
                              "L2, so DRAM carries only `traffic` of it and the kernel is bound by its gather "
                              "issue rate, not by DRAM",
                     "dram_gbs": (traffic / (ms_step / 1e3) / 1e9) if traffic else None,
                     "kernel": "dsa::sparse::sparse_prefill_kernel<32,9>",
                     "algorithmic_bytes": abytes, "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs)"},
        "hot_l2": {"ms_per_step": hot_ms, "value": job_throughput(w.T, world, hot_ms), "unit": "query-tokens/s",
                   "l2": "not flushed between steps"},
        "e2e": {"value": job_throughput(w.T, world, e2e_ms), "unit": "query-tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "call": "dsa_sparse_prefill_host",
                "form": "streamed: one kernel launch over all tokens, copies in chunks",
                "chunk_tokens": chunk, "kernel_ms": ms_step,
                "ring_form_ms_per_step": ring_ms,
                "h2d_gbs": h2d_gbs, "d2h_gbs": d2h_gbs,
                "copy_floor_ms": max(h2d / h2d_gbs, d2h / d2h_gbs) / 1e6,
                "note": "copy floor = the larger direction's bytes at the rate measured for one plain copy of "
                        "the same pinned buffers; the step cannot be shorter than it or than the kernel"},
        "gpu_launches": args.steps,
        "clocks": clocks.summary(),
    }
    if rank == 0 and not args.no_modes:
        del hq, hkv, hidx, hout, hlse
        try:
            modes = run_modes(dev, stream, peaks, args.steps, args.warmup, flush)
        except Exception as e:  # report, never hide the headline
            modes = {"error": repr(e)}
        # the grouped form on its own workload (21504 queries after 11264
        # cached rows, H = 16, G = 8) as a top-level key, ahead of `modes`
        g = modes.get("grouped_21k_of_32k", {})
        if "grouped" in g and "union_build" in g:
            grouped = {"workload": "grouped_21k_of_32k", "ms": g["grouped"].get("ms"),
                       "union_build_ms": g["union_build"]["ms"],
                       "with_union_build_ms": g["grouped"].get("with_union_build_ms"),
                       "union_plus_useful_tflops": g["grouped"].get("union_plus_useful_tflops"),
                       "tensor_frac": g["grouped"].get("tensor_frac"),
                       "peak_tflops": peaks["bf16_tflops"], "union_mean": g.get("union_mean")}
            keys = list(line)
            at = keys.index("roofline") + 1
            line = {k: line[k] for k in keys[:at]} | {"grouped": grouped} | {k: line[k] for k in keys[at:]}
        line["modes"] = modes
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        log("cpu baseline")
        line["cpu_baseline"] = cpu_baseline(w, x, budget_s=args.cpu_budget, pool=pool, cores=cores)
        pool.close()
        pool.join()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def _attach_shared(spec):
    """Views of the arrays the parent placed in shared memory (name, shape, dtype)."""
    from multiprocessing import shared_memory
    global _SHM
    _SHM = []
    out = []
    for name, shape, dtype in spec:
        shm = shared_memory.SharedMemory(name=name)
        _SHM.append(shm)
        out.append(np.ndarray(shape, dtype=dtype, buffer=shm.buf))
    return out


def _oracle_pass_worker(args):
    """The oracle over the tokens [lo, hi) of the shared workload, 16 per call.
    Returns the seconds it took."""
    spec, lo, hi, k, scale, d_qk, d_v = args
    q, kv, idx = _attach_shared(spec)
    from oracle.dsa_oracle import sparse_prefill
    t0 = time.perf_counter()
    for s in range(lo, hi, 16):
        e = min(hi, s + 16)
        sparse_prefill(q[s:e], kv, idx[s:e], k, scale, d_qk, d_v)
    return time.perf_counter() - t0


def run_reference(args):
    """The oracle, as it stands, timed on the host cores on the headline
    workload (rank 0 only; the other ranks exit).  The inputs sit in shared
    memory; each timed step is one pass of all cores over the same tokens: the
    whole 16384-token chunk when K such passes (and W warm-up passes over a
    quarter of it) fit in about five minutes, else a fixed share of it spread
    over the chunk (stated in the line).  ms_per_step is
    the measured wall time of a step; value = tokens per step / that time."""
    from multiprocessing import shared_memory
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from synth import WORKLOADS, make_sparse_inputs
    w = WORKLOADS[HEADLINE]
    x = make_sparse_inputs(w)
    cores = os.cpu_count() or 1
    shms, spec = [], []
    for a in (x.q, x.kv, x.idx):
        a = np.ascontiguousarray(a)
        shm = shared_memory.SharedMemory(create=True, size=max(1, a.nbytes))
        np.ndarray(a.shape, dtype=a.dtype, buffer=shm.buf)[...] = a
        shms.append(shm)
        spec.append((shm.name, a.shape, a.dtype.str))
    pool = oracle_pool(cores)
    try:
        def one_pass(n):
            # core c takes n / cores consecutive tokens starting at its
            # c / cores point of the chunk: the whole chunk when n = T, else
            # equal ranges spread over the chunk (early and late positions)
            width = -(-n // cores)
            tasks = []
            for c in range(cores):
                lo = w.T * c // cores
                hi = min(lo + width, w.T * (c + 1) // cores)
                if hi > lo:
                    tasks.append((spec, lo, hi, w.k, w.scale, w.d_qk, w.d_v))
            t0 = time.perf_counter()
            pool.map(_oracle_pass_worker, tasks)
            return time.perf_counter() - t0, sum(t[2] - t[1] for t in tasks)

        # rate estimate from a small pass, then the largest share that fits
        est_s, est_n = one_pass(min(w.T, 32 * cores))
        per_token = est_s / est_n
        # warm-up passes take a quarter of the step's tokens; the K timed
        # passes and the warm-up together stay within about five minutes
        budget = 300.0 / max(1, args.steps + args.warmup / 4)
        n = w.T if per_token * w.T <= budget else max(16 * cores, int(budget / per_token) // (16 * cores) * 16 * cores)
        for _ in range(args.warmup):
            one_pass(max(cores, n // 4))
        secs = []
        for _ in range(args.steps):
            sec, done = one_pass(n)
            secs.append(sec)
    finally:
        pool.close()
        pool.join()
        for shm in shms:
            shm.close()
            shm.unlink()
    step_s = statistics.mean(secs)
    value = done / step_s
    full = done == w.T
    sample = (f"{'all' if full else 'a share of'} {done} of {w.T} tokens of {w.name} per step "
              f"({'one whole pass' if full else 'contiguous ranges spread over the chunk'}), fp64 numpy oracle in "
              f"batches of 16, {cores} spawn workers x 1 BLAS thread, inputs in shared memory; "
              f"{args.steps} timed passes of {step_s:.2f} s")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "query-tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": headline_config(w, x, world),
            "cpu_baseline": {"value": value, "unit": "query-tokens/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "query-tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def traced_launch(fn, cap, out_path=None):
    """One launch with the diagnostic timeline on (CTAs 0 and 1, first `cap`
    tiles, 8 clock64 stamps per tile).  Returns per-event medians in cycles
    relative to event 2 of the same tile, and the median tile period."""
    import torch
    import dsa_sparse_mla_prefill_gb300 as dsa
    buf = torch.zeros(2 * cap * 8, dtype=torch.int64, device="cuda")
    dsa.dsa_debug_trace(buf, cap)
    try:
        fn()
        torch.cuda.synchronize()
    finally:
        dsa.dsa_debug_trace()
    arr = buf.cpu().numpy().reshape(2, cap, 8).astype(np.int64)
    if out_path:
        np.save(out_path, arr)
    out = {}
    for c in range(2):
        a = arr[c]
        ok = np.all(a[:, 1:] > 0, axis=1) if a.shape[0] else np.zeros(0, bool)
        a = a[ok]
        if len(a) < 3:
            out[f"cta{c}"] = {"tiles": int(len(a))}
            continue
        rel = {f"ev{e}-ev2": float(np.median(a[:, e] - a[:, 2])) for e in range(8)}
        per = float(np.median(np.diff(a[:, 2])))
        out[f"cta{c}"] = {"tiles": int(len(a)), "period_cycles": per, **rel}
    return out


def measure_forms(L, dev, stream, flush, steps, warmup):
    """The three forms on one causal request of L tokens, DeepSeek-V3.2 at TP4
    (H = 32, top-2048; latent 576/512 for per-token and grouped with G = 4,
    per-head 192/128 for masked, the same indices): median ms of each kernel,
    the union rows and the device error counts."""
    import torch
    import dsa_sparse_mla_prefill_gb300 as dsa
    from synth import Workload, make_masked_inputs, make_sparse_inputs
    common = dict(q_lens=(L,), kv_lens=(L,), H=32, k=2048, ld=2048, scale=1.0 / math.sqrt(192.0),
                  index_gen="locality", seed=7)
    ws = Workload(name=f"causal_{L}", mode="sparse", d_qk=576, d_v=512, G=4, **common)
    wm = Workload(name=f"causal_{L}", mode="masked", d_qk=192, d_v=128, **common)
    x = make_sparse_inputs(ws)
    q, kv = to_dev(x.q, dev), to_dev(x.kv, dev)
    idx = torch.from_numpy(x.idx).to(dev)
    med = lambda fn: statistics.median(timed_steps(fn, steps, warmup, stream, flush))
    res = {"L": L, "H": 32, "k": 2048}
    o = torch.empty((L, 32, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((L, 32), dtype=torch.float32, device=dev)
    res["per_token_ms"] = med(lambda: dsa.dsa_sparse_prefill(q, kv, idx, ws.k, ws.scale, out=o, lse=lse))
    upad = dsa.dsa_union_pad(4, ws.k, 128)
    ng = dsa.dsa_num_groups(x.cu_seqlens_q, L, 4)
    u = torch.empty((ng, upad), dtype=torch.int32, device=dev)
    ul = torch.empty((ng,), dtype=torch.int32, device=dev)
    m = torch.empty((ng, upad), dtype=torch.uint8, device=dev)
    res["union_ms"] = med(lambda: dsa.dsa_union_build(idx, ws.k, 4, L, cu_seqlens_q=x.cu_seqlens_q,
                                                      union_pad=upad, out=(u, ul, m)))
    res["union_rows"] = int(ul.sum().item())
    res["grouped_ms"] = med(lambda: dsa.dsa_grouped_prefill(q, kv, u, ul, m, 4, ws.scale,
                                                            cu_seqlens_q=x.cu_seqlens_q, out=o, lse=lse))
    del q, kv, o, u, ul, m
    torch.cuda.empty_cache()
    xm = make_masked_inputs(wm)
    assert np.array_equal(xm.idx, x.idx)
    words = ((L + 31) // 32 + 3) // 4 * 4
    km = torch.empty((L, words), dtype=torch.int32, device=dev)
    res["key_mask_ms"] = med(lambda: dsa.dsa_topk_to_key_mask(idx, wm.k, words, cu_seqlens_q=xm.cu_seqlens_q,
                                                              cu_seqlens_kv=xm.cu_seqlens_kv, out=km))
    qm, mk, mv = to_dev(xm.q, dev), to_dev(xm.k, dev), to_dev(xm.v, dev)
    om = torch.empty((L, 32, 128), dtype=torch.bfloat16, device=dev)
    res["masked_ms"] = med(lambda: dsa.dsa_masked_mha_prefill(qm, mk, mv, km, wm.scale, cu_seqlens_q=xm.cu_seqlens_q,
                                                              cu_seqlens_kv=xm.cu_seqlens_kv, out=om, lse=lse))
    st, counts = dsa.dsa_last_device_error()
    res["device_errors"] = counts
    del qm, mk, mv, om, km, idx
    torch.cuda.empty_cache()
    return res


def run_form_sweep(args):
    """measure_forms at each prompt length of --sweep-forms, one JSON line
    each, with the form model's prediction beside the measurement: the
    crossovers the form dispatcher is calibrated on."""
    import torch
    import dsa_sparse_mla_prefill_gb300 as dsa
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    flush_buf = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush = lambda: flush_buf.zero_()
    steps = max(3, min(args.steps, 10))
    for L in [int(v) for v in args.sweep_forms.split(",")]:
        res = measure_forms(L, dev, stream, flush, steps, args.warmup)
        measured = {"per_token": res["per_token_ms"], "grouped": res["union_ms"] + res["grouped_ms"],
                    "masked": res["key_mask_ms"] + res["masked_ms"]}
        form, pred, _ = dsa.dsa_choose_form([L], [L], 32, 2048, 576, (192, 128), union_rows=res["union_rows"])
        res["measured_best"] = min(measured, key=measured.get)
        res["model_choice"] = form
        res["model_ms"] = pred
        print(json.dumps(res), flush=True)
        if any(res["device_errors"][1:3]):
            raise SystemExit(1)


def run_profile_case(args):
    """A small, bounded case of one kernel for ncu captures: inputs larger than
    the L2 but a few hundred MB at most; runs warmup + steps launches."""
    import torch
    import dsa_sparse_mla_prefill_gb300 as dsa
    from synth import WORKLOADS, make_masked_inputs, make_sparse_inputs, scaled_down
    dev = torch.device("cuda", 0)
    n = args.profile_tokens
    if args.profile in ("sparse", "sparse_fp8", "union", "grouped"):
        base = WORKLOADS[args.profile_workload or
                         ("v32_h32_16k" if args.profile.startswith("sparse") else "grouped_21k_of_32k")]
        w = scaled_down(base, (n,), (base.N,), name=f"{base.name}_last{n}")
        x = make_sparse_inputs(w)
        q, kv = to_dev(x.q, dev), to_dev(x.kv, dev)
        idx = torch.from_numpy(x.idx).to(dev)
        if args.profile == "sparse":
            fn = lambda: dsa.dsa_sparse_prefill(q, kv, idx, w.k, w.scale)
        elif args.profile == "sparse_fp8":
            d_rope = w.d_qk - 512
            f8 = dsa.dsa_kv_fp8_quantize(kv, d_rope)
            fn = lambda: dsa.dsa_sparse_prefill_fp8(q, f8, idx, w.k, w.scale, d_rope=d_rope)
        else:
            upad = dsa.dsa_union_pad(w.G, w.k, 128)
            u, ul, m = dsa.dsa_union_build(idx, w.k, w.G, w.N, cu_seqlens_q=x.cu_seqlens_q, union_pad=upad)
            if args.profile == "union":
                fn = lambda: dsa.dsa_union_build(idx, w.k, w.G, w.N, cu_seqlens_q=x.cu_seqlens_q, union_pad=upad,
                                                 out=(u, ul, m))
            else:
                fn = lambda: dsa.dsa_grouped_prefill(q, kv, u, ul, m, w.G, w.scale, cu_seqlens_q=x.cu_seqlens_q)
    elif args.profile == "masked":
        base = WORKLOADS[args.profile_workload or "masked_2x8192"]
        w = scaled_down(base, (n,), (base.kv_lens[0],), name=f"{base.name}_last{n}")
        x = make_masked_inputs(w)
        words = ((max(w.kv_lens) + 31) // 32 + 3) // 4 * 4
        idx = torch.from_numpy(x.idx).to(dev)
        km = dsa.dsa_topk_to_key_mask(idx, w.k, words, cu_seqlens_q=x.cu_seqlens_q, cu_seqlens_kv=x.cu_seqlens_kv)
        q = to_dev(x.q, dev)
        if w.split_kv:
            dn = w.d_qk - w.d_rope
            kvp = to_dev(x.kvp, dev)
            k_pe = to_dev(x.k_pe, dev) if x.k_pe is not None else None
            fn = lambda: dsa.dsa_masked_mha_prefill_strided(q, kvp[..., :dn], kvp[..., dn:], km, w.scale, k_pe=k_pe,
                                                            cu_seqlens_q=x.cu_seqlens_q,
                                                            cu_seqlens_kv=x.cu_seqlens_kv)
        else:
            k, v = to_dev(x.k, dev), to_dev(x.v, dev)
            fn = lambda: dsa.dsa_masked_mha_prefill(q, k, v, km, w.scale, cu_seqlens_q=x.cu_seqlens_q,
                                                    cu_seqlens_kv=x.cu_seqlens_kv)
    else:
        raise ValueError(args.profile)
    ms = timed_steps(fn, args.steps, args.warmup, torch.cuda.current_stream(dev))
    st, counts = dsa.dsa_last_device_error()
    res = {"profile": args.profile, "workload": w.name, "T": w.T, "ms": statistics.median(ms), "device_errors": counts}
    if args.trace > 0:
        res["trace"] = traced_launch(fn, args.trace, args.trace_out)
    print(json.dumps(res), flush=True)
    if st != 0:
        raise SystemExit(1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-modes", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-chunk", type=int, default=1216, help="tokens per chunk of the host-buffer call (8 per SM)")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work per core")
    ap.add_argument("--profile", choices=["sparse", "sparse_fp8", "union", "grouped", "masked"], default=None,
                    help="run a small case of one kernel (for ncu) instead of the benchmark")
    ap.add_argument("--profile-tokens", type=int, default=2048)
    ap.add_argument("--profile-workload", default=None,
                    help="profile mode: base workload, e.g. nope_2x8192 or masked_nope_2x8192")
    ap.add_argument("--sweep-forms", default=None,
                    help="comma list of prompt lengths: time per-token, grouped and masked on one causal request each")
    ap.add_argument("--trace", type=int, default=0, help="profile mode: record a per-tile timeline of N tiles")
    ap.add_argument("--trace-out", default=None, help="profile mode: save the raw timeline (.npy)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.profile:
        run_profile_case(args)
    elif args.sweep_forms:
        run_form_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
