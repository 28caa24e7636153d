#!/usr/bin/env python
"""Benchmark: paged MLA decode on GB300.

One step = the whole decode path for one batch of synthetic inputs already
resident in HBM: schedule (mla_get_metadata) + split-KV decode + combine
(mla_decode).  The headline workload is the memory-bound dense mix (batch
128, 16 heads, lengths U[1024, 8192]); its KV (~680 MB) is larger than L2, so
no flush is needed between steps.  At one GPU the compute-bound dense and the
two sparse FP8 workloads are measured too and reported under "workloads".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mla|reference]

Prints one JSON line (rank 0).  --impl reference times the fp64 CPU oracle
on a bounded sample of the same workload (the reference arm).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from paged_mla_decode_07_gb300 import workloads as W  # noqa: E402

METRIC = "MLA decode TFLOPS & KV GB/s (bf16 dense, fp8 sparse) as % of GB300 roofline"
HEADLINE = "dense_membound"
D_QK, D_V, FP8_ROW = 576, 512, 656


# ----------------------------------------------------------------------------
# algorithmic work per step
# ----------------------------------------------------------------------------
def algorithmic(inp) -> dict:
    """Nominal FLOPs 2*h_q*s_q*s_k*(576+512) (s_k = length, or topk in sparse mode), the valid-only
    FLOPs, and the bytes the path must move once: KV rows (each cached token once per element in
    dense mode; each valid gathered row in sparse mode) + q + out + lse + tables/indices."""
    w = inp.workload
    lens = inp.cache_seqlens.cpu().numpy().astype(np.int64)
    rows = w.batch * w.s_q * w.h_q
    q_bytes = rows * D_QK * 2
    out_bytes = rows * D_V * 2 + rows * 4
    if w.mode == "sparse":
        idx = inp.indices
        valid = ((idx >= 0) & (idx < inp.cache_seqlens.view(-1, 1, 1))).sum().item()
        row = (644 if w.fp8_scales == "token" else FP8_ROW) if w.is_fp8 else D_QK * 2  # 640 B + a 4-byte scale
        kv_bytes = valid * row
        flops = 2.0 * w.h_q * w.s_q * w.topk * w.batch * (D_QK + D_V)
        vflops = 2.0 * w.h_q * valid * (D_QK + D_V)
        tab = idx.numel() * 4 + inp.block_table.numel() * 4
    else:
        kv_bytes = int(lens.sum()) * (FP8_ROW if w.is_fp8 else D_QK * 2)  # dense over bf16 or FP8 rows
        flops = 2.0 * w.h_q * w.s_q * float(lens.sum()) * (D_QK + D_V)
        if w.causal:
            vk = sum(max(0, min(L, L - w.s_q + i + 1)) for L in lens for i in range(w.s_q))
            vflops = 2.0 * w.h_q * vk * (D_QK + D_V)
        else:
            vflops = flops
        tab = int(((lens + 63) // 64).sum()) * 4 + w.batch * 4
    return dict(flops=flops, valid_flops=vflops, kv_bytes=kv_bytes,
                bytes=kv_bytes + q_bytes + out_bytes + tab)


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the dominant kernel
# of the headline workload, from one `ncu --clock-control none` capture of those two metrics (a
# `--set full` capture gives the same figure) of `bench.py --workload dense_membound --no-extras
# --steps 3 --warmup 3`.  A figure holds only for the kernel sources it was taken with: their
# SHA-256 prefix is stored beside it and the bench reports null once the sources differ.
NCU_TRAFFIC = {
    "dense_membound": (651.06e6, "62004e45a5329671"),
}
# the sources the headline's dominant kernel (the single-CTA decode kernel) is built from
KERNEL_SOURCES = ("mla_decode.cu", "mla_device.cuh", "mla_internal.h")


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "paged_mla_decode_07_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(workload: str):
    """Bytes per launch of the dominant kernel from the stored capture, or None if stale/absent."""
    entry = NCU_TRAFFIC.get(workload)
    if entry is None or entry[1] != kernel_source_hash():
        return None
    return entry[0]


def kernel_name(w) -> str:
    """The decode kernel the library runs for workload w: problems of more than 64 rows, dense over
    the bf16 cache or sparse over the FP8 cache, run on CTA pairs; the rest on single CTAs of 16, 32
    or 64 rows."""
    rows = w.h_q if w.mode == "sparse" else w.s_q * w.h_q
    kmode = ("sparse" if w.is_fp8 else "sparse_bf16") if w.mode == "sparse" else ("dense_fp8" if w.is_fp8 else "dense")
    if rows > 64 and kmode in ("dense", "sparse"):
        return f"mla_decode_pair_kernel<{kmode}>"
    rpc = 16 if rows <= 16 else (32 if rows <= 32 else 64)
    return f"mla_decode_kernel<{rpc},{kmode}>"


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        lines = [l.strip() for l in open(self.file.name) if l.strip()]
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------
# the CUDA path
# ----------------------------------------------------------------------------
class DecodeStep:
    """Device-resident inputs + preallocated outputs; __call__ runs one step on the current stream."""

    def __init__(self, inp, device):
        import paged_mla_decode_07_gb300 as mla
        self.mla = mla
        self.w = inp.workload
        self.d = inp.to(device) if inp.q.device != torch.device(device) else inp
        self.topk = 0 if self.d.indices is None else self.d.indices.shape[-1]
        b, s, h = self.w.batch, self.w.s_q, self.w.h_q
        self.is_fp8 = self.d.kvcache.dtype == torch.uint8
        self.cfg = dict(h_q=h, s_q=s, topk=self.topk, is_fp8=self.is_fp8)
        self.out = torch.empty((b, s, h, D_V), dtype=torch.bfloat16, device=device)
        self.lse = torch.empty((b, s, h), dtype=torch.float32, device=device)
        self.ws = torch.empty(max(256, mla.workspace_size(b, **self.cfg)), dtype=torch.uint8, device=device)
        ns, nn = mla.metadata_size(b, **self.cfg)
        self.sched = torch.empty(ns, dtype=torch.int32, device=device)
        self.nsplit = torch.empty(nn, dtype=torch.int32, device=device)
        self.g_step = self.g_decode = None

    def metadata(self):
        self.mla.get_metadata(self.d.cache_seqlens, **self.cfg, sched=self.sched, num_splits=self.nsplit)

    def decode(self):
        d = self.d
        self.mla.decode(d.q, d.kvcache, d.block_table, d.cache_seqlens, d.sm_scale, self.sched, self.nsplit,
                        is_causal=self.w.causal, indices=d.indices, out=self.out, lse=self.lse,
                        workspace=self.ws, kv_scales=d.kv_scales, topk_lengths=d.topk_lengths)

    def __call__(self):
        self.metadata()
        self.decode()

    def capture(self):
        """Record one step (and one decode call) as CUDA graphs, so a timed step is the device work
        alone, not the host-side argument marshalling of each call.  Returns False (eager steps)
        if capture is unavailable."""
        try:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                self()
            torch.cuda.current_stream().wait_stream(side)
            self.g_step = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.g_step):
                self()
            self.g_decode = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.g_decode):
                self.decode()
            torch.cuda.synchronize()
            return True
        except Exception as e:  # capture unsupported in this environment: time eager calls
            print(f"CUDA graph capture unavailable ({e}); timing eager calls", file=sys.stderr)
            self.g_step = self.g_decode = None
            return False

    def replay_step(self):
        if self.g_step is not None:
            self.g_step.replay()
        else:
            self()

    def replay_decode(self):
        if self.g_decode is not None:
            self.g_decode.replay()
        else:
            self.decode()


L2_BYTES = 129 * 1000 * 1000  # GB300 L2


class L2Flush:
    """Writes a buffer twice the size of L2 between timed calls (outside the timed region), for
    workloads whose bytes fit in L2."""

    def __init__(self, device):
        self.buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=device)

    def __call__(self):
        self.buf.add_(1)


def time_events(fn, n: int, flush=None):
    """Per-call device durations (ms) with CUDA events on the current stream; `flush` (if given)
    runs before each call, outside its events."""
    s = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    torch.cuda.synchronize()
    for a, b in ev:
        if flush is not None:
            flush()
        a.record(s)
        fn()
        b.record(s)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def e2e_step_factory(inp, device, resident_cache=False):
    """End to end through the public API: pinned host inputs -> H2D copies -> schedule + decode ->
    D2H of out and lse, every step.  With resident_cache the KV cache stays in device memory (as it
    does in a serving loop) and only q, the block table and the lengths cross the link."""
    import paged_mla_decode_07_gb300 as mla
    w = inp.workload
    names = ("q", "block_table", "cache_seqlens") if resident_cache else ("q", "kvcache", "block_table",
                                                                          "cache_seqlens")
    host = {k: getattr(inp, k).cpu().pin_memory() for k in names}
    if inp.indices is not None:
        host["indices"] = inp.indices.cpu().pin_memory()
    dev = {k: torch.empty_like(v, device=device) for k, v in host.items()}
    if resident_cache:
        dev["kvcache"] = inp.kvcache.to(device)
    topk = 0 if inp.indices is None else inp.indices.shape[-1]
    b, s, h = w.batch, w.s_q, w.h_q
    cfg = dict(h_q=h, s_q=s, topk=topk, is_fp8=inp.kvcache.dtype == torch.uint8)
    out = torch.empty((b, s, h, D_V), dtype=torch.bfloat16, device=device)
    lse = torch.empty((b, s, h), dtype=torch.float32, device=device)
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    ws = torch.empty(max(256, mla.workspace_size(b, **cfg)), dtype=torch.uint8, device=device)
    ns, nn = mla.metadata_size(b, **cfg)
    sched = torch.empty(ns, dtype=torch.int32, device=device)
    nsplit = torch.empty(nn, dtype=torch.int32, device=device)
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = out.numel() * 2 + lse.numel() * 4

    def step():
        for k, v in host.items():
            dev[k].copy_(v, non_blocking=True)
        mla.get_metadata(dev["cache_seqlens"], **cfg, sched=sched, num_splits=nsplit)
        mla.decode(dev["q"], dev["kvcache"], dev["block_table"], dev["cache_seqlens"], inp.sm_scale, sched, nsplit,
                   is_causal=w.causal, indices=dev.get("indices"), out=out, lse=lse, workspace=ws)
        out_h.copy_(out, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)

    return step, h2d, d2h


def measure_workload(name, device, reps=50, warmup=10):
    """Kernel-level measurement of one workload (decode call = split-KV kernel + combine): the
    median of `reps` calls after `warmup` untimed ones."""
    inp = W.make_inputs(name, device=device)
    st = DecodeStep(inp, device)
    st.capture()
    st.metadata()
    for _ in range(warmup):
        st.replay_decode()
    a = algorithmic(inp)
    times = time_events(st.replay_decode, reps, flush=L2Flush(device) if a["bytes"] < L2_BYTES else None)
    ms = statistics.median(times)
    return inp, a, ms, st


def measure_store(device, peaks, batch=32, new_tokens=4096, reps=20):
    """FP8 cache write (mla_fp8_cache_store) of a prefill-sized chunk: batch x new_tokens bf16 tokens
    quantised into fresh pages.  Bytes = 1152 read + 656 written per token (larger than L2)."""
    import paged_mla_decode_07_gb300 as mla
    g = torch.Generator(device=device).manual_seed(1006)
    n = batch * new_tokens
    x = torch.randn((n, D_QK), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    offs = torch.arange(0, n + 1, new_tokens, dtype=torch.int32, device=device)
    lens = torch.zeros(batch, dtype=torch.int32, device=device)
    per = new_tokens // 64
    table = torch.randperm(batch * per, generator=g, device=device).int().reshape(batch, per)
    cache = torch.empty((batch * per, 64, 1, FP8_ROW), dtype=torch.uint8, device=device)
    fn = lambda: mla.fp8_cache_store(x, offs, lens, table, cache)
    for _ in range(3):
        fn()
    ms = statistics.median(time_events(fn, reps))
    gbs = n * (D_QK * 2 + FP8_ROW) / (ms * 1e-3) / 1e9
    return {"ms": round(ms, 5), "tokens": n, "gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4),
            "bytes_per_token": D_QK * 2 + FP8_ROW}


def measure_prefill(device, peaks, reps=10):
    """Sparse prefill (mla_sparse_prefill) on the named prefill workload: TFLOPS nominal
    (2 * h_q * s_q * topk * 1088) and valid-only, fraction of the measured bf16 peak."""
    import paged_mla_decode_07_gb300 as mla
    inp = W.make_prefill_inputs("sparse_prefill", device=device)
    w = inp.workload
    out = torch.empty((w.s_q, w.h_q, D_V), dtype=torch.bfloat16, device=device)
    lse = torch.empty((w.s_q, w.h_q), dtype=torch.float32, device=device)
    ws = torch.empty(mla.sparse_prefill_workspace_size(w.s_q, w.h_q, w.topk), dtype=torch.uint8, device=device)
    fn = lambda: mla.sparse_prefill(inp.q, inp.kv, inp.indices, inp.sm_scale, out=out, lse=lse, workspace=ws)
    for _ in range(3):
        fn()
    ms = statistics.median(time_events(fn, reps))
    valid = int(((inp.indices >= 0) & (inp.indices < w.s_kv)).sum().item())
    flops = 2.0 * w.h_q * w.s_q * w.topk * (D_QK + D_V)
    vflops = 2.0 * w.h_q * valid * (D_QK + D_V)
    tf = flops / (ms * 1e-3) / 1e12
    return {"ms": round(ms, 4), "tflops": round(tf, 2), "tflops_valid": round(vflops / (ms * 1e-3) / 1e12, 2),
            "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
            "shape": f"s_q {w.s_q}, s_kv {w.s_kv}, h_q {w.h_q}, topk {w.topk}"}


def measure_index(device, peaks, reps=10):
    """FP8 top-k indexer (mla_index_topk) on the named indexer workload.  Algorithmic bytes: every
    cached key once per element (128 code bytes + a 4-byte scale) + the query codes, scales and
    weights + the int32 ids written; FLOPs of the head dots 2 * 128 * h_idx per (query row, key)."""
    import paged_mla_decode_07_gb300 as mla
    inp = W.make_index_inputs("index_decode", device=device)
    w = inp.workload
    T = int(inp.row_offsets[-1])
    idx = torch.empty((T, w.topk), dtype=torch.int32, device=device)
    ws = torch.empty(mla.index_topk_workspace_size(T, inp.block_table.shape[1]), dtype=torch.uint8, device=device)
    fn = lambda: mla.index_topk(inp.q_codes, inp.q_scales, inp.weights, inp.row_offsets, inp.k_codes, inp.k_scales,
                                inp.block_table, inp.cache_seqlens, w.topk, relu=w.relu, max_new_tokens=w.n_new,
                                indices=idx, workspace=ws)
    for _ in range(3):
        fn()
    ms = statistics.median(time_events(fn, reps))
    lens = inp.cache_seqlens.cpu().numpy().astype(np.int64)
    nbytes = int(lens.sum()) * 132 + T * w.h_idx * (128 + 8) + T * w.topk * 4
    flops = 2.0 * 128 * w.h_idx * float(np.sum(lens * w.n_new))
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"ms": round(ms, 4), "gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4),
            "tflops_fp8": round(flops / (ms * 1e-3) / 1e12, 1),
            "shape": f"batch {w.batch}, {w.n_new} query tokens each, {w.h_idx} heads x 128, L {w.seqlen}, topk {w.topk}"}


# ----------------------------------------------------------------------------
# the oracle beside each workload: a bounded sample timed on the host cores
# ----------------------------------------------------------------------------
def _repeat(fn, min_s=1.0, max_reps=50):
    """Run fn until at least min_s seconds have passed; returns (seconds per run, runs)."""
    t0 = time.perf_counter()
    n = 0
    while True:
        fn()
        n += 1
        dt = time.perf_counter() - t0
        if dt >= min_s or n >= max_reps:
            return dt / n, n


def _cpu(sample: str, seconds: float, value: float, unit: str, threads: int = 0) -> dict:
    threads = threads or os.cpu_count()
    return {"value": round(value, 6), "unit": unit, "cores": threads, "kind": "oracle",
            "sample": f"{sample}, {seconds:.2f} s, fp64, {threads} thread{'s' if threads > 1 else ''}"}


def oracle_decode_rate(inp, max_rows=32) -> dict:
    """Oracle decode of the first rows of the first problem; TFLOPS counted as the GPU line counts them
    (2 * s_k * 1088 per row, s_k = the element's length, or topk in sparse mode)."""
    import oracle
    oracle.build()
    w = inp.workload
    cpu = inp.to("cpu")
    rows_per = w.h_q if w.mode == "sparse" else w.s_q * w.h_q
    rows = np.arange(min(rows_per, max_rows), dtype=np.int64)
    s_k = w.topk if w.mode == "sparse" else int(cpu.cache_seqlens[0])
    dt, n = _repeat(lambda: oracle.mla_decode(cpu.q, cpu.kvcache, cpu.block_table, cpu.cache_seqlens, cpu.sm_scale,
                                              is_causal=w.causal, indices=cpu.indices, rows=rows,
                                              kv_scales=cpu.kv_scales, topk_lengths=cpu.topk_lengths))
    flops = 2.0 * len(rows) * s_k * (D_QK + D_V)
    return _cpu(f"{len(rows)} rows of the first problem (s_k {s_k}) x{n}", dt * n, flops / dt / 1e12, "TFLOPS")


def oracle_prefill_rate(inp, max_rows=32) -> dict:
    import oracle
    oracle.build()
    w = inp.workload
    rows = np.arange(min(w.h_q, max_rows), dtype=np.int64)
    q, kv, idx = inp.q.cpu(), inp.kv.cpu(), inp.indices.cpu()
    dt, n = _repeat(lambda: oracle.sparse_prefill(q, kv, idx, inp.sm_scale, rows=rows))
    flops = 2.0 * len(rows) * w.topk * (D_QK + D_V)
    return _cpu(f"{len(rows)} rows of the first query token x{n}", dt * n, flops / dt / 1e12, "TFLOPS")


def oracle_index_rate(inp) -> dict:
    """Oracle top-k of the first element's query rows; GB/s of that element's algorithmic bytes."""
    import oracle
    oracle.build()
    w = inp.workload
    r1 = int(inp.row_offsets[1])
    sub = W.IndexInputs(w, inp.q_codes[:r1].cpu(), inp.q_scales[:r1].cpu(), inp.weights[:r1].cpu(),
                        torch.tensor([0, r1], dtype=torch.int32), inp.k_codes.cpu(), inp.k_scales.cpu(),
                        inp.block_table[:1].cpu(), inp.cache_seqlens[:1].cpu(), w.topk, w.relu, inp.seed)
    dt, n = _repeat(lambda: oracle.index_topk(sub))
    L = int(sub.cache_seqlens[0])
    nbytes = L * 132 + r1 * w.h_idx * (128 + 8) + r1 * w.topk * 4
    return _cpu(f"the first element ({r1} query rows x {L} keys) x{n}", dt * n, nbytes / dt / 1e9, "GB/s", threads=1)


def oracle_store_rate(n_tokens=2048) -> dict:
    import oracle
    oracle.build()
    g = torch.Generator().manual_seed(1006)
    x = torch.randn((n_tokens, D_QK), generator=g).to(torch.bfloat16)
    per = n_tokens // 64
    offs = torch.tensor([0, n_tokens], dtype=torch.int32)
    lens = torch.zeros(1, dtype=torch.int32)
    table = torch.randperm(per, generator=g).int().reshape(1, per)
    cache = torch.zeros((per, 64, 1, FP8_ROW), dtype=torch.uint8)
    dt, n = _repeat(lambda: oracle.fp8_cache_store(x, offs, lens, table, cache))
    return _cpu(f"{n_tokens} tokens x{n}", dt * n, n_tokens * (D_QK * 2 + FP8_ROW) / dt / 1e9, "GB/s", threads=1)


def max_over_ranks(x: float, device) -> float:
    """The largest x over all ranks of the default process group (x itself without one)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(name: str, rank: int) -> int:
    """Each rank decodes its own batch (weak scaling): rank r draws with the workload's seed + 100000*r."""
    return W.SEEDS[name] + 100000 * rank


def job_throughput(units_per_rank: float, world: int, ms_max: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time (per second)."""
    return units_per_rank * world / (ms_max * 1e-3)


def run_mla(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    import paged_mla_decode_07_gb300 as mla
    mla.build()
    peaks = load_peaks()

    # ---- headline workload: full steps
    wname = args.workload
    wdef = W.WORKLOADS[wname]
    if args.batch:
        # a reduced batch of the same workload (same per-CTA shape): for profiler captures
        from dataclasses import replace
        wdef = replace(wdef, batch=args.batch,
                       seqlens=wdef.seqlens[:args.batch] if wdef.seqlens is not None else None)
    inp = W.make_inputs(wdef, seed=rank_seed(wname, rank), device=device)
    a = algorithmic(inp)
    step = DecodeStep(inp, device)
    graphs = step.capture()
    for _ in range(args.warmup):
        step.replay_step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    # inputs smaller than L2 (reduced-batch profiling runs): L2 is flushed before each timed step
    flush = L2Flush(device) if a["bytes"] < L2_BYTES else None
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        if flush is None:
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record()
            for _ in range(args.steps):
                step.replay_step()
            t1.record()
            torch.cuda.synchronize()
            local_ms = t0.elapsed_time(t1)
        else:
            local_ms = sum(time_events(step.replay_step, args.steps, flush=flush))
    if world > 1:
        torch.distributed.barrier()
    total_ms = max_over_ranks(local_ms, device)
    ms = total_ms / args.steps
    flags = mla.device_status()
    value = job_throughput(a["bytes"], world, ms) / 1e9  # GB/s over all ranks

    # ---- dominant kernel: decode call (split-KV kernel + combine), same workload: median of >= 50
    step.metadata()
    dts = time_events(step.replay_decode, max(50, args.steps), flush=flush)
    dec_ms = statistics.median(dts)
    wl = inp.workload
    if wname in ("dense_membound", "tiny", "dense_membound_fp8"):
        roof = {"bound": "hbm", "achieved": round(a["bytes"] / (dec_ms * 1e-3) / 1e9, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": round(a["flops"] / (dec_ms * 1e-3) / 1e12, 2),
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    roof["traffic"] = measured_traffic(wname)
    roof["algorithmic_bytes"] = a["bytes"] if roof["bound"] == "hbm" else None
    roof["kernel"] = kernel_name(wl) + " + combine (one decode call)"
    roof["peak_source"] = peaks["source"]

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16 q/KV, random page permutation)",
        "config": {"workload": wname, "batch": wl.batch, "h_q": wl.h_q, "s_q": wl.s_q,
                   "seqlens": W.describe_lengths(wl), "page_size": 64,
                   "mode": ("dense fp8 cache" if wl.is_fp8 else "dense bf16 cache") if wl.mode == "dense"
                           else f"sparse top-{wl.topk} fp8 cache",
                   "parallelism": f"replicas x{world}",
                   "l2": ("inputs larger than L2 (%.0f MB > 129 MB), no flush" % (a["bytes"] / 1e6)) if flush is None
                         else ("L2 flushed before each timed step (inputs %.0f MB < 129 MB)" % (a["bytes"] / 1e6)),
                   "step_launch": "CUDA graph of schedule + decode + combine" if graphs else "eager calls"},
        "tflops": round(a["flops"] * world / (ms * 1e-3) / 1e12, 2),
        "roofline": roof,
        "gpu_launches": 3 * args.steps,
        "device_status": flags,
        "clocks": clk.summary(),
    }
    del step
    torch.cuda.empty_cache()

    if rank == 0 and world == 1 and not args.no_extras and wname == HEADLINE:
        # ---- end to end through the public API with host buffers: every input (the whole KV
        # cache included) copied in each step, and beside it the same with the cache resident
        for key, resident in (("e2e", False), ("e2e_resident_cache", True)):
            estep, h2d, d2h = e2e_step_factory(inp, device, resident_cache=resident)
            for _ in range(3):
                estep()
            et = time_events(estep, max(5, min(args.steps, 20)))
            ems = statistics.median(et)
            result[key] = {"value": round(a["bytes"] / (ems * 1e-3) / 1e9, 1), "unit": "GB/s",
                           "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                           "ms_per_step": round(ems, 4),
                           "note": "KV cache resident in device memory; q, block table and lengths copied "
                                   "from pinned host memory each step, out and lse copied back" if resident else
                                   "inputs incl. the whole KV cache copied from pinned host memory each step"}
            del estep
            torch.cuda.empty_cache()
        # ---- the other workloads (kernel level)
        extra = {}
        for name in ("tiny", "dense_computebound", "sparse_fp8", "sparse_fp8_long", "dense_membound_fp8",
                     "sparse_bf16", "sparse_fp8_token"):
            winp, wa, wms, st = measure_workload(name, device)
            bound = "hbm" if name in ("tiny", "dense_membound_fp8") else "tensor"
            e = {"ms": round(wms, 5), "tflops": round(wa["flops"] / (wms * 1e-3) / 1e12, 2),
                 "tflops_valid": round(wa["valid_flops"] / (wms * 1e-3) / 1e12, 2),
                 "kv_gbs": round(wa["bytes"] / (wms * 1e-3) / 1e9, 1)}
            if bound == "tensor":
                e["frac_of_bf16_peak"] = round(e["tflops"] / peaks["bf16_tflops"], 4)
            else:
                e["frac_of_hbm"] = round(e["kv_gbs"] / peaks["hbm_gbs"], 4)
            e["cpu_oracle"] = oracle_decode_rate(winp)
            extra[name] = e
            del st, winp
            torch.cuda.empty_cache()
        extra["fp8_cache_store"] = measure_store(device, peaks)
        extra["fp8_cache_store"]["cpu_oracle"] = oracle_store_rate()
        extra["sparse_prefill"] = measure_prefill(device, peaks)
        extra["sparse_prefill"]["cpu_oracle"] = oracle_prefill_rate(W.make_prefill_inputs("sparse_prefill"))
        extra["fp8_index_topk"] = measure_index(device, peaks)
        extra["fp8_index_topk"]["cpu_oracle"] = oracle_index_rate(W.make_index_inputs("index_decode"))
        result["workloads"] = extra
        # ---- the oracle on the host cores, bounded sample
        result["cpu_baseline"] = cpu_baseline(inp, target_s=args.cpu_seconds)
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


# ----------------------------------------------------------------------------
# the oracle (CPU baseline / reference arm)
# ----------------------------------------------------------------------------
def _oracle_sample(inp_cpu, n_elems):
    """Oracle decode of the first n_elems batch elements; returns (seconds, kv bytes processed)."""
    import oracle
    w = inp_cpu.workload
    rows_per = w.s_q * w.h_q
    rows = np.arange(n_elems * rows_per, dtype=np.int64)
    t = time.perf_counter()
    oracle.mla_decode(inp_cpu.q, inp_cpu.kvcache, inp_cpu.block_table, inp_cpu.cache_seqlens, inp_cpu.sm_scale,
                      is_causal=w.causal, indices=inp_cpu.indices, rows=rows)
    dt = time.perf_counter() - t
    lens = inp_cpu.cache_seqlens[:n_elems].numpy().astype(np.int64)
    kv = int(lens.sum()) * D_QK * 2 + n_elems * rows_per * (D_QK * 2 + D_V * 2 + 4)
    return dt, kv


def cpu_baseline(inp, target_s=15.0):
    """The oracle on the host cores over a bounded sample: the first n batch elements, repeated
    until about target_s seconds of work (the whole batch is one sample when it is shorter)."""
    import oracle
    oracle.build()
    cpu = inp.to("cpu")
    dt1, _ = _oracle_sample(cpu, 1)
    n = max(1, min(cpu.workload.batch, int(target_s / max(dt1, 1e-3))))
    total_t, total_kv, reps = 0.0, 0, 0
    while total_t < target_s and reps < 1000:
        dt, kv = _oracle_sample(cpu, n)
        total_t += dt
        total_kv += kv
        reps += 1
    return {"value": round(total_kv / total_t / 1e9, 4), "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"first {n} of {cpu.workload.batch} batch elements (all heads) of {HEADLINE}, x{reps}, "
                      f"{total_t:.1f} s, fp64, {os.cpu_count()} threads"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    inp = W.make_inputs(HEADLINE)
    a = algorithmic(inp)
    # size one step to about 2 s of CPU work, capped so the whole run stays within minutes
    dt1, _ = _oracle_sample(inp, 1)
    per_step = min(2.0, 150.0 / max(1, args.steps + args.warmup))
    n = max(1, min(inp.workload.batch, int(per_step / max(dt1, 1e-3))))
    for _ in range(args.warmup):
        _oracle_sample(inp, n)
    times, kvs = [], []
    for _ in range(args.steps):
        dt, kv = _oracle_sample(inp, n)
        times.append(dt)
        kvs.append(kv)
    ms = 1e3 * sum(times) / len(times)
    value = sum(kvs) / sum(times) / 1e9
    sample = f"first {n} of {inp.workload.batch} batch elements (all heads) per step, fp64, {os.cpu_count()} threads"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": HEADLINE, "batch": inp.workload.batch, "h_q": inp.workload.h_q,
                   "s_q": inp.workload.s_q, "page_size": 64, "mode": "dense bf16 cache"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "algorithmic_bytes_full_step": a["bytes"],
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["mla", "reference"], default="mla")
    ap.add_argument("--no-extras", action="store_true", help="headline workload only")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(W.WORKLOADS),
                    help="workload timed as the step (default: the memory-bound dense mix)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--batch", type=int, default=0,
                    help="run the workload with this batch size instead of its own (profiler captures of a "
                         "reduced case; implies --no-extras)")
    ap.add_argument("--extra", choices=["sparse_prefill", "fp8_index_topk", "fp8_cache_store"],
                    help="time only this entry point (one JSON line; used for profiling captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.batch:
        args.no_extras = True
    if args.extra:
        device = "cuda"
        peaks = load_peaks()
        fn = {"sparse_prefill": measure_prefill, "fp8_index_topk": measure_index,
              "fp8_cache_store": measure_store}[args.extra]
        print(json.dumps({"extra": args.extra, **fn(device, peaks)}), flush=True)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_mla(args)


if __name__ == "__main__":
    main()
