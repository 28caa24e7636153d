"""Shared helpers for the GPU tests: run the CUDA path through the binding and
compare it with the oracle at the acceptance tolerance."""
import contextlib
import os

import numpy as np
import torch

import oracle
import paged_mla_decode_07_gb300 as mla

# Acceptance bar for floating point: max|out - oracle| <= 1e-2 * max|oracle| + 2e-3,
# |lse - oracle| <= 1e-3 on finite entries, infinities equal.
OUT_RTOL = 1e-2
OUT_ATOL = 2e-3
LSE_ATOL = 1e-3


@contextlib.contextmanager
def env(**kw):
    old = {k: os.environ.get(k) for k in kw}
    try:
        for k, v in kw.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = str(v)
        yield
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def run_cuda(inp, device="cuda"):
    """Decode ``inp`` on the GPU; returns (out float64 [b,s_q,h_q,512], lse float64, status flags)."""
    w = inp.workload
    d = inp.to(device)
    topk = 0 if d.indices is None else d.indices.shape[-1]
    sched, ns = mla.get_metadata(d.cache_seqlens, w.s_q, w.h_q, topk)
    out, lse = mla.decode(d.q, d.kvcache, d.block_table, d.cache_seqlens, d.sm_scale, sched, ns,
                          is_causal=w.causal, indices=d.indices, kv_scales=d.kv_scales,
                          topk_lengths=d.topk_lengths)
    flags = mla.device_status()
    return out.double().cpu().numpy(), lse.double().cpu().numpy(), flags


def run_oracle(inp, rows=None):
    return oracle.mla_decode(inp.q, inp.kvcache, inp.block_table, inp.cache_seqlens, inp.sm_scale,
                             is_causal=inp.workload.causal, indices=inp.indices, rows=rows,
                             kv_scales=inp.kv_scales, topk_lengths=inp.topk_lengths)


def compare(out, lse, ref_out, ref_lse, what=""):
    out = np.asarray(out, np.float64).reshape(-1, 512)
    ref_out = np.asarray(ref_out, np.float64).reshape(-1, 512)
    lse = np.asarray(lse, np.float64).reshape(-1)
    ref_lse = np.asarray(ref_lse, np.float64).reshape(-1)
    assert np.all(np.isfinite(out)), f"{what}: non-finite output"
    scale = float(np.max(np.abs(ref_out))) if ref_out.size else 0.0
    err = float(np.max(np.abs(out - ref_out))) if out.size else 0.0
    assert err <= OUT_RTOL * scale + OUT_ATOL, f"{what}: max|out-ref| = {err:.3e} (max|ref| = {scale:.3e})"
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin), f"{what}: lse finiteness differs"
    assert np.array_equal(lse[~fin], ref_lse[~fin]), f"{what}: lse infinities differ"
    if fin.any():
        lerr = float(np.max(np.abs(lse[fin] - ref_lse[fin])))
        assert lerr <= LSE_ATOL, f"{what}: max|lse-ref| = {lerr:.3e}"
    return err, scale
