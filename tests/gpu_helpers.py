"""Shared helpers for the GPU tests: run the CUDA path through the binding and
compare it with the oracle at the acceptance tolerance.

Every output and scratch buffer the helpers hand to the library sits between
two guard regions filled with a known byte pattern (canaries); after each call
the helpers assert that the pattern is intact, so a kernel that writes past
either end of a buffer fails the test even where the values it was meant to
write are right."""
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


GUARD_BYTES = 4096
GUARD_FILL = 0xA5


class Guarded:
    """A device buffer of ``nbytes`` between two GUARD_BYTES guard regions of GUARD_FILL bytes."""

    def __init__(self, nbytes, device="cuda"):
        self.nbytes = int(nbytes)
        self.buf = torch.full((GUARD_BYTES + self.nbytes + GUARD_BYTES,), GUARD_FILL, dtype=torch.uint8,
                              device=device)
        self.body = self.buf[GUARD_BYTES:GUARD_BYTES + self.nbytes]

    def view(self, dtype, shape):
        return self.body.view(dtype).view(shape)

    def check(self, what=""):
        head = self.buf[:GUARD_BYTES]
        tail = self.buf[GUARD_BYTES + self.nbytes:]
        bad_head = int((head != GUARD_FILL).sum().item())
        bad_tail = int((tail != GUARD_FILL).sum().item())
        assert bad_head == 0 and bad_tail == 0, (
            f"{what}: {bad_head} guard bytes before and {bad_tail} after the buffer were overwritten")


def guarded_tensor(shape, dtype, device="cuda"):
    n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    g = Guarded(n, device)
    return g, g.view(dtype, shape)


def check_guards(guards, what=""):
    torch.cuda.synchronize()
    for name, g in guards.items():
        g.check(f"{what} {name}")


@contextlib.contextmanager
def overrides(num_parts=None, debug_stall=False):
    """The library's test hooks for the duration of a block: a forced part count, a stalled
    softmax role."""
    mla.set_test_hooks(int(num_parts or 0), bool(debug_stall))
    try:
        yield
    finally:
        mla.set_test_hooks(0, False)


def metadata(d, w):
    """Schedule for inputs ``d`` (on the device) of workload ``w``."""
    topk = 0 if d.indices is None else d.indices.shape[-1]
    return mla.get_metadata(d.cache_seqlens, h_q=w.h_q, s_q=w.s_q, topk=topk,
                            is_fp8=d.kvcache.dtype == torch.uint8)


def run_cuda(inp, device="cuda"):
    """Decode ``inp`` on the GPU into guarded out / lse / workspace buffers; returns (out float64
    [b,s_q,h_q,512], lse float64, status flags) after checking every guard region."""
    w = inp.workload
    d = inp.to(device)
    topk = 0 if d.indices is None else d.indices.shape[-1]
    is_fp8 = d.kvcache.dtype == torch.uint8
    sched, ns = metadata(d, w)
    g_out, out = guarded_tensor((w.batch, w.s_q, w.h_q, 512), torch.bfloat16, device)
    g_lse, lse = guarded_tensor((w.batch, w.s_q, w.h_q), torch.float32, device)
    g_ws = Guarded(max(256, mla.workspace_size(w.batch, h_q=w.h_q, s_q=w.s_q, topk=topk, is_fp8=is_fp8)), device)
    out, lse = mla.decode(d.q, d.kvcache, d.block_table, d.cache_seqlens, d.sm_scale, sched, ns,
                          is_causal=w.causal, indices=d.indices, kv_scales=d.kv_scales,
                          topk_lengths=d.topk_lengths, out=out, lse=lse, workspace=g_ws.body)
    flags = mla.device_status()
    check_guards({"out": g_out, "lse": g_lse, "workspace": g_ws}, w.name)
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
