"""mla_decode_noalloc: decode for callers that cannot allocate device memory.

Some callers cannot obtain GPU memory at the moment they decode — code running
inside a host runtime or plugin that owns no CUDA memory pool, or a
latency-critical path where a cudaMalloc (which may synchronise the device) is
not allowed.  mla_decode_noalloc serves them: its split-KV scratch is a fixed
array inside the library instead of a caller workspace.  These tests call it
through the C ABI twice in a row and check each result against the allocating
entry point, mla_decode, at the tolerance the parity tests use.

This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_mla_decode_07_gb300 as mla
from paged_mla_decode_07_gb300 import workloads as W

from gpu_helpers import compare, metadata

pytestmark = pytest.mark.gpu

MLA_ERR_WORKSPACE = 3


def _lib():
    L = mla.lib()
    L.mla_decode_noalloc.argtypes = [ctypes.POINTER(mla.DecodeArgs), ctypes.c_void_p]
    L.mla_decode_noalloc.restype = ctypes.c_int
    return L


def _args(d, sched, ns, out, lse):
    w = d.workload
    a = mla.DecodeArgs()
    a.q = d.q.data_ptr()
    a.batch, a.s_q, a.h_q = w.batch, w.s_q, w.h_q
    a.kvcache = d.kvcache.data_ptr()
    a.num_pages, a.page_size = d.kvcache.shape[0], d.kvcache.shape[1]
    a.block_table = d.block_table.data_ptr()
    a.block_table_stride = d.block_table.shape[1]
    a.cache_seqlens = d.cache_seqlens.data_ptr()
    a.sm_scale = d.sm_scale
    a.is_causal = int(w.causal)
    a.is_fp8 = int(d.kvcache.dtype == torch.uint8)
    a.indices = d.indices.data_ptr() if d.indices is not None else None
    a.topk = 0 if d.indices is None else d.indices.shape[-1]
    a.sched = sched.data_ptr()
    a.num_splits = ns.data_ptr()
    a.workspace = None
    a.workspace_bytes = 0
    a.out = out.data_ptr()
    a.lse = lse.data_ptr()
    return a


CASES = {
    "dense_membound": lambda: W.make_inputs("dense_membound"),
    "sparse_split": lambda: W.make_inputs(W.custom(name="na_sparse", batch=3, h_q=128, s_q=2, mode="sparse",
                                                   seqlens=(5000, 3000, 700), topk=640), seed=77),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_noalloc_matches_the_allocating_entry_point_on_two_calls(name):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mla.build()
    L = _lib()
    d = CASES[name]().to("cuda")
    w = d.workload
    sched, ns = metadata(d, w)
    ref_out, ref_lse = mla.decode(d.q, d.kvcache, d.block_table, d.cache_seqlens, d.sm_scale, sched, ns,
                                  is_causal=w.causal, indices=d.indices)
    ref_out = ref_out.double().cpu().numpy()
    ref_lse = ref_lse.double().cpu().numpy()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        out = torch.full((w.batch, w.s_q, w.h_q, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((w.batch, w.s_q, w.h_q), float("nan"), dtype=torch.float32, device="cuda")
        a = _args(d, sched, ns, out, lse)
        st = L.mla_decode_noalloc(ctypes.byref(a), stream)
        assert st == 0, mla.last_error()
        assert mla.device_status() == 0
        compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out, ref_lse,
                f"{name} no-alloc call {call + 1}")


def test_noalloc_rejects_scratch_beyond_its_fixed_size():
    """A decode whose split-KV scratch exceeds the fixed array is refused before any launch: the
    call gets real buffers of a small decode (so nothing could go wrong even if it launched) with
    the large configuration's sizes, returns MLA_ERR_WORKSPACE and leaves the outputs untouched."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mla.build()
    L = _lib()
    w = W.WORKLOADS["sparse_fp8"]  # its split-KV scratch exceeds the fixed 32 MiB
    assert mla.workspace_size(w.batch, h_q=w.h_q, s_q=w.s_q, topk=w.topk, is_fp8=True) > 32 << 20
    small = W.make_inputs(W.custom(name="tiny_sparse", batch=2, h_q=16, s_q=1, mode="sparse", seqlens=(100, 50),
                                   topk=64), seed=3).to("cuda")
    sched, ns = metadata(small, small.workload)
    out = torch.full((2, 1, 16, 512), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((2, 1, 16), 7.0, dtype=torch.float32, device="cuda")
    a = _args(small, sched, ns, out, lse)
    a.batch, a.s_q, a.h_q, a.topk = w.batch, w.s_q, w.h_q, w.topk
    st = L.mla_decode_noalloc(ctypes.byref(a), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == MLA_ERR_WORKSPACE
    assert "32" in mla.last_error() or "33554432" in mla.last_error()
    assert "scratch" in mla.last_error()
    torch.cuda.synchronize()
    assert bool((out == 7.0).all()) and bool((lse == 7.0).all())
    assert mla.device_status() == 0
