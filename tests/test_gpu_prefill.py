"""Parity of sparse attention over bf16 rows with the fp64 oracle, through the C ABI:

* sparse decode over the paged bf16 cache (the mode variant beside sparse
  decode over the FP8 cache), against the decode oracle;
* sparse prefill (mla_sparse_prefill: unpaged KV, no batch), against the
  oracle's sparse prefill: every element on small cases, sampled rows at the
  benchmark's full size and across the 16384-token chunk boundary.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_mla_decode_07_gb300 as mla
from paged_mla_decode_07_gb300 import workloads as W

from gpu_helpers import Guarded, check_guards, compare, guarded_tensor, metadata, overrides, run_cuda, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mla.build()
    mla.lib()


# ---------------------------------------------------------------- sparse decode over the bf16 cache
@pytest.mark.parametrize("h_q", [16, 32, 64, 128])
def test_sparse_decode_over_bf16_cache(h_q):
    w = W.custom(name=f"sb{h_q}", batch=3, h_q=h_q, s_q=2, mode="sparse", fp8=False, seqlens=(700, 90, 4000),
                 topk=320)
    inp = W.make_inputs(w, seed=300 + h_q)
    idx = inp.indices.clone()
    idx[0, 0, 5] = idx[0, 0, 6]            # a repeated id counts twice
    idx[1, 1, 3] = 90                      # == seqlen: skipped
    idx[2, 0, :] = -1                      # no valid key: out 0, lse -inf
    inp.indices = idx
    out, lse, flags = run_cuda(inp)
    assert flags == 0, f"device status 0x{flags:x}"
    ref_out, ref_lse = run_oracle(inp)
    compare(out, lse, ref_out, ref_lse, w.name)
    assert np.all(out[2, 0] == 0) and np.all(lse[2, 0] == -np.inf)


def test_sparse_bf16_bad_page_skips_its_tokens():
    """A block-table entry outside the pool: flagged, and its tokens count as invalid ids."""
    w = W.custom(name="sbbad", batch=2, h_q=64, s_q=1, mode="sparse", fp8=False, seqlens=(700, 300), topk=256)
    inp = W.make_inputs(w, seed=5)
    good_table = inp.block_table
    bt = good_table.clone()
    bt[0, 3] = inp.kvcache.shape[0] + 7          # tokens 192..255 of element 0 sit on no page
    inp.block_table = bt
    out, lse, flags = run_cuda(inp)
    assert flags & mla.DEVICE_BAD_PAGE
    idx = inp.indices.clone()
    e0 = idx[0]
    e0[(e0 >= 192) & (e0 < 256)] = -1
    assert int(((inp.indices[0] >= 192) & (inp.indices[0] < 256)).sum()) > 0
    inp.indices = idx
    inp.block_table = good_table
    ref_out, ref_lse = run_oracle(inp)
    compare(out, lse, ref_out, ref_lse, w.name)


def test_sparse_bf16_and_fp8_caches_agree_on_dequantised_values():
    """The same keys as FP8 rows and as their dequantised bf16 values give the same result."""
    w = W.custom(name="sx", batch=2, h_q=64, s_q=1, mode="sparse", seqlens=(1500, 600), topk=256)
    inp = W.make_inputs(w, seed=77, poison_tail=False)
    out_f, lse_f, _ = run_cuda(inp)
    flat = inp.kvcache.reshape(-1, 656)
    n = flat.shape[0]
    codes = flat[:, :512].contiguous().view(torch.float8_e4m3fn).float().reshape(n, 4, 128)
    scales = flat[:, 512:528].contiguous().view(torch.float32).reshape(n, 4)
    nope = (codes * scales[:, :, None]).reshape(n, 512).to(torch.bfloat16)
    rope = flat[:, 528:].contiguous().view(torch.bfloat16)
    kvb = torch.cat([nope, rope], 1).reshape(inp.kvcache.shape[0], 64, 1, 576)
    inp_b = W.Inputs(W.with_fields(w, fp8=False), inp.q, kvb, inp.block_table, inp.cache_seqlens, inp.indices,
                     inp.sm_scale, inp.seed)
    out_b, lse_b, flags = run_cuda(inp_b)
    assert flags == 0
    compare(out_b, lse_b, out_f, lse_f, "bf16-vs-fp8 cache")


# ---------------------------------------------------------------- sparse prefill
def run_prefill(inp, rows=None):
    """Prefill into guarded out / lse / workspace buffers (guards checked after the call)."""
    d = inp.to("cuda")
    w = inp.workload
    g_out, out = guarded_tensor((w.s_q, w.h_q, 512), torch.bfloat16)
    g_lse, lse = guarded_tensor((w.s_q, w.h_q), torch.float32)
    g_ws = Guarded(mla.sparse_prefill_workspace_size(w.s_q, w.h_q, w.topk))
    out, lse = mla.sparse_prefill(d.q, d.kv, d.indices, d.sm_scale, out=out, lse=lse, workspace=g_ws.body)
    flags = mla.device_status()
    check_guards({"out": g_out, "lse": g_lse, "workspace": g_ws}, w.name)
    out = out.reshape(-1, 512)
    lse = lse.reshape(-1)
    if rows is not None:
        r = torch.as_tensor(rows, device="cuda")
        out, lse = out[r], lse[r]
    return out.double().cpu().numpy(), lse.double().cpu().numpy(), flags


def check_prefill(inp, rows=None):
    out, lse, flags = run_prefill(inp, rows)
    assert flags == 0, f"device status 0x{flags:x}"
    ref_out, ref_lse = oracle.sparse_prefill(inp.q, inp.kv, inp.indices, inp.sm_scale, rows=rows)
    compare(out, lse, ref_out, ref_lse, inp.workload.name)
    return out, lse


def test_prefill_tiny_workload():
    check_prefill(W.make_prefill_inputs("prefill_tiny"))


@pytest.mark.parametrize("h_q,topk,s_kv", [(8, 64, 100), (16, 1, 50), (32, 130, 3000), (64, 257, 1000),
                                           (128, 512, 5000), (96, 200, 700)])
def test_prefill_shapes(h_q, topk, s_kv):
    """16/32/64-row CTAs, two row groups, ghost rows (h_q 8, 96), a single key, a ragged last tile."""
    w = W.PrefillWorkload(f"p{h_q}_{topk}", s_q=37, s_kv=s_kv, h_q=h_q, topk=topk, invalid_frac=0.05)
    check_prefill(W.make_prefill_inputs(w, seed=h_q + topk))


def test_prefill_invalid_repeated_and_empty_rows():
    w = W.PrefillWorkload("p_edge", s_q=6, s_kv=333, h_q=64, topk=96)
    inp = W.make_prefill_inputs(w, seed=9)
    idx = inp.indices.clone()
    idx[0, :] = -1                        # no valid key
    idx[1, :] = 332                       # one key, 96 times
    idx[2, ::3] = 333                     # == s_kv: skipped
    idx[3, 10:20] = -5
    idx[4, :48] = idx[4, 48:]             # every key twice
    inp.indices = idx
    out, lse = check_prefill(inp)
    out = out.reshape(6, 64, 512)
    lse = lse.reshape(6, 64)
    assert np.all(out[0] == 0) and np.all(lse[0] == -np.inf)


def test_prefill_is_sparse_decode_on_one_element():
    """Prefill equals sparse decode over the same rows laid out as an identity-paged bf16 cache."""
    w = W.PrefillWorkload("p_vs_dec", s_q=20, s_kv=640, h_q=64, topk=200, invalid_frac=0.1)
    inp = W.make_prefill_inputs(w, seed=31)
    out_p, lse_p, _ = run_prefill(inp)
    d = inp.to("cuda")
    cache = d.kv.reshape(10, 64, 1, 576)
    table = torch.arange(10, dtype=torch.int32, device="cuda")[None]
    lens = torch.tensor([640], dtype=torch.int32, device="cuda")
    sched, ns = mla.get_metadata(lens, h_q=64, s_q=20, topk=200, is_fp8=False)
    out_d, lse_d = mla.decode(d.q[None], cache, table, lens, d.sm_scale, sched, ns, indices=d.indices[None])
    np.testing.assert_array_equal(out_p, out_d.reshape(-1, 512).double().cpu().numpy())
    np.testing.assert_array_equal(lse_p, lse_d.reshape(-1).double().cpu().numpy())


def test_prefill_full_size_sampled_rows():
    """The benchmark's prefill workload at full size, in its launch configuration."""
    inp = W.make_prefill_inputs("sparse_prefill")
    w = inp.workload
    rng = np.random.default_rng(5)
    n = w.s_q * w.h_q
    rows = np.unique(np.concatenate([rng.integers(0, n, 200), [0, n - 1, w.h_q - 1, n - w.h_q]]))
    check_prefill(inp, rows=rows)


def test_prefill_across_the_chunk_boundary():
    """More than 16384 query tokens: the library runs two chunks."""
    w = W.PrefillWorkload("p_chunks", s_q=16384 + 300, s_kv=2000, h_q=16, topk=64, invalid_frac=0.05)
    inp = W.make_prefill_inputs(w, seed=12)
    n = w.s_q * w.h_q
    rng = np.random.default_rng(2)
    rows = np.unique(np.concatenate([rng.integers(0, n, 150), np.arange(16380 * 16, 16390 * 16), [n - 1]]))
    check_prefill(inp, rows=rows)


def test_prefill_with_parts_forced_small_splits_problems():
    """Few parts: every part covers several query tokens and splits some; the combine merges them."""
    w = W.PrefillWorkload("p_split", s_q=9, s_kv=4000, h_q=64, topk=1024)
    inp = W.make_prefill_inputs(w, seed=4)
    with overrides(num_parts=7):
        check_prefill(inp)


def test_prefill_many_heads():
    """512 heads: eight row groups of 64 per query token."""
    w = W.PrefillWorkload("p512", s_q=7, s_kv=900, h_q=512, topk=130, invalid_frac=0.05)
    check_prefill(W.make_prefill_inputs(w, seed=512))
