"""Parity of the FP8 top-k indexer (mla_index_topk, through the C ABI) with the oracle.

Where floating point decides the selection, the two sides may legitimately
differ on keys whose scores lie within the kernel's rounding of each other,
so the unique parts are compared exactly and the rest is checked for
validity: per query row the number of selected keys and the -1 fill are
exact, every id is a distinct visible key, no unselected visible key scores
above a selected one, and the order is descending — each comparison on the
oracle's fp64 scores, widened by a bound on the kernel's fp32 error.

Error bound: the kernel's head dot sums 128 exact E4M3 products in fp32 and
then multiplies by two scales, applies f and accumulates h weighted terms in
fp32; the rounding is at most (128 + h + 4) * 2^-24 of
A = sum_h |w_h| qs_h ks sum_d |q_hd k_d|.  The tests allow 2^-14 * A
(about 8x that figure for h <= 256).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_mla_decode_07_gb300 as mla
from paged_mla_decode_07_gb300 import workloads as W

from gpu_helpers import Guarded, check_guards, compare, guarded_tensor, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mla.build()
    mla.lib()


def decode_e4m3(codes):
    return codes.contiguous().view(torch.float8_e4m3fn).to(torch.float64).numpy()


def abs_bound(inp, width):
    """A[t, s] = sum_h |w| qs ks sum_d |q k| for visible keys (numpy, fp64)."""
    q = np.abs(decode_e4m3(inp.q_codes))
    kflat = inp.k_codes.reshape(-1, 128)
    qs = inp.q_scales.double().numpy()
    ks = inp.k_scales.reshape(-1).double().numpy()
    w = np.abs(inp.weights.double().numpy())
    offs = inp.row_offsets.numpy()
    lens = inp.cache_seqlens.numpy()
    table = inp.block_table.numpy()
    A = np.zeros((offs[-1], width))
    for b in range(len(lens)):
        L = int(lens[b])
        if L <= 0 or offs[b + 1] == offs[b]:
            continue
        s = np.arange(L)
        rows = table[b, s // 64].astype(np.int64) * 64 + s % 64
        k = np.abs(decode_e4m3(kflat[torch.from_numpy(rows)]))
        for t in range(offs[b], offs[b + 1]):
            A[t, :L] = (w[t] * qs[t]) @ (q[t] @ k.T) * ks[rows]
    return A


def run_index(inp):
    """Indexer into guarded ids / workspace buffers (guards checked after the call)."""
    d = inp.to("cuda")
    T = int(inp.row_offsets[-1])
    g_idx, idx = guarded_tensor((T, inp.topk), torch.int32)
    g_ws = Guarded(max(16, mla.index_topk_workspace_size(T, d.block_table.shape[1])))
    out = mla.index_topk(d.q_codes, d.q_scales, d.weights, d.row_offsets, d.k_codes, d.k_scales, d.block_table,
                         d.cache_seqlens, inp.topk, relu=inp.relu, indices=idx, workspace=g_ws.body)
    flags = mla.device_status()
    check_guards({"indices": g_idx, "workspace": g_ws}, inp.workload.name)
    return out.cpu().numpy(), flags


def check_selection(idx, inp):
    lens = inp.cache_seqlens.numpy()
    offs = inp.row_offsets.numpy()
    width = int(max(1, lens.max()))
    sigma = oracle.index_scores(inp, width=width)
    eps = 2.0 ** -14 * abs_bound(inp, width)
    k = inp.topk
    for b in range(len(lens)):
        n_b = offs[b + 1] - offs[b]
        for j in range(n_b):
            t = offs[b] + j
            vis = max(0, min(int(lens[b]) - n_b + j + 1, int(lens[b])))
            row = idx[t]
            n_sel = min(k, vis)
            assert np.all(row[n_sel:] == -1), f"row {t}: -1 fill"
            sel = row[:n_sel]
            assert np.all((sel >= 0) & (sel < vis)), f"row {t}: id outside the visible keys"
            assert len(np.unique(sel)) == n_sel, f"row {t}: repeated id"
            if n_sel == 0:
                continue
            s, e = sigma[t], eps[t]
            rest = np.setdiff1d(np.arange(vis), sel)
            if rest.size:
                assert np.min(s[sel] + e[sel]) >= np.max(s[rest] - e[rest]), f"row {t}: a better key was left out"
            assert np.all(s[sel[:-1]] + e[sel[:-1]] >= s[sel[1:]] - e[sel[1:]]), f"row {t}: not in descending order"


@pytest.mark.parametrize("relu", [False, True])
def test_index_tiny(relu):
    inp = W.make_index_inputs(W.IndexWorkload("it", batch=2, n_new=2, h_idx=8, topk=64, seqlens=(300, 90),
                                              relu=relu), seed=3)
    idx, flags = run_index(inp)
    assert flags == 0
    check_selection(idx, inp)


@pytest.mark.parametrize("h_idx,rows", [(8, (1, 5, 2)), (32, (3, 1, 8)), (64, (4, 1, 2)), (128, (2, 2, 1)),
                                        (256, (1, 1, 1))])
def test_index_heads_and_ragged_rows(h_idx, rows):
    w = W.IndexWorkload(f"ih{h_idx}", batch=3, n_new=1, h_idx=h_idx, topk=200, seqlens=(1000, 130, 2500),
                        rows=rows, relu=h_idx % 64 == 0)
    inp = W.make_index_inputs(w, seed=h_idx)
    idx, flags = run_index(inp)
    assert flags == 0
    check_selection(idx, inp)


def test_index_fewer_visible_keys_than_k():
    inp = W.make_index_inputs(W.IndexWorkload("ifew", batch=3, n_new=3, h_idx=16, topk=300, seqlens=(5, 290, 64)),
                              seed=8)
    idx, flags = run_index(inp)
    assert flags == 0
    check_selection(idx, inp)
    assert np.all(idx[0, 3:] == -1) and sorted(idx[0, :3].tolist()) == [0, 1, 2]   # 5 keys, first row sees 3


def test_index_equal_scores_take_smallest_ids():
    inp = W.make_index_inputs(W.IndexWorkload("ieq", batch=1, n_new=1, h_idx=16, topk=50, seqlens=(700,)), seed=2)
    inp.k_codes[:] = inp.k_codes[0, 0]
    inp.k_scales[:] = 0.25
    idx, _ = run_index(inp)
    np.testing.assert_array_equal(idx[0], np.arange(50))


def test_index_long_rows_and_many_tiles():
    w = W.IndexWorkload("ilong", batch=2, n_new=2, h_idx=64, topk=2048, seqlens=(40000, 9000))
    inp = W.make_index_inputs(w, seed=21)
    idx, flags = run_index(inp)
    assert flags == 0
    check_selection(idx, inp)


def test_index_runs_cross_many_short_elements():
    """More elements than SMs, short and ragged: the score kernel's per-CTA runs of the tile line
    cross several elements each, among them elements without query rows or without keys (no tiles)."""
    rng = np.random.default_rng(77)
    batch = 300
    lens = tuple(0 if i % 37 == 5 else int(x) for i, x in enumerate(rng.integers(1, 700, size=batch)))
    rows = tuple(0 if i % 23 == 7 else 1 + i % 2 for i in range(batch))
    w = W.IndexWorkload("ishort", batch=batch, n_new=2, h_idx=32, topk=100, seqlens=lens, rows=rows, relu=True)
    inp = W.make_index_inputs(w, seed=77)
    idx, flags = run_index(inp)
    assert flags == 0
    check_selection(idx, inp)


def test_index_bad_page_is_flagged_and_never_selected():
    w = W.IndexWorkload("ibad", batch=2, n_new=1, h_idx=16, topk=400, seqlens=(300, 200))
    inp = W.make_index_inputs(w, seed=4)
    bt = inp.block_table.clone()
    bt[0, 1] = inp.k_codes.shape[0] + 3              # keys 64..127 of element 0 sit on no page
    inp.block_table = bt
    idx, flags = run_index(inp)
    assert flags & mla.DEVICE_BAD_PAGE
    sel = idx[0][idx[0] >= 0]
    assert len(sel) == 300 - 64 and not np.any((sel >= 64) & (sel < 128))


def test_index_full_size_sampled_elements():
    """The benchmark's indexer workload at full size; the oracle checks three elements."""
    inp = W.make_index_inputs("index_decode")
    idx, flags = run_index(inp)
    assert flags == 0
    w = inp.workload
    for b in (0, 57, w.batch - 1):
        r0, r1 = int(inp.row_offsets[b]), int(inp.row_offsets[b + 1])
        sub = W.IndexInputs(w, inp.q_codes[r0:r1], inp.q_scales[r0:r1], inp.weights[r0:r1],
                            torch.tensor([0, r1 - r0], dtype=torch.int32), inp.k_codes, inp.k_scales,
                            inp.block_table[b:b + 1], inp.cache_seqlens[b:b + 1], w.topk, w.relu, inp.seed)
        check_selection(idx[r0:r1], sub)


def test_indexer_feeds_sparse_decode():
    """Indexer output as the indices of sparse FP8 decode over the same elements."""
    iw = W.IndexWorkload("ifeed", batch=3, n_new=2, h_idx=64, topk=256, seqlens=(3000, 900, 5000))
    iinp = W.make_index_inputs(iw, seed=5)
    idx, flags = run_index(iinp)
    assert flags == 0
    dw = W.custom(name="fed", batch=3, h_q=64, s_q=2, mode="sparse", seqlens=(3000, 900, 5000), topk=256)
    dinp = W.make_inputs(dw, seed=6)
    dinp.indices = torch.from_numpy(idx.reshape(3, 2, 256).copy())
    d = dinp.to("cuda")
    sched, ns = mla.get_metadata(d.cache_seqlens, h_q=64, s_q=2, topk=256, is_fp8=True)
    out, lse = mla.decode(d.q, d.kvcache, d.block_table, d.cache_seqlens, d.sm_scale, sched, ns, indices=d.indices)
    assert mla.device_status() == 0
    ref_out, ref_lse = run_oracle(dinp)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out, ref_lse, "indexer->decode")


@pytest.mark.parametrize("L", [12000, 20000])
def test_index_largest_topk(L):
    """top-k 16384 (the largest supported): every visible key when there are fewer, else a selection."""
    w = W.IndexWorkload(f"imax{L}", batch=1, n_new=1, h_idx=16, topk=16384, seqlens=(L,))
    inp = W.make_index_inputs(w, seed=L)
    idx, flags = run_index(inp)
    assert flags == 0
    check_selection(idx, inp)
