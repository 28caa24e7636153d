"""Parity of the CUDA decode path (through the C ABI) with the fp64 oracle.

Small cases and the named workloads at full size (in the benchmark's launch
configuration) compare every output element with the oracle run over all
rows; whole-output properties are checked beside them.  Every output and
scratch buffer sits between guard regions that must survive each call.
"""
import math

import numpy as np
import pytest
import torch

import paged_mla_decode_07_gb300 as mla
from paged_mla_decode_07_gb300 import workloads as W

from gpu_helpers import compare, metadata, overrides, run_cuda, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mla.build()
    mla.lib()


def check(w, seed, parts=None, poison=True, **mk):
    inp = W.make_inputs(w, seed=seed, poison_tail=poison, **mk)
    with overrides(num_parts=parts):
        out, lse, flags = run_cuda(inp)
    ref_out, ref_lse = run_oracle(inp)
    assert flags == 0, f"device status 0x{flags:x}"
    compare(out, lse, ref_out, ref_lse, w.name)
    return out, lse, ref_out, ref_lse


# ---------------------------------------------------------------- dense mode
def test_tiny_workload():
    check(W.WORKLOADS["tiny"], W.SEEDS["tiny"])


@pytest.mark.parametrize("L", [1, 2, 63, 64, 65, 127, 128, 129, 255, 256, 300, 1000])
def test_dense_lengths(L):
    check(W.custom(name=f"len{L}", batch=2, h_q=16, s_q=1, mode="dense", seqlens=(L, max(1, L // 3))), 10 + L)


@pytest.mark.parametrize("h_q,s_q", [(16, 1), (8, 1), (32, 1), (24, 1), (64, 1), (48, 1), (128, 1),
                                     (128, 2), (16, 4), (40, 3)])
def test_dense_row_shapes(h_q, s_q):
    """rows per problem = s_q*h_q covers 16/32/64-row CTAs, several row groups and ghost rows."""
    check(W.custom(name=f"h{h_q}s{s_q}", batch=3, h_q=h_q, s_q=s_q, mode="dense", seqlens=(200, 77, 513)),
          100 + h_q + s_q)


@pytest.mark.parametrize("s_q", [1, 2, 3])
def test_dense_causal(s_q):
    check(W.custom(name=f"causal{s_q}", batch=3, h_q=64, s_q=s_q, mode="dense", seqlens=(129, 64, 1),
                   causal=True), 200 + s_q)


def test_dense_empty_and_single():
    w = W.custom(name="empty", batch=4, h_q=16, s_q=1, mode="dense", seqlens=(0, 1, 0, 70))
    out, lse, _, _ = check(w, 7)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(out[2] == 0) and np.all(np.isneginf(lse[2]))


@pytest.mark.parametrize("parts", [1, 2, 3, 7, 40, 152, 400])
def test_forced_split_counts(parts):
    """Any partition of the tile line (1 part .. more parts than tiles) gives the same answer."""
    w = W.custom(name=f"parts{parts}", batch=5, h_q=64, s_q=2, mode="dense",
                 seqlens=(1000, 130, 1, 700, 2049), causal=True)
    check(w, 300, parts=parts)


def test_rescale_path_large_logits():
    """Large sm_scale: the running max grows by far more than the lazy-rescale threshold."""
    check(W.custom(name="bigscale", batch=2, h_q=64, s_q=1, mode="dense", seqlens=(1500, 800), sm_scale=0.6),
          11)


def test_rescale_path_increasing_logits():
    """Logits that grow along the sequence force an O rescale on every tile.

    Key j is pushed along head 0's query direction by 0.15*j*24/|q|, so head 0's logit grows by
    about 9.6 (13.9 in log2 units, above the threshold of 8) per 64-token tile and ends near 165:
    large enough to exercise the rescale, small enough for fp32 accumulation to meet the
    absolute lse bound."""
    w = W.custom(name="ramp", batch=1, h_q=32, s_q=1, mode="dense", seqlens=(1100,))
    inp = W.make_inputs(w, seed=12)
    q = inp.q.float()
    qn = q[0, 0, 0].norm()
    unit = q[0, 0, 0] / qn
    kv = inp.kvcache.float()
    for j in range(1100):
        page, slot = int(inp.block_table[0, j // 64]), j % 64
        kv[page, slot, 0] = kv[page, slot, 0] * 0.1 + unit * (0.15 * j * 24.0 / qn)
    inp.kvcache = kv.to(torch.bfloat16)
    with overrides(num_parts=1):
        out, lse, flags = run_cuda(inp)
    ref_out, ref_lse = run_oracle(inp)
    assert flags == 0
    compare(out, lse, ref_out, ref_lse, "ramp")


# ---------------------------------------------------------------- CTA-pair kernel (more than 64 rows, bf16 cache)
@pytest.mark.parametrize("L", [1, 63, 64, 65, 127, 128, 129, 200, 256, 257, 1000])
def test_pair_lengths(L):
    """128-token tiles of two pages: a tile whose second page holds no token, ragged last pages."""
    check(W.custom(name=f"pl{L}", batch=2, h_q=128, s_q=1, mode="dense", seqlens=(L, max(1, L // 3))), 1500 + L)


@pytest.mark.parametrize("h_q,s_q", [(96, 1), (80, 2), (128, 3), (65, 1), (256, 1)])
def test_pair_row_shapes(h_q, s_q):
    """Ghost rows in the odd CTA or the second pair, several pairs per problem."""
    check(W.custom(name=f"ph{h_q}s{s_q}", batch=3, h_q=h_q, s_q=s_q, mode="dense", seqlens=(300, 77, 700)),
          1600 + h_q + s_q)


@pytest.mark.parametrize("parts", [1, 3, 38, 200])
def test_pair_forced_splits_causal(parts):
    w = W.custom(name=f"pp{parts}", batch=4, h_q=128, s_q=2, mode="dense", seqlens=(1000, 0, 130, 2049),
                 causal=True)
    out, lse, _, _ = check(w, 1700 + parts, parts=parts)
    assert np.all(out[1] == 0) and np.all(np.isneginf(lse[1]))


def test_pair_bad_page_is_flagged_not_faulted():
    w = W.custom(name="pbad", batch=2, h_q=128, s_q=1, mode="dense", seqlens=(300, 100))
    inp = W.make_inputs(w, seed=19)
    bt = inp.block_table.clone()
    bt[0, 1] = inp.kvcache.shape[0] + 9   # the odd CTA's page of tile 0
    bt[0, 2] = -3                         # the even CTA's page of tile 1
    inp.block_table = bt
    out, lse, flags = run_cuda(inp)
    assert flags & mla.DEVICE_BAD_PAGE
    assert np.all(np.isfinite(out))


def test_pair_rescale_path():
    """A large scale makes later tiles raise the running max by far more than the threshold."""
    check(W.custom(name="pbig", batch=2, h_q=128, s_q=1, mode="dense", seqlens=(1500, 800), sm_scale=0.6), 1801,
          parts=1)


@pytest.mark.parametrize("fp8", [True, False], ids=["fp8", "bf16"])
@pytest.mark.parametrize("h_q,topk", [(128, 64), (128, 127), (128, 129), (128, 640), (96, 200), (256, 300)])
def test_pair_sparse_shapes(h_q, topk, fp8):
    """Sparse decode on CTA pairs over FP8 or bf16 rows: 128-slot tiles (a partial last tile, a
    single one), ghost rows, two pairs per query token."""
    check(W.custom(name=f"ps{h_q}_{topk}", batch=2, h_q=h_q, s_q=2, mode="sparse", fp8=fp8, seqlens=(3000, 700),
                   topk=topk), 1900 + h_q + topk)


@pytest.mark.parametrize("fp8", [True, False], ids=["fp8", "bf16"])
def test_pair_sparse_duplicates_invalid_and_bad_pages(fp8):
    w = W.custom(name="psdup", batch=2, h_q=128, s_q=2, mode="sparse", fp8=fp8, seqlens=(300, 900), topk=256)
    inp = W.make_inputs(w, seed=23)
    idx = inp.indices.clone()
    idx[0, 0, :40] = 7           # one id forty times
    idx[0, 1, 70] = 300          # == seqlen: skipped
    idx[1, 0, 130] = 10 ** 7     # far out of range: skipped
    idx[1, 1, :] = -1            # empty key set
    inp.indices = idx
    out, lse, flags = run_cuda(inp)
    ref_out, ref_lse = run_oracle(inp)
    assert flags == 0
    compare(out, lse, ref_out, ref_lse, "psdup")
    assert np.all(out[1, 1] == 0) and np.all(np.isneginf(lse[1, 1]))
    # a page outside the pool: flagged, its tokens count as invalid ids
    bt = inp.block_table.clone()
    bt[1, 2] = inp.kvcache.shape[0] + 3
    inp.block_table = bt
    out, lse, flags = run_cuda(inp)
    assert flags & mla.DEVICE_BAD_PAGE
    idx2 = inp.indices.clone()
    e1 = idx2[1]
    e1[(e1 >= 128) & (e1 < 192)] = -1
    inp.indices = idx2
    ref_out, ref_lse = run_oracle(inp)
    compare(out, lse, ref_out, ref_lse, "psbad")


@pytest.mark.parametrize("fp8", [True, False], ids=["fp8", "bf16"])
@pytest.mark.parametrize("parts", [1, 5, 300])
def test_pair_sparse_forced_splits(parts, fp8):
    w = W.custom(name=f"psp{parts}", batch=3, h_q=128, s_q=2, mode="sparse", fp8=fp8, seqlens=(5000, 3000, 700),
                 topk=640)
    check(w, 2000 + parts, parts=parts)


def test_pair_sparse_token_scales_and_ragged_topk():
    check(W.custom(name="pstok", batch=3, h_q=128, s_q=1, mode="sparse", seqlens=(2000, 300, 5000), topk=384,
                   fp8_scales="token"), 2101)
    w = W.custom(name="psrag", batch=3, h_q=128, s_q=2, mode="sparse", seqlens=(1500, 200, 3000), topk=320,
                 ragged_topk=True)
    inp = W.make_inputs(w, seed=2102)
    tl = inp.topk_lengths.clone()
    tl[0, 0] = 0
    tl[1, 1] = 320
    tl[2, 0] = 129
    inp.topk_lengths = tl
    out, lse, flags = run_cuda(inp)
    assert flags == 0
    ref_out, ref_lse = run_oracle(inp)
    compare(out, lse, ref_out, ref_lse, w.name)


def test_pair_sparse_rescale_path():
    check(W.custom(name="psbig", batch=2, h_q=128, s_q=1, mode="sparse", seqlens=(4000, 2000), topk=1024,
                   sm_scale=0.6), 2201, parts=1)


# ---------------------------------------------------------------- sparse mode
@pytest.mark.parametrize("h_q,topk", [(16, 64), (16, 200), (64, 128), (128, 300), (32, 1000), (48, 129)])
def test_sparse_small(h_q, topk):
    w = W.custom(name=f"sp{h_q}_{topk}", batch=2, h_q=h_q, s_q=2, mode="sparse", seqlens=(1500, 400),
                 topk=topk)
    check(w, 400 + h_q + topk)


def test_sparse_duplicates_and_invalid_ids():
    w = W.custom(name="spdup", batch=2, h_q=64, s_q=2, mode="sparse", seqlens=(300, 90), topk=256)
    inp = W.make_inputs(w, seed=21)
    idx = inp.indices.clone()
    idx[0, 0, :40] = 7           # one id forty times
    idx[0, 1, 5] = 300           # == seqlen: skipped
    idx[1, 0, 9] = 10 ** 7       # far out of range: skipped
    idx[1, 1, :] = -1            # empty key set
    inp.indices = idx
    out, lse, flags = run_cuda(inp)
    ref_out, ref_lse = run_oracle(inp)
    assert flags == 0
    compare(out, lse, ref_out, ref_lse, "spdup")
    assert np.all(out[1, 1] == 0) and np.all(np.isneginf(lse[1, 1]))


@pytest.mark.parametrize("parts", [1, 5, 300])
def test_sparse_forced_splits(parts):
    w = W.custom(name=f"sparts{parts}", batch=3, h_q=128, s_q=2, mode="sparse", seqlens=(5000, 3000, 700),
                 topk=640)
    check(w, 500 + parts, parts=parts)


def test_sparse_equals_dense_over_all_tokens():
    """indices = all tokens of the FP8 cache equals dense decode over the dequantised bf16 cache."""
    L = (700, 129)
    w = W.custom(name="spall", batch=2, h_q=64, s_q=1, mode="sparse", seqlens=L, topk=768, invalid_frac=0.0)
    inp = W.make_inputs(w, seed=31, poison_tail=False)
    idx = torch.full((2, 1, 768), -1, dtype=torch.int32)
    for b in range(2):
        idx[b, 0, :L[b]] = torch.randperm(L[b], generator=torch.Generator().manual_seed(b)).int()
    inp.indices = idx
    out_s, lse_s, _ = run_cuda(inp)
    flat = inp.kvcache.reshape(-1, 656)
    n = flat.shape[0]
    codes = flat[:, :512].contiguous().view(torch.float8_e4m3fn).float().reshape(n, 4, 128)
    scales = flat[:, 512:528].contiguous().view(torch.float32).reshape(n, 4)
    nope = (codes * scales[:, :, None]).reshape(n, 512).to(torch.bfloat16)
    rope = flat[:, 528:].contiguous().view(torch.bfloat16)
    kvb = torch.cat([nope, rope], 1).reshape(inp.kvcache.shape[0], 64, 1, 576)
    dense = W.Inputs(W.custom(name="d", batch=2, h_q=64, s_q=1, mode="dense", seqlens=L), inp.q, kvb,
                     inp.block_table, inp.cache_seqlens, None, inp.sm_scale, 0)
    out_d, lse_d, _ = run_cuda(dense)
    compare(out_s, lse_s, out_d, lse_d, "sparse-vs-dense")


# ---------------------------------------------------------------- schedule
@pytest.mark.parametrize("topk,lens", [(0, (5000, 1, 0, 130, 64, 20000)), (512, (100, 100, 100))])
def test_schedule_covers_every_tile_once(topk, lens):
    s_q, h_q = 2, 128
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    sched, ns = mla.get_metadata(sl, h_q=h_q, s_q=s_q, topk=topk, is_fp8=topk > 0)
    sched = sched.view(-1, 8).cpu().numpy()
    ns = ns.cpu().numpy()
    np_ = len(lens) * (s_q if topk else 1)
    tiles = [math.ceil(topk / 64) if topk else math.ceil(L / 64) for L in
             ([lens[p // s_q] for p in range(np_)] if topk else lens)]
    seen = {}
    count = np.zeros(np_, int)
    for k, (p0, t0, p1, t1, sp0, *_rest) in enumerate(sched):
        touched = []
        for p in range(p0, min(p1, np_ - 1) + 1):
            tb = t0 if p == p0 else 0
            te = t1 if p == p1 else tiles[p]
            for t in range(tb, min(te, tiles[p])):
                assert (p, t) not in seen
                seen[(p, t)] = k
            if tb < min(te, tiles[p]):
                touched.append(p)
        for p in touched:
            count[p] += 1
        if touched and touched[0] == p0:
            assert sp0 == count[p0] - 1
    assert len(seen) == sum(tiles)
    # partial-result slots: one per piece of a split problem, none for a single piece
    assert ns[0] == 0 and np.array_equal(np.diff(ns), np.where(count > 1, count, 0))
    assert ns[-1] <= min(2 * len(sched), np_ + len(sched))


# ---------------------------------------------------------------- device status
@pytest.mark.parametrize("case", ["parts", "mode"])
def test_schedule_of_another_configuration_is_flagged(case):
    """A schedule made for another part count or another cache format is reported by the decode
    (it checks the first record's part count and configuration tag) and nothing else is read."""
    w = W.custom(name="mismatch", batch=2, h_q=64, s_q=1, mode="dense", seqlens=(300, 100))
    d = W.make_inputs(w, seed=8).to("cuda")
    mla.device_status()
    if case == "parts":
        with overrides(num_parts=5):
            sched, ns = metadata(d, w)
    else:
        sched, ns = mla.get_metadata(d.cache_seqlens, h_q=w.h_q, s_q=w.s_q, topk=0, is_fp8=True)
    out, lse = mla.decode(d.q, d.kvcache, d.block_table, d.cache_seqlens, d.sm_scale, sched, ns)
    flags = mla.device_status()
    assert flags & mla.DEVICE_BAD_SCHEDULE
    # the same inputs with a matching schedule still decode correctly
    out, lse, flags = run_cuda(W.make_inputs(w, seed=8))
    assert flags == 0



@pytest.mark.parametrize("h_q", [16, 64])
def test_bad_page_is_flagged_not_faulted(h_q):
    """16 rows: one full barrier per tile; 64 rows: one per ring item, armed with no bytes for a bad page."""
    w = W.custom(name="badpage", batch=2, h_q=h_q, s_q=1, mode="dense", seqlens=(200, 100))
    inp = W.make_inputs(w, seed=3)
    bt = inp.block_table.clone()
    bt[0, 1] = inp.kvcache.shape[0] + 5
    inp.block_table = bt
    out, lse, flags = run_cuda(inp)
    assert flags & mla.DEVICE_BAD_PAGE
    assert np.all(np.isfinite(out))
    assert mla.device_status() == 0  # cleared by the previous read


# ---------------------------------------------------------------- full-size workloads
FULL_SIZE = ["tiny", "dense_membound", "dense_computebound", "sparse_fp8", "sparse_fp8_long", "sparse_bf16",
             "sparse_fp8_token", "dense_membound_fp8"]


@pytest.mark.parametrize("name", FULL_SIZE)
def test_full_size_workload(name):
    """Every output row of a named workload, in the launch configuration the benchmark times,
    against the oracle run over all rows (all host threads)."""
    inp = W.make_inputs(name)
    out, lse, flags = run_cuda(inp)
    assert flags == 0
    assert np.all(np.isfinite(out))
    ref_out, ref_lse = run_oracle(inp)
    compare(out, lse, ref_out, ref_lse, name)
    # property at any size: each output row is a convex combination of value rows
    if inp.workload.mode == "dense" and not inp.workload.is_fp8:
        vmax = float(inp.kvcache[..., :512].float().nan_to_num(0.0).abs().max())
        assert float(np.abs(out).max()) <= vmax * (1 + 1e-2)


# ---------------------------------------------------------------- dense over the FP8 cache
@pytest.mark.parametrize("L", [1, 63, 64, 65, 200, 1000])
def test_dense_fp8_lengths(L):
    check(W.custom(name=f"dfp8_{L}", batch=2, h_q=16, s_q=1, mode="dense", fp8=True, seqlens=(L, max(1, L // 3))),
          700 + L)


@pytest.mark.parametrize("h_q,s_q,causal", [(32, 1, False), (64, 1, False), (128, 2, True), (16, 4, True),
                                            (40, 3, False)])
def test_dense_fp8_row_shapes_and_causal(h_q, s_q, causal):
    check(W.custom(name=f"dfp8h{h_q}s{s_q}", batch=3, h_q=h_q, s_q=s_q, mode="dense", fp8=True,
                   seqlens=(200, 77, 513), causal=causal), 800 + h_q + s_q)


@pytest.mark.parametrize("parts", [1, 7, 300])
def test_dense_fp8_forced_splits_and_empty(parts):
    w = W.custom(name=f"dfp8p{parts}", batch=4, h_q=64, s_q=2, mode="dense", fp8=True,
                 seqlens=(1000, 0, 130, 2049), causal=True)
    out, lse, _, _ = check(w, 900 + parts, parts=parts)
    assert np.all(out[1] == 0) and np.all(np.isneginf(lse[1]))


def test_dense_fp8_equals_dense_over_dequantised_cache():
    """Dense decode over an FP8 cache equals dense decode over its dequantised bf16 copy."""
    w = W.custom(name="dfp8eq", batch=2, h_q=64, s_q=1, mode="dense", fp8=True, seqlens=(700, 129))
    inp = W.make_inputs(w, seed=33, poison_tail=False)
    out_f, lse_f, _ = run_cuda(inp)
    flat = inp.kvcache.reshape(-1, 656)
    n = flat.shape[0]
    codes = flat[:, :512].contiguous().view(torch.float8_e4m3fn).float().reshape(n, 4, 128)
    scales = flat[:, 512:528].contiguous().view(torch.float32).reshape(n, 4)
    nope = (codes * scales[:, :, None]).reshape(n, 512).to(torch.bfloat16)
    rope = flat[:, 528:].contiguous().view(torch.bfloat16)
    kvb = torch.cat([nope, rope], 1).reshape(inp.kvcache.shape[0], 64, 1, 576)
    dense = W.Inputs(W.custom(name="d", batch=2, h_q=64, s_q=1, mode="dense", seqlens=(700, 129)), inp.q, kvb,
                     inp.block_table, inp.cache_seqlens, None, inp.sm_scale, 0)
    out_d, lse_d, _ = run_cuda(dense)
    compare(out_f, lse_f, out_d, lse_d, "dense-fp8-vs-dense")


# ---------------------------------------------------------------- per-token-scale FP8 rows, ragged top-k
@pytest.mark.parametrize("h_q,s_q", [(16, 1), (64, 2), (128, 1)])
def test_sparse_token_scale_cache(h_q, s_q):
    """640-byte FP8 rows with one scale per token (16/64-row CTAs, two row groups)."""
    check(W.custom(name=f"stok{h_q}", batch=3, h_q=h_q, s_q=s_q, mode="sparse", seqlens=(2000, 300, 5000),
                   topk=384, fp8_scales="token"), 1100 + h_q)


@pytest.mark.parametrize("h_q,s_q,causal", [(16, 1, False), (64, 1, False), (128, 2, True)])
def test_dense_token_scale_cache(h_q, s_q, causal):
    check(W.custom(name=f"dtok{h_q}", batch=3, h_q=h_q, s_q=s_q, mode="dense", fp8=True, fp8_scales="token",
                   seqlens=(200, 77, 513), causal=causal), 1200 + h_q)


@pytest.mark.parametrize("fp8", [True, False])
@pytest.mark.parametrize("h_q", [16, 64])
def test_sparse_topk_lengths(h_q, fp8):
    """Ragged top-k: the slots past each row's length hold valid-looking ids that must be ignored."""
    w = W.custom(name=f"rag{h_q}{int(fp8)}", batch=3, h_q=h_q, s_q=2, mode="sparse", fp8=fp8,
                 seqlens=(1500, 200, 3000), topk=320, ragged_topk=True)
    inp = W.make_inputs(w, seed=1300 + h_q)
    tl = inp.topk_lengths.clone()
    tl[0, 0] = 0          # empty row
    tl[1, 1] = 320        # every slot
    tl[2, 0] = -5         # negative: empty
    inp.topk_lengths = tl
    out, lse, flags = run_cuda(inp)
    assert flags == 0
    ref_out, ref_lse = run_oracle(inp)
    compare(out, lse, ref_out, ref_lse, w.name)
    assert np.all(out[0, 0] == 0) and np.all(lse[0, 0] == -np.inf)


# ---------------------------------------------------------------- largest supported shapes
def test_dense_max_rows_per_problem():
    """1024 query rows per problem (s_q 8 x 128 heads): 16 row groups, causal."""
    check(W.custom(name="rows1024", batch=2, h_q=128, s_q=8, mode="dense", seqlens=(300, 70), causal=True), 1401)


def test_sparse_max_heads():
    """1024 heads of one sparse query token: 16 row groups reading the same gathered rows."""
    check(W.custom(name="heads1024", batch=1, h_q=1024, s_q=1, mode="sparse", seqlens=(900,), topk=200), 1402)
