"""Pins for the fp64 oracle: each checks it against something other than itself.

* an independent numpy/scipy brute force over an explicitly gathered
  contiguous K (torch's float8 cast for FP8 decoding) on tiny inputs;
* closed forms (one key, equal logits, q = 0) and invariants (page
  permutation, sparse-over-all-tokens = dense, split/merge, causal);
* the E4M3 code table against torch.float8_e4m3fn, the 656-byte layout
  against the numbers printed in the FlashMLA article;
* mutation tests: plausible mistakes planted in a copy of the oracle source
  must make at least one pin fail.
"""
import math
import os
import re
import tempfile

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from paged_mla_decode_07_gb300 import workloads as W

HERE = os.path.dirname(os.path.abspath(__file__))
LN2 = math.log(2.0)


# ----------------------------------------------------------------------------
# independent brute force (numpy / scipy / torch library casts only)
# ----------------------------------------------------------------------------
def torch_dequant_rows(rows_u8: torch.Tensor) -> np.ndarray:
    """[n, 656] uint8 -> [n, 576] float64 via torch's float8 cast and fp32 multiply."""
    n = rows_u8.shape[0]
    codes = rows_u8[:, :512].contiguous().view(torch.float8_e4m3fn).float().reshape(n, 4, 128)
    scales = rows_u8[:, 512:528].contiguous().view(torch.float32).reshape(n, 4)
    nope = (codes * scales[:, :, None]).reshape(n, 512).to(torch.bfloat16)
    rope = rows_u8[:, 528:656].contiguous().view(torch.bfloat16).reshape(n, 64)
    return torch.cat([nope, rope], dim=1).double().numpy()


def brute_force(inp):
    w = inp.workload
    q = inp.q.float().double().numpy()
    kv = inp.kvcache
    ps = kv.shape[1]
    flat = kv.reshape(kv.shape[0] * ps, kv.shape[-1])
    table = inp.block_table.numpy()
    lens = inp.cache_seqlens.numpy()
    b_, s_q, h_q, _ = q.shape
    out = np.zeros((b_, s_q, h_q, 512))
    lse = np.zeros((b_, s_q, h_q))
    for b in range(b_):
        L = int(lens[b])
        for i in range(s_q):
            if inp.indices is not None:
                ids = inp.indices[b, i].numpy().astype(np.int64)
                ids = ids[(ids >= 0) & (ids < L)]
            else:
                last = L - s_q + i if w.causal else L - 1
                ids = np.arange(0, min(last, L - 1) + 1, dtype=np.int64)
            if ids.size == 0:
                lse[b, i] = -np.inf
                continue
            pos = table[b, ids // ps].astype(np.int64) * ps + ids % ps
            if w.is_fp8:
                K = torch_dequant_rows(flat[torch.from_numpy(pos)])
            else:
                K = flat[torch.from_numpy(pos)].double().numpy()
            s = q[b, i] @ K.T * inp.sm_scale                     # [h_q, n]
            lnat = scipy.special.logsumexp(s, axis=1)
            out[b, i] = np.exp(s - lnat[:, None]) @ K[:, :512]
            lse[b, i] = lnat / LN2
    return out, lse


def run_oracle(inp, **kw):
    return oracle.mla_decode(inp.q, inp.kvcache, inp.block_table, inp.cache_seqlens, inp.sm_scale,
                             is_causal=inp.workload.causal, indices=inp.indices, **kw)


def assert_close(a, b, rtol=1e-12, atol=1e-12):
    a = np.asarray(a)
    b = np.asarray(b)
    fin = np.isfinite(b)
    assert np.array_equal(np.isfinite(a), fin)
    assert np.array_equal(a[~fin], b[~fin])
    np.testing.assert_allclose(a[fin], b[fin], rtol=rtol, atol=atol)


def tiny_cases(n, seed=0):
    rng = np.random.default_rng(seed)
    for c in range(n):
        mode = "sparse" if c % 2 else "dense"
        batch = int(rng.integers(1, 4))
        s_q = int(rng.integers(1, 3))
        h_q = int(rng.integers(1, 5))
        lens = tuple(int(x) for x in rng.integers(1, 201, size=batch))
        kw = dict(batch=batch, h_q=h_q, s_q=s_q, mode=mode, seqlens=lens)
        if mode == "sparse":
            kw["topk"] = int(rng.integers(1, 97))
        else:
            kw["causal"] = bool(rng.integers(0, 2))
        kw["sm_scale"] = float(rng.choice([1.0 / math.sqrt(576), 0.1, 0.02]))
        yield W.custom(name=f"tiny{c}", **kw), 100 + c


# ----------------------------------------------------------------------------
# pins
# ----------------------------------------------------------------------------
def test_e4m3_table_matches_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).float().double().numpy()
    mine = np.array([oracle.e4m3_to_double(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(mine))
    assert nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(ref[~nan], mine[~nan])
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9


def test_fp8_layout_golden():
    g = {}
    for line in open(os.path.join(HERE, "golden", "fp8_layout.txt")):
        if line.strip() and not line.startswith("#"):
            k, v = line.split()
            g[k] = float(v)
    assert g["nope_bytes"] + g["scale_bytes"] + g["rope_bytes"] == g["token_bytes"] == W.FP8_ROW_BYTES
    assert g["nope_dims"] + g["rope_dims"] == W.D_QK and g["nope_dims"] == W.D_V
    assert g["scales_per_token"] * 4 == g["scale_bytes"]
    assert g["scales_per_token"] * g["scale_tile"] == g["nope_dims"]
    assert g["bf16_token_bytes"] == 2 * W.D_QK
    assert round(100 * (1 - g["token_bytes"] / g["bf16_token_bytes"])) == g["saving_percent"]
    gib = W.D_QK * 2 * g["layers_in_size_example"] * 128 * 1024 / 2 ** 30
    assert abs(gib - g["request_128k_gib"]) < 0.005


def test_dequant_layout_offsets():
    """Known bytes at each field land on the documented dims."""
    row = np.zeros(656, np.uint8)
    scales = np.array([0.5, 2.0, 3.0, 0.25], np.float32)
    row[512:528] = scales.view(np.uint8)
    for d in (0, 127, 128, 300, 511):
        row[d] = 0x38  # e4m3 1.0
    rope = torch.tensor([1.5 + t for t in range(64)], dtype=torch.bfloat16)
    row[528:656] = rope.view(torch.uint8).numpy()
    k = oracle.dequant_row(row)
    assert k[0] == 0.5 and k[127] == 0.5 and k[128] == 2.0 and k[300] == 3.0 and k[511] == 0.25
    assert k[1] == 0.0 and k[256] == 0.0
    np.testing.assert_array_equal(k[512:], rope.double().numpy())


def test_dequant_matches_torch_on_random_rows():
    x = torch.randn(300, 576, generator=torch.Generator().manual_seed(3)) * 3
    rows = W.encode_fp8_rows(x)
    ref = torch_dequant_rows(rows)
    mine = np.stack([oracle.dequant_row(r) for r in rows.numpy()])
    assert np.array_equal(ref, mine)


def test_quantiser_roundtrip_bound():
    """Generator encoding + oracle decoding stays within e4m3 and bf16 rounding of the source."""
    x = torch.randn(200, 576, generator=torch.Generator().manual_seed(4), dtype=torch.float32)
    rows = W.encode_fp8_rows(x)
    deq = np.stack([oracle.dequant_row(r) for r in rows.numpy()])
    src = x.double().numpy()
    scale = rows[:, 512:528].contiguous().view(torch.float32).double().numpy()
    sc = np.repeat(scale, 128, axis=1)
    err = np.abs(deq[:, :512] - src[:, :512])
    assert np.all(err <= (2.0 ** -4 + 2.0 ** -8) * np.abs(src[:, :512]) + sc * 2.0 ** -9)
    assert np.all(np.abs(deq[:, 512:] - src[:, 512:]) <= 2.0 ** -8 * np.abs(src[:, 512:]))


@pytest.mark.parametrize("case", list(tiny_cases(50)), ids=lambda c: c[0].name)
def test_bruteforce_tiny(case):
    w, seed = case
    inp = W.make_inputs(w, seed=seed)
    o_ref, l_ref = brute_force(inp)
    o, l = run_oracle(inp)
    assert_close(o, o_ref)
    assert_close(l, l_ref)


def test_bruteforce_duplicates_and_invalid_ids():
    w = W.custom(batch=2, h_q=3, s_q=2, mode="sparse", seqlens=(90, 130), topk=40)
    inp = W.make_inputs(w, seed=9)
    idx = inp.indices.clone()
    idx[0, 0, :10] = 5           # repeated id counts ten times
    idx[0, 1, 3] = 90            # == seqlen -> skipped
    idx[1, 0, 7] = 10 ** 6       # far out of range -> skipped
    idx[1, 1, :] = -1            # all invalid -> empty row
    inp.indices = idx
    o_ref, l_ref = brute_force(inp)
    o, l = run_oracle(inp)
    assert_close(o, o_ref)
    assert_close(l, l_ref)
    assert np.all(l[1, 1] == -np.inf) and np.all(o[1, 1] == 0)


def test_empty_dense_row():
    w = W.custom(batch=2, h_q=2, s_q=1, mode="dense", seqlens=(0, 5))
    inp = W.make_inputs(w, seed=1)
    o, l = run_oracle(inp)
    assert np.all(o[0] == 0) and np.all(l[0] == -np.inf)
    assert np.all(np.isfinite(l[1]))


def test_paging_invariant_bit_exact():
    """The same logical cache under a random page permutation gives identical results."""
    w = W.custom(batch=3, h_q=4, s_q=2, mode="dense", seqlens=(130, 64, 200), causal=True)
    inp = W.make_inputs(w, seed=21)
    o1, l1 = run_oracle(inp)
    rng = np.random.default_rng(0)
    P = inp.kvcache.shape[0]
    perm = rng.permutation(P)                 # new physical slot of each old page
    kv2 = torch.empty_like(inp.kvcache)
    kv2[torch.from_numpy(perm)] = inp.kvcache
    t2 = torch.from_numpy(perm[inp.block_table.numpy()].astype(np.int32))
    inp2 = W.Inputs(w, inp.q, kv2, t2, inp.cache_seqlens, None, inp.sm_scale, 0)
    o2, l2 = run_oracle(inp2)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_sparse_over_all_tokens_equals_dense():
    """indices = every token (shuffled) over an FP8 cache equals dense decode over the
    bf16 cache holding the same dequantised values."""
    L = (150, 77)
    w = W.custom(batch=2, h_q=4, s_q=2, mode="sparse", seqlens=L, topk=150, invalid_frac=0.0)
    inp = W.make_inputs(w, seed=33, poison_tail=False)
    rng = np.random.default_rng(1)
    idx = np.full((2, 2, 150), -1, np.int32)
    for b in range(2):
        for i in range(2):
            idx[b, i, :L[b]] = rng.permutation(L[b])
    inp.indices = torch.from_numpy(idx)
    o_sp, l_sp = run_oracle(inp)
    flat = inp.kvcache.reshape(-1, 656)
    deq = torch.from_numpy(torch_dequant_rows(flat)).to(torch.bfloat16)
    kv_bf16 = deq.reshape(inp.kvcache.shape[0], 64, 1, 576)
    wd = W.custom(batch=2, h_q=4, s_q=2, mode="dense", seqlens=L)
    dense = W.Inputs(wd, inp.q, kv_bf16, inp.block_table, inp.cache_seqlens, None, inp.sm_scale, 0)
    o_d, l_d = run_oracle(dense)
    assert_close(o_sp, o_d)
    assert_close(l_sp, l_d)


def test_single_key_closed_form():
    w = W.custom(batch=1, h_q=3, s_q=1, mode="dense", seqlens=(1,), sm_scale=0.07)
    inp = W.make_inputs(w, seed=5)
    o, l = run_oracle(inp)
    k0 = inp.kvcache[inp.block_table[0, 0], 0, 0].double().numpy()
    q = inp.q[0, 0].double().numpy()
    np.testing.assert_array_equal(o[0, 0], np.broadcast_to(k0[:512], (3, 512)))
    np.testing.assert_allclose(l[0, 0], (q @ k0) * 0.07 / LN2, rtol=1e-13)


def test_equal_logits_give_mean_of_v():
    """Zero NoPE query and shared RoPE key dims -> equal logits -> out = mean(V),
    lse = log2(n) + s/ln2; q = 0 -> out = mean(V), lse = log2(n)."""
    n = 93
    w = W.custom(batch=1, h_q=2, s_q=1, mode="dense", seqlens=(n,))
    inp = W.make_inputs(w, seed=6, poison_tail=False)
    kv = inp.kvcache.clone()
    kv[:, :, :, 512:] = kv[0, 0, :, 512:]
    q = inp.q.clone()
    q[..., :512] = 0
    toks = []
    for j in range(n):
        toks.append(kv[inp.block_table[0, j // 64], j % 64, 0].double().numpy())
    K = np.stack(toks)
    mean_v = K[:, :512].mean(axis=0)
    inp2 = W.Inputs(w, q, kv, inp.block_table, inp.cache_seqlens, None, inp.sm_scale, 0)
    o, l = run_oracle(inp2)
    s = (q[0, 0].double().numpy() @ K[0]) * inp.sm_scale
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(mean_v, (2, 512)), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l[0, 0], math.log2(n) + s / LN2, rtol=1e-12)
    inp3 = W.Inputs(w, torch.zeros_like(q), inp.kvcache, inp.block_table, inp.cache_seqlens, None,
                    inp.sm_scale, 0)
    o, l = run_oracle(inp3)
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(mean_v, (2, 512)), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l[0, 0], math.log2(n), rtol=1e-13)


def test_lse_is_base2():
    w = W.custom(batch=1, h_q=2, s_q=1, mode="dense", seqlens=(37,), sm_scale=0.05)
    inp = W.make_inputs(w, seed=7)
    o, l = run_oracle(inp)
    q = inp.q[0, 0].double().numpy()
    K = np.stack([inp.kvcache[inp.block_table[0, j // 64], j % 64, 0].double().numpy()
                  for j in range(37)])
    z = np.exp((q @ K.T) * 0.05).sum(axis=1)
    np.testing.assert_allclose(2.0 ** l[0, 0], z, rtol=1e-12)


@pytest.mark.parametrize("mode", ["dense", "sparse"])
def test_split_merge_invariant(mode):
    kw = dict(topk=120) if mode == "sparse" else dict(causal=True)
    w = W.custom(batch=2, h_q=3, s_q=2, mode=mode, seqlens=(200, 131), **kw)
    inp = W.make_inputs(w, seed=11)
    full_o, full_l = oracle.mla_decode(inp.q, inp.kvcache, inp.block_table, inp.cache_seqlens,
                                       inp.sm_scale, is_causal=w.causal, indices=inp.indices,
                                       rows=np.arange(12))
    cuts = [0, 17, 64, 65, 129, 10 ** 6]
    parts = [oracle.mla_partial(inp.q, inp.kvcache, inp.block_table, inp.cache_seqlens,
                                inp.sm_scale, a, b, is_causal=w.causal, indices=inp.indices)
             for a, b in zip(cuts[:-1], cuts[1:])]
    for r in range(12):
        o, l = oracle.lse_merge(np.stack([p[0][r] for p in parts]), [p[1][r] for p in parts])
        np.testing.assert_allclose(o, full_o[r], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(l, full_l[r], rtol=1e-13)
    o, l = oracle.lse_merge(np.zeros((2, 512)), [-np.inf, -np.inf])
    assert l == -np.inf and np.all(o == 0)


def test_causal_cases():
    w1 = W.custom(batch=2, h_q=3, s_q=1, mode="dense", seqlens=(70, 9), causal=True)
    inp = W.make_inputs(w1, seed=12)
    oc, lc = run_oracle(inp)
    on, ln = oracle.mla_decode(inp.q, inp.kvcache, inp.block_table, inp.cache_seqlens, inp.sm_scale)
    assert np.array_equal(oc, on) and np.array_equal(lc, ln)
    # s_q = 2: query token 0 sees seqlen-1 keys
    w2 = W.custom(batch=1, h_q=3, s_q=2, mode="dense", seqlens=(70,), causal=True)
    inp2 = W.make_inputs(w2, seed=13)
    o2, l2 = run_oracle(inp2)
    short = W.Inputs(W.custom(batch=1, h_q=3, s_q=1, mode="dense", seqlens=(69,)),
                     inp2.q[:, :1].contiguous(), inp2.kvcache, inp2.block_table,
                     torch.tensor([69], dtype=torch.int32), None, inp2.sm_scale, 0)
    o3, l3 = run_oracle(short)
    assert np.array_equal(o2[:, 0], o3[:, 0]) and np.array_equal(l2[:, 0], l3[:, 0])
    o4, l4 = oracle.mla_decode(inp2.q, inp2.kvcache, inp2.block_table, inp2.cache_seqlens,
                               inp2.sm_scale)
    assert np.array_equal(o2[:, 1], o4[:, 1])


def test_named_workload_shapes():
    """The generator reproduces the structure of the five named workloads (small ones drawn)."""
    t = W.make_inputs("tiny")
    assert t.kvcache.shape == (7, 64, 1, 576) and t.cache_seqlens.tolist() == [100, 257]
    assert sorted(t.block_table[0, :2].tolist() + t.block_table[1, :5].tolist()) == list(range(7))
    w = W.WORKLOADS["sparse_fp8"]
    assert (w.batch, w.h_q, w.s_q, w.topk, w.seqlen) == (128, 128, 2, 2048, 32768)
    small = W.with_fields(w, batch=2, seqlen=4096, topk=256)
    s = W.make_inputs(small, seed=1)
    assert s.kvcache.shape[-1] == 656 and s.kvcache.dtype == torch.uint8
    idx = s.indices.numpy()
    assert np.all(idx[..., 256 - 12:] == -1) and np.all(idx[..., :256 - 12] >= 0)
    for b in range(2):
        for i in range(2):
            v = idx[b, i][idx[b, i] >= 0]
            assert len(np.unique(v)) == len(v) and v.max() < 4096


# ----------------------------------------------------------------------------
# mutation tests: each planted mistake must be caught by a pin above
# ----------------------------------------------------------------------------
MUTATIONS = {
    "rope_dims_dropped_from_logits": ("for (int d = 0; d < D_QK; ++d) acc += bf16_bits_to_double(q[d]) * kbuf[d];",
                                      "for (int d = 0; d < D_V; ++d) acc += bf16_bits_to_double(q[d]) * kbuf[d];"),
    "natural_log_lse": ("  *lse = (m + log(z)) / log(2.0);\n  return 1;", "  *lse = (m + log(z));\n  return 1;"),
    "page_slot_swapped": ("int slot = j % p->page_size;", "int slot = (j + 1) % p->page_size;"),
    "wrong_scale_tile": ("4 * (d / 128)", "4 * (d / 256)"),
    "causal_off_by_one": ("last = L - p->s_q + i;", "last = L - p->s_q + i - 1;"),
    "rope_offset": ("FP8_ROPE_OFFSET + 2 * (d - D_V)", "FP8_ROPE_OFFSET + 2 * (d - D_V + 1) % 128"),
    "invalid_index_kept": ("if (idx[k] >= 0 && idx[k] < L)", "if (idx[k] >= 0)"),
    "v_from_rope_end": ("out[d] += w * kbuf[d];", "out[d] += w * kbuf[d + 64];"),
    "merge_sign": ("double w = exp2(lses[i] - L);", "double w = exp2(L - lses[i]);"),
    "topk_lengths_ignored": ("n_slots = len < 0 ? 0 : (len < p->topk ? len : p->topk);", "n_slots = p->topk;"),
    "token_scale_rope_offset": ("memcpy(&h, row + D_V + 2 * (d - D_V), sizeof h);",
                                "memcpy(&h, row + D_V + 16 + 2 * (d - D_V), sizeof h);"),
}


def _mutant_checks():
    """Run a compact set of pins; return True if all pass."""
    try:
        for w, seed in list(tiny_cases(8, seed=5)):
            inp = W.make_inputs(w, seed=seed)
            o_ref, l_ref = brute_force(inp)
            o, l = run_oracle(inp)
            assert_close(o, o_ref)
            assert_close(l, l_ref)
        w = W.custom(batch=2, h_q=2, s_q=2, mode="sparse", seqlens=(90, 70), topk=40)
        inp = W.make_inputs(w, seed=3)
        idx = inp.indices.clone()
        idx[0, 0, 0] = 95
        inp.indices = idx
        o_ref, l_ref = brute_force(inp)
        o, l = run_oracle(inp)
        assert_close(o, o_ref)
        test_split_merge_invariant("dense")
        test_token_scale_dequant_matches_torch()
        test_topk_lengths_ignore_the_slots_past_them()
        return True
    except AssertionError:
        return False


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "mla_oracle.c")).read()
    assert src.count(old) == 1, f"mutation anchor not found: {old}"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = oracle.build(force=True, src=str(path), out=str(tmp_path / "libmutant.so"))
    with oracle.use_library(lib):
        assert not _mutant_checks(), f"planted mistake '{name}' went unnoticed"
    assert _mutant_checks()


# ----------------------------------------------------------------------------
# per-token-scale FP8 rows and ragged top-k lengths
# ----------------------------------------------------------------------------
def test_token_scale_dequant_matches_torch():
    """640-byte rows with one fp32 scale per token, against torch's E4M3 cast and fp32 multiply."""
    g = torch.Generator().manual_seed(12)
    x = torch.randn(40, 576, generator=g) * torch.rand(40, 1, generator=g) * 5
    rows, scales = W.encode_fp8_token_rows(x)
    for n in range(40):
        k = oracle.dequant_row_token_scale(rows[n].numpy(), float(scales[n]))
        codes = rows[n, :512].contiguous().view(torch.float8_e4m3fn).float()
        ref = (codes * scales[n]).to(torch.bfloat16).double().numpy()
        np.testing.assert_array_equal(k[:512], ref)
        np.testing.assert_array_equal(k[512:], x[n, 512:].to(torch.bfloat16).double().numpy())


def test_token_scale_cache_equals_its_dequantised_bf16_cache():
    w = W.custom(name="tok", batch=2, h_q=4, s_q=2, mode="sparse", seqlens=(150, 90), topk=48,
                 fp8_scales="token")
    inp = W.make_inputs(w, seed=13, poison_tail=False)
    assert inp.kvcache.shape[-1] == 640 and inp.kv_scales.shape == inp.kvcache.shape[:2]
    flat = inp.kvcache.reshape(-1, 640)
    sc = inp.kv_scales.reshape(-1)
    kb = np.stack([oracle.dequant_row_token_scale(flat[n].numpy(), float(sc[n])) for n in range(flat.shape[0])])
    kvb = torch.from_numpy(kb).float().to(torch.bfloat16).reshape(inp.kvcache.shape[0], 64, 1, 576)
    o1, l1 = oracle.mla_decode(inp.q, inp.kvcache, inp.block_table, inp.cache_seqlens, inp.sm_scale,
                               indices=inp.indices, kv_scales=inp.kv_scales)
    o2, l2 = oracle.mla_decode(inp.q, kvb, inp.block_table, inp.cache_seqlens, inp.sm_scale, indices=inp.indices)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_topk_lengths_ignore_the_slots_past_them():
    """Ragged top-k: slots past topk_lengths hold valid-looking ids that must not count; the result
    equals the same rows with those slots set to -1, and a zero length gives an empty row."""
    w = W.custom(name="rag", batch=3, h_q=2, s_q=2, mode="sparse", seqlens=(200, 90, 130), topk=40,
                 ragged_topk=True)
    inp = W.make_inputs(w, seed=14)
    tl = inp.topk_lengths.clone()
    tl[1, 1] = 0
    tl[2, 0] = 40
    o, l = oracle.mla_decode(inp.q, inp.kvcache, inp.block_table, inp.cache_seqlens, inp.sm_scale,
                             indices=inp.indices, topk_lengths=tl)
    masked = inp.indices.clone()
    for b in range(3):
        for i in range(2):
            masked[b, i, int(tl[b, i]):] = -1
    o2, l2 = oracle.mla_decode(inp.q, inp.kvcache, inp.block_table, inp.cache_seqlens, inp.sm_scale, indices=masked)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(l, l2)
    assert np.all(o[1, 1] == 0) and np.all(l[1, 1] == -np.inf)
    o3, _ = oracle.mla_decode(inp.q, inp.kvcache, inp.block_table, inp.cache_seqlens, inp.sm_scale,
                              indices=inp.indices)
    assert not np.array_equal(o3, o)   # the ids past the lengths would have changed the result
