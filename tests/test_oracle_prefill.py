"""Pins for the oracle's sparse prefill (flash_mla_sparse_fwd semantics of the
FlashMLA article's usage section), each against something other than itself:

* an independent numpy/scipy brute force (gather, logits, logsumexp) on tiny
  inputs with invalid, out-of-range and repeated ids;
* the sparse decode oracle (itself pinned in test_oracle_pins.py) on the same
  KV laid out as a permuted paged bf16 cache with one batch element;
* closed forms: one valid id, n copies of one id, no valid id;
* invariance under a permutation of each index row;
* planted mistakes in a copy of the oracle source must fail a pin.
"""
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from paged_mla_decode_07_gb300 import workloads as W

LN2 = math.log(2.0)


def brute_force(inp):
    q = inp.q.double().numpy()
    kv = inp.kv.double().numpy()
    idx = inp.indices.numpy().astype(np.int64)
    s_q, h_q, _ = q.shape
    out = np.zeros((s_q, h_q, 512))
    lse = np.full((s_q, h_q), -np.inf)
    for i in range(s_q):
        ids = idx[i][(idx[i] >= 0) & (idx[i] < kv.shape[0])]
        if ids.size == 0:
            continue
        K = kv[ids]
        s = q[i] @ K.T * inp.sm_scale
        lnat = scipy.special.logsumexp(s, axis=1)
        out[i] = np.exp(s - lnat[:, None]) @ K[:, :512]
        lse[i] = lnat / LN2
    return out, lse


def run(inp, **kw):
    return oracle.sparse_prefill(inp.q, inp.kv, inp.indices, inp.sm_scale, **kw)


def assert_close(a, b, rtol=1e-12, atol=1e-12):
    a, b = np.asarray(a), np.asarray(b)
    fin = np.isfinite(b)
    assert np.array_equal(np.isfinite(a), fin)
    assert np.array_equal(a[~fin], b[~fin])
    np.testing.assert_allclose(a[fin], b[fin], rtol=rtol, atol=atol)


def tiny(seed, s_q=3, s_kv=150, h_q=3, topk=40, invalid_frac=0.1):
    w = W.PrefillWorkload("t", s_q=s_q, s_kv=s_kv, h_q=h_q, topk=topk, invalid_frac=invalid_frac)
    inp = W.make_prefill_inputs(w, seed=seed)
    # out-of-range ids, negative ids other than -1 and repeats must be handled
    rng = np.random.default_rng(seed)
    idx = inp.indices.numpy().copy()
    for i in range(s_q):
        idx[i, rng.integers(0, topk)] = s_kv + int(rng.integers(0, 5))
        idx[i, rng.integers(0, topk)] = -7
        a, b = rng.integers(0, topk, size=2)
        idx[i, a] = idx[i, b]
    inp.indices = torch.from_numpy(idx)
    return inp


@pytest.mark.parametrize("seed", range(6))
def test_bruteforce_tiny(seed):
    inp = tiny(seed, s_q=1 + seed % 3, h_q=1 + seed % 4, topk=10 + 7 * seed)
    o, l = run(inp)
    o_ref, l_ref = brute_force(inp)
    assert_close(o, o_ref)
    assert_close(l, l_ref)


def test_equals_sparse_decode_over_a_paged_bf16_cache():
    inp = tiny(11, s_q=2, s_kv=200, h_q=4, topk=64)
    # the same rows as a paged cache: page j of the flat KV goes to a random slot of the pool
    n_pages = (inp.kv.shape[0] + 63) // 64
    perm = np.random.default_rng(0).permutation(n_pages)
    cache = torch.zeros((n_pages, 64, 1, 576), dtype=torch.bfloat16)
    flat = torch.zeros((n_pages * 64, 576), dtype=torch.bfloat16)
    flat[:inp.kv.shape[0]] = inp.kv
    for j in range(n_pages):
        cache[perm[j], :, 0] = flat[64 * j:64 * j + 64]
    table = torch.from_numpy(perm.astype(np.int32))[None]
    lens = torch.tensor([inp.kv.shape[0]], dtype=torch.int32)
    o_d, l_d = oracle.mla_decode(inp.q[None], cache, table, lens, inp.sm_scale, indices=inp.indices[None])
    o, l = run(inp)
    # the two restatements divide by the sum at different points: rounding only
    assert_close(o, o_d[0])
    assert_close(l, l_d[0])


def test_single_valid_id_closed_form():
    inp = tiny(3, s_q=2, h_q=2, topk=8, invalid_frac=0.0)
    idx = torch.full((2, 8), -1, dtype=torch.int32)
    idx[0, 5] = 17
    idx[1, 0] = 149
    inp.indices = idx
    o, l = run(inp)
    kv = inp.kv.double().numpy()
    q = inp.q.double().numpy()
    for i, j in ((0, 17), (1, 149)):
        np.testing.assert_array_equal(o[i], np.broadcast_to(kv[j, :512], (2, 512)))
        np.testing.assert_allclose(l[i], (q[i] @ kv[j]) * inp.sm_scale / LN2, rtol=1e-13)


def test_repeated_id_adds_log2_count():
    inp = tiny(4, s_q=1, h_q=3, topk=6, invalid_frac=0.0)
    inp.indices = torch.full((1, 6), 42, dtype=torch.int32)
    o, l = run(inp)
    kv = inp.kv.double().numpy()
    q = inp.q.double().numpy()
    np.testing.assert_allclose(o[0], np.broadcast_to(kv[42, :512], (3, 512)), rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(l[0], (q[0] @ kv[42]) * inp.sm_scale / LN2 + math.log2(6), rtol=1e-13)


def test_no_valid_id_gives_zero_and_minus_inf():
    inp = tiny(5, s_q=2, h_q=2, topk=5)
    inp.indices = torch.tensor([[-1, 150, 10_000, -3, -1], [3, -1, -1, -1, -1]], dtype=torch.int32)
    o, l = run(inp)
    assert np.all(o[0] == 0) and np.all(l[0] == -np.inf)
    assert np.all(np.isfinite(l[1]))


def test_index_order_does_not_matter():
    inp = tiny(6, s_q=3, h_q=2, topk=50)
    o, l = run(inp)
    perm = torch.from_numpy(np.random.default_rng(1).permutation(50))
    inp.indices = inp.indices[:, perm].contiguous()
    o2, l2 = run(inp)
    assert_close(o2, o)
    assert_close(l2, l)


def test_selected_rows_match_all_rows():
    inp = tiny(8, s_q=3, h_q=4, topk=30)
    o, l = run(inp)
    rows = [0, 5, 11, 7]
    o_r, l_r = run(inp, rows=rows)
    np.testing.assert_array_equal(o_r, o.reshape(-1, 512)[rows])
    np.testing.assert_array_equal(l_r, l.reshape(-1)[rows])


MUTATIONS = {
    "out_of_range_kept": ("if (idx[k] < 0 || idx[k] >= j->s_kv) continue;", "if (idx[k] < 0) continue;"),
    "lse_natural_log": ("*lse = (m + log(z)) / log(2.0);\n  /* step 4", "*lse = m + log(z);\n  /* step 4"),
    "query_token_of_row": ("const int64_t i = row / j->h_q;", "const int64_t i = row % j->h_q;"),
    "value_from_rope_end": ("out[d] += w * bf16_bits_to_double(kr[d]);",
                            "out[d] += w * bf16_bits_to_double(kr[d + 64]);"),
    "scale_dropped": ("p[k] = j->sm_scale * acc;", "p[k] = acc;"),
}


def _pins_pass():
    try:
        for seed in range(3):
            inp = tiny(seed, s_q=2, h_q=3, topk=24)
            o, l = run(inp)
            o_ref, l_ref = brute_force(inp)
            assert_close(o, o_ref)
            assert_close(l, l_ref)
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
        assert not _pins_pass(), f"planted mistake '{name}' went unnoticed"
    assert _pins_pass()
