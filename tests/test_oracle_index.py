"""Pins for the oracle's FP8 top-k indexer, each against something other than itself:

* an independent numpy brute force (torch's float8_e4m3fn cast to decode
  the codes, einsum for the head dots, lexsort for the selection) on small
  ragged, paged inputs, with and without ReLU;
* closed forms: equal scores select the smallest ids in order, fewer visible
  keys than k fill with -1, the visible-key count follows the causal rule,
  scaling every key scale by 2 doubles the scores and keeps the selection;
* planted mistakes in a copy of the oracle source must fail a pin.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from paged_mla_decode_07_gb300 import workloads as W


def decode_e4m3(codes: torch.Tensor) -> np.ndarray:
    return codes.contiguous().view(torch.float8_e4m3fn).to(torch.float64).numpy()


def brute_scores(inp):
    q = decode_e4m3(inp.q_codes)                           # [T, h, 128]
    kc = decode_e4m3(inp.k_codes.reshape(-1, 128))         # [rows, 128]
    qs = inp.q_scales.double().numpy()
    ks = inp.k_scales.reshape(-1).double().numpy()
    w = inp.weights.double().numpy()
    offs = inp.row_offsets.numpy()
    lens = inp.cache_seqlens.numpy()
    table = inp.block_table.numpy()
    width = int(max(1, lens.max()))
    out = np.full((offs[-1], width), -np.inf)
    for b in range(len(lens)):
        n_b = offs[b + 1] - offs[b]
        for j in range(n_b):
            t = offs[b] + j
            vis = min(int(lens[b]) - n_b + j + 1, int(lens[b]))
            if vis <= 0:
                continue
            s = np.arange(vis)
            rows = table[b, s // 64].astype(np.int64) * 64 + s % 64
            dots = np.einsum("hd,sd->hs", q[t], kc[rows]) * qs[t][:, None] * ks[rows][None, :]
            if inp.relu:
                dots = np.maximum(dots, 0.0)
            out[t, :vis] = w[t] @ dots
    return out


def brute_topk(scores, k):
    out = np.full((scores.shape[0], k), -1, np.int32)
    for t in range(scores.shape[0]):
        vis = np.flatnonzero(np.isfinite(scores[t]))
        order = vis[np.lexsort((vis, -scores[t, vis]))]
        out[t, :min(k, len(order))] = order[:k]
    return out


def small(seed, lens=(200, 77, 130), n_new=2, h=4, topk=40, relu=False):
    w = W.IndexWorkload("s", batch=len(lens), n_new=n_new, h_idx=h, topk=topk, seqlens=tuple(lens), relu=relu)
    return W.make_index_inputs(w, seed=seed)


@pytest.mark.parametrize("seed,relu", [(0, False), (1, True), (2, False), (3, True)])
def test_bruteforce(seed, relu):
    inp = small(seed, relu=relu, n_new=1 + seed % 3)
    s = oracle.index_scores(inp)
    ref = brute_scores(inp)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(s), fin)
    np.testing.assert_allclose(s[fin], ref[fin], rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(oracle.index_topk(inp), brute_topk(ref, inp.topk))


def test_equal_scores_select_smallest_ids_in_order():
    inp = small(5, lens=(150,), n_new=1, h=2, topk=20)
    inp.k_codes[:] = inp.k_codes[0, 0]                     # every key identical
    inp.k_scales[:] = 0.5
    np.testing.assert_array_equal(oracle.index_topk(inp)[0], np.arange(20))


def test_fewer_visible_keys_than_k_fill_minus_one():
    inp = small(6, lens=(30, 5), n_new=3, h=2, topk=40)
    top = oracle.index_topk(inp)
    for b, L in enumerate((30, 5)):
        for j in range(3):
            vis = L - 3 + j + 1
            row = top[3 * b + j]
            assert np.all(row[vis:] == -1) and sorted(row[:vis].tolist()) == list(range(vis))


def test_key_scale_linearity():
    inp = small(7, relu=True)
    s1, t1 = oracle.index_scores(inp), oracle.index_topk(inp)
    inp.k_scales.mul_(2.0)
    s2, t2 = oracle.index_scores(inp), oracle.index_topk(inp)
    fin = np.isfinite(s1)
    np.testing.assert_allclose(s2[fin], 2 * s1[fin], rtol=1e-13)
    np.testing.assert_array_equal(t1, t2)


def test_relu_clips_each_head_before_the_weighted_sum():
    inp = small(8, lens=(64,), n_new=1, h=3, topk=5, relu=True)
    inp.weights[:] = torch.tensor([1.0, -1.0, 0.5])
    ref = brute_scores(inp)
    s = oracle.index_scores(inp)
    np.testing.assert_allclose(s, ref, rtol=1e-12, atol=1e-12)
    inp.relu = False
    assert not np.allclose(oracle.index_scores(inp), s)


MUTATIONS = {
    "ties_to_larger_id": ("if (best < 0 || sc[s] > sc[best]) best = s;",
                          "if (best < 0 || sc[s] >= sc[best]) best = s;"),
    "causal_off_by_one": ("int64_t last = L - n_b + j;", "int64_t last = L - n_b + j - 1;"),
    "key_scale_dropped": ("(double)p->q_scales[t * p->h_idx + h] * (double)p->k_scales[row] * dot;",
                          "(double)p->q_scales[t * p->h_idx + h] * dot;"),
    "relu_after_weight": ("acc += (double)p->weights[t * p->h_idx + h] * v;",
                          "acc += (p->relu && p->weights[t * p->h_idx + h] < 0) ? 0.0 : (double)p->weights[t * p->h_idx + h] * v;"),
    "page_slot_swapped": ("const int64_t row = (int64_t)page * p->page_size + s % p->page_size;",
                          "const int64_t row = (int64_t)page * p->page_size + (s + 1) % p->page_size;"),
}


def _pins_pass():
    try:
        for seed, relu in ((0, False), (1, True)):
            inp = small(seed, relu=relu)
            ref = brute_scores(inp)
            s = oracle.index_scores(inp)
            fin = np.isfinite(ref)
            assert np.array_equal(np.isfinite(s), fin)
            np.testing.assert_allclose(s[fin], ref[fin], rtol=1e-12, atol=1e-12)
            np.testing.assert_array_equal(oracle.index_topk(inp), brute_topk(ref, inp.topk))
        test_equal_scores_select_smallest_ids_in_order()
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
