"""Parity of the FP8 cache write (mla_fp8_cache_store, through the C ABI) with
the oracle: the written rows must be byte-identical (integer/byte work), and
untouched rows must keep their bytes."""
import numpy as np
import pytest
import torch

import oracle
import paged_mla_decode_07_gb300 as mla

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mla.build()
    oracle.build()


def _case(seed, lens, new, pages, stride, scale=1.0, specials=False):
    g = torch.Generator().manual_seed(seed)
    batch = len(lens)
    offs = torch.tensor(np.concatenate([[0], np.cumsum(new)]), dtype=torch.int32)
    x = (torch.randn(int(offs[-1]), 576, generator=g) * scale)
    if specials and x.shape[0] >= 4:
        x[0, :128] = 0                        # all-zero tile: scale 1, codes 0
        x[1, 128:256] *= 1e-6                 # tiny values: subnormal codes
        x[2, 256:384] = 3.0                   # constant tile: every code 448
        x[3, ::7] *= -1
    x = x.to(torch.bfloat16)
    perm = torch.randperm(pages, generator=g).int()
    table = torch.full((batch, stride), -1, dtype=torch.int32)
    k = 0
    for b in range(batch):
        need = (lens[b] + new[b] + 63) // 64
        for j in range(min(need, stride)):
            table[b, j] = perm[k % pages]
            k += 1
    cache = torch.randint(0, 256, (pages, 64, 1, 656), generator=g, dtype=torch.uint8)
    return x, offs, torch.tensor(lens, dtype=torch.int32), table, cache


def _run(x, offs, lens, table, cache):
    ref, skipped = oracle.fp8_cache_store(x, offs, lens, table, cache)
    c = cache.cuda()
    mla.device_status()
    mla.fp8_cache_store(x.cuda(), offs.cuda(), lens.cuda(), table.cuda(), c)
    flags = mla.device_status()
    return c.cpu().numpy(), ref, skipped, flags


@pytest.mark.parametrize("lens,new", [
    ([0], [1]),                                   # first token of an empty sequence
    ([63, 64, 65], [1, 1, 1]),                    # one decode token at page edges
    ([100, 0, 4000], [300, 64, 129]),             # ragged prefill chunks crossing pages
    ([5, 7], [0, 200]),                           # an element with no new tokens
])
def test_store_matches_oracle_bytes(lens, new):
    pages = sum((l + n + 63) // 64 for l, n in zip(lens, new)) + 3
    x, offs, lens_t, table, cache = _case(17 + sum(new), lens, new, pages, stride=80, specials=True)
    got, ref, skipped, flags = _run(x, offs, lens_t, table, cache)
    assert skipped == 0 and flags == 0
    assert np.array_equal(got, ref)


def test_store_large_values_and_many_tokens():
    lens, new = [1000] * 8, [513] * 8
    pages = sum((l + n + 63) // 64 for l, n in zip(lens, new))
    x, offs, lens_t, table, cache = _case(5, lens, new, pages, stride=32, scale=1e4)
    got, ref, skipped, flags = _run(x, offs, lens_t, table, cache)
    assert skipped == 0 and flags == 0
    assert np.array_equal(got, ref)


def test_store_skips_missing_pages_and_flags_them():
    x, offs, lens_t, table, cache = _case(8, [60, 10], [10, 10], 4, stride=2)
    table[0, 1] = -1          # element 0 crosses into a missing page
    table[1, 0] = 99          # element 1's page is outside the pool
    got, ref, skipped, flags = _run(x, offs, lens_t, table, cache)
    assert skipped == 6 + 10
    assert flags & mla.DEVICE_BAD_PAGE
    assert np.array_equal(got, ref)


def test_store_then_sparse_decode_reads_the_rows():
    """Tokens written by the store and then gathered by the sparse decode give the oracle's result."""
    from paged_mla_decode_07_gb300 import workloads as W
    w = W.custom(name="st", batch=2, h_q=64, s_q=1, mode="sparse", seqlens=(300, 129), topk=256)
    inp = W.make_inputs(w, seed=41, poison_tail=False)
    g = torch.Generator().manual_seed(2)
    # rewrite the last 100 / 29 tokens of each element with freshly quantised values
    lens = torch.tensor([200, 100], dtype=torch.int32)
    offs = torch.tensor([0, 100, 129], dtype=torch.int32)
    x = torch.randn(129, 576, generator=g).to(torch.bfloat16)
    c = inp.kvcache.clone().cuda()
    mla.fp8_cache_store(x.cuda(), offs.cuda(), lens.cuda(), inp.block_table.cuda(), c)
    inp.kvcache = c.cpu()
    d = inp.to("cuda")
    sched, ns = mla.get_metadata(d.cache_seqlens, h_q=w.h_q, s_q=w.s_q, topk=256, is_fp8=True)
    out, lse = mla.decode(d.q, d.kvcache, d.block_table, d.cache_seqlens, d.sm_scale, sched, ns, indices=d.indices)
    ref_out, ref_lse = oracle.mla_decode(inp.q, inp.kvcache, inp.block_table, inp.cache_seqlens, inp.sm_scale,
                                         indices=inp.indices)
    from gpu_helpers import compare
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out.reshape(out.shape),
            ref_lse.reshape(lse.shape), "store+decode")


def _boundary_tokens(n_tokens, seed):
    """Tokens whose tiles put quotients x / scale on and next to E4M3 rounding
    boundaries: each tile holds its amax (a bf16 value) and values x with
    448 x / amax equal to a midpoint between two E4M3 values.  With a scale
    amax / 448 that rounds in float32, the quotient lands within a float32
    ulp of the midpoint, on either side; with an exact scale, on it (a tie)."""
    rng = np.random.default_rng(seed)
    vals = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    mids = (vals[:-1] + vals[1:]) / 2
    amaxes = [1.0, 1.5, 2.5, 0.75, 100.0, 3e-3, 448.0, 1344.0, 5.0, 0.3]
    x = np.zeros((n_tokens, 576))
    near = ties = 0
    for t in range(n_tokens):
        for tile in range(4):
            amax = float(torch.tensor(amaxes[(4 * t + tile) % len(amaxes)] * (1 + 0.01 * rng.integers(0, 8)))
                         .to(torch.bfloat16))
            scale = np.float32(amax) / np.float32(448.0)
            cand = amax * mids / 448.0
            exact = torch.tensor(cand).to(torch.bfloat16).double().numpy() == cand
            pick = cand[exact & (cand <= amax)]
            row = rng.uniform(-amax, amax, 128)
            row[0] = amax
            k = min(len(pick), 127)
            row[1:1 + k] = pick[rng.permutation(len(pick))[:k]] * rng.choice([-1.0, 1.0], k)
            x[t, 128 * tile:128 * tile + 128] = row
            q = np.abs(np.float32(row[1:1 + k]) / scale).astype(np.float64)
            m = np.abs(row[1:1 + k]) * 448.0 / amax
            near += int(np.sum((q != m) & (np.abs(q - m) <= m * 2.0 ** -21)))
            ties += int(np.sum(q == m))
        x[t, 512:] = rng.standard_normal(64)
    return torch.tensor(x).to(torch.bfloat16), near, ties


def test_store_values_at_e4m3_rounding_boundaries():
    """Quotients on (ties to the even code) and within a float32 ulp of E4M3
    rounding boundaries quantise exactly as the float32 division decides."""
    n = 256
    x, near, ties = _boundary_tokens(n, seed=11)
    assert near > 100 and ties > 1000         # the data does reach both kinds of boundary case
    offs = torch.tensor([0, n], dtype=torch.int32)
    lens = torch.tensor([0], dtype=torch.int32)
    table = torch.arange(n // 64, dtype=torch.int32)[None]
    cache = torch.zeros((n // 64, 64, 1, 656), dtype=torch.uint8)
    got, ref, skipped, flags = _run(x, offs, lens, table, cache)
    assert skipped == 0 and flags == 0
    assert np.array_equal(got, ref)
