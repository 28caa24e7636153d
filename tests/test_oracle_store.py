"""Pins of the oracle's FP8 cache write (quantiser and ragged store) against
what the format and a library routine fix: every E4M3 code round-trips, the
rounding agrees with torch's float8_e4m3fn cast (round to nearest even) and
saturates at 448, the dequantised row is within the format's error bound,
and tokens land at cache_lengths[b] + i through the block table."""
import numpy as np
import pytest
import torch

import oracle

E4M3_MAX = 448.0


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


def test_every_finite_code_round_trips():
    for code in range(256):
        if code & 0x7F == 0x7F:  # NaN codes
            continue
        v = oracle.e4m3_to_double(code)
        assert oracle.e4m3_from_float(np.float32(v)) == code, hex(code)


def test_rounding_matches_torch_cast_including_ties():
    rng = np.random.default_rng(5)
    vals = np.concatenate([
        rng.uniform(-E4M3_MAX, E4M3_MAX, 4000),
        rng.uniform(-1, 1, 2000) * 2.0 ** rng.integers(-12, 8, 2000),
    ]).astype(np.float32)
    # exact midpoints between neighbouring positive codes (ties go to the even code)
    pos = [oracle.e4m3_to_double(c) for c in range(0x7F)]
    mids = np.array([(pos[c] + pos[c + 1]) / 2 for c in range(0x7E)], dtype=np.float32)
    vals = np.concatenate([vals, mids, -mids])
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([oracle.e4m3_from_float(v) for v in vals], dtype=np.uint8)
    assert np.array_equal(ours, ref)


def test_saturation_and_specials():
    assert oracle.e4m3_from_float(np.float32(448.0)) == 0x7E
    assert oracle.e4m3_from_float(np.float32(464.0)) == 0x7E   # above the top value: satfinite
    assert oracle.e4m3_from_float(np.float32(1e30)) == 0x7E
    assert oracle.e4m3_from_float(np.float32(-1e30)) == 0xFE
    assert oracle.e4m3_from_float(np.float32(np.nan)) == 0x7F
    assert oracle.e4m3_from_float(np.float32(2.0 ** -10)) == 0x00  # half the smallest step: tie to 0
    assert oracle.e4m3_from_float(np.float32(3 * 2.0 ** -10)) == 0x02  # tie between 1 and 2: even


def _row(x):
    r = oracle.fp8_quantize_row(x)
    codes = r[:512]
    scales = r[512:528].view(np.float32)
    rope = r[528:].view(np.uint16)
    return r, codes, scales, rope


def test_row_layout_scale_and_amax_code():
    g = torch.Generator().manual_seed(3)
    x = (torch.randn(576, generator=g) * 3).to(torch.bfloat16)
    r, codes, scales, rope = _row(x)
    xf = x.float().numpy()
    for t in range(4):
        tile = xf[128 * t:128 * t + 128]
        amax = np.float32(np.abs(tile).max())
        assert scales[t] == np.float32(amax / np.float32(E4M3_MAX))
        k = int(np.abs(tile).argmax())
        assert codes[128 * t + k] & 0x7F == 0x7E            # the largest magnitude maps to 448
    assert np.array_equal(rope, x[512:].view(torch.int16).numpy().view(np.uint16))  # RoPE copied


def test_zero_tile_and_error_bound():
    g = torch.Generator().manual_seed(4)
    x = torch.randn(576, generator=g)
    x[128:256] = 0
    x[256:384] *= 1e-3
    x = x.to(torch.bfloat16)
    r, codes, scales, _ = _row(x)
    assert scales[1] == 1.0 and np.all(codes[128:256] == 0)
    k = oracle.dequant_row(r)
    xf = x.float().numpy().astype(np.float64)
    for t in range(4):
        s = float(scales[t])
        err = np.abs(k[128 * t:128 * t + 128] - xf[128 * t:128 * t + 128])
        # 3 mantissa bits: half an ulp is 2^-4 relative; subnormal codes have step 2^-9 * scale;
        # the final bf16 rounding of the dequantised value adds 2^-9 relative
        bound = np.abs(xf[128 * t:128 * t + 128]) * (2.0 ** -4 + 2.0 ** -8) + s * 2.0 ** -10
        assert np.all(err <= bound + 1e-30)
    assert np.array_equal(k[512:], xf[512:])


def test_ragged_store_routes_through_the_block_table():
    g = torch.Generator().manual_seed(9)
    pages, psize = 12, 64
    table = torch.tensor([[3, 7, 1, -1], [0, 5, 11, 99]], dtype=torch.int32)
    lens = torch.tensor([188, 128], dtype=torch.int32)
    offs = torch.tensor([0, 10, 75], dtype=torch.int32)          # 10 and 65 new tokens
    x = torch.randn(75, 576, generator=g).to(torch.bfloat16)
    cache = torch.randint(0, 256, (pages, psize, 1, 656), generator=g, dtype=torch.uint8)
    new, skipped = oracle.fp8_cache_store(x, offs, lens, table, cache)
    # element 0: positions 188..197, block 3 is -1 -> 6 skipped (and it crosses a page boundary);
    # element 1: positions 128..192, position 192 maps to page 99, outside the pool -> 1 skipped
    assert skipped == 7
    old = cache.numpy()
    touched = set()
    for b in range(2):
        for i in range(int(offs[b + 1] - offs[b])):
            pos = int(lens[b]) + i
            page = int(table[b, pos // psize]) if pos // psize < table.shape[1] else -1
            if not 0 <= page < pages:
                continue
            touched.add((page, pos % psize))
            assert np.array_equal(new[page, pos % psize, 0], oracle.fp8_quantize_row(x[int(offs[b]) + i]))
    for p in range(pages):
        for s in range(psize):
            if (p, s) not in touched:
                assert np.array_equal(new[p, s], old[p, s])
