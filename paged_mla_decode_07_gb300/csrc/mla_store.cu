// K3 — FP8 KV-cache write: new tokens (576 bf16 values each) quantised into
// the 656-byte cache row and written through the block table.
//
// The row format follows the FlashMLA article (Design 2): the 512 NoPE dims
// become float8_e4m3 codes in four 1 x 128 tiles, each with one float32
// scale = amax / 448 (1 for an all-zero tile), code = E4M3 of x / scale
// rounded to nearest even and saturated at 448; the 64 RoPE dims are copied
// as bf16.  Placement follows the MAX kernels summary (KV-cache store): the
// new tokens of batch element b, rows input_row_offsets[b] ..
// input_row_offsets[b+1]-1 of x, go to logical positions cache_lengths[b] +
// i, i.e. page block_table[b][pos / 64], slot pos % 64.
//
// One warp per token: lane l holds NoPE dims [16l, 16l+16) (a tile is eight
// lanes; its amax is a three-step shuffle), lanes 0..7 the RoPE dims.  Each
// lane reads 32 + 16 bytes and writes 16 + 16 bytes with 16-byte accesses.
// Memory-bound: 1152 bytes read and 656 written per token.
#include <cuda_bf16.h>

#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kStoreWarps = 8;  // warps per block

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two floats -> two E4M3 codes (round to nearest even, saturating), low byte = lo.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Quantise one token (this lane's 16 NoPE values a, c and, for lanes 0..7,
// 8 RoPE values rp) into the row at dst.
__device__ __forceinline__ void store_row(uint8_t* dst, const uint4 a, const uint4 c, const uint4 rp, int lane) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
  float v[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = bf16_lo(w[i]);
    v[2 * i + 1] = bf16_hi(w[i]);
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
  for (int o = 4; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float scale = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  uint32_t code[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    code[i] = e4m3x2(__fdiv_rn(v[4 * i], scale), __fdiv_rn(v[4 * i + 1], scale)) |
              (e4m3x2(__fdiv_rn(v[4 * i + 2], scale), __fdiv_rn(v[4 * i + 3], scale)) << 16);
  *reinterpret_cast<uint4*>(dst + 16 * lane) = make_uint4(code[0], code[1], code[2], code[3]);
  // scales: tile t is held by lanes 8t .. 8t+7
  const float s0 = __shfl_sync(0xffffffffu, scale, 0), s1 = __shfl_sync(0xffffffffu, scale, 8);
  const float s2 = __shfl_sync(0xffffffffu, scale, 16), s3 = __shfl_sync(0xffffffffu, scale, 24);
  if (lane == 0)
    *reinterpret_cast<uint4*>(dst + kFp8ScaleOffset) =
        make_uint4(__float_as_uint(s0), __float_as_uint(s1), __float_as_uint(s2), __float_as_uint(s3));
  if (lane < 8) *reinterpret_cast<uint4*>(dst + kFp8RopeOffset + 16 * lane) = rp;
}

// Each warp takes a contiguous range of token rows (one search for its first
// batch element, then advanced as rows cross element boundaries) and handles
// two rows per step, loading both rows before resolving their pages so the
// loads overlap the block-table lookups.
__global__ void __launch_bounds__(kStoreWarps * 32)
    fp8_store_kernel(const uint16_t* __restrict__ x, int num_tokens, const int32_t* __restrict__ row_offsets,
                     const int32_t* __restrict__ cache_lengths, int batch, const int32_t* __restrict__ block_table,
                     int block_table_stride, uint8_t* __restrict__ kvcache, int num_pages, uint32_t* status) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * kStoreWarps;
  const int64_t wid = static_cast<int64_t>(blockIdx.x) * kStoreWarps + (threadIdx.x >> 5);
  const int64_t per = (num_tokens + warps - 1) / warps;
  const int r0 = static_cast<int>(wid * per);
  const int r1 = static_cast<int>(((static_cast<int64_t>(r0) + per < num_tokens) ? static_cast<int64_t>(r0) + per : static_cast<int64_t>(num_tokens)));
  if (r0 >= r1) return;
  // batch element of row r0: the last b with row_offsets[b] <= r0
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(row_offsets + mid) <= r0)
      lo = mid;
    else
      hi = mid - 1;
  }
  int b = lo;
  int off_b = __ldg(row_offsets + b), off_n = __ldg(row_offsets + b + 1), len_b = __ldg(cache_lengths + b);
  // destination of row r (advances b while r is past the element's rows)
  auto dest = [&](int r) -> uint8_t* {
    while (r >= off_n && b + 1 < batch) {
      ++b;
      off_b = off_n;
      off_n = __ldg(row_offsets + b + 1);
      len_b = __ldg(cache_lengths + b);
    }
    const int64_t pos = static_cast<int64_t>(len_b) + (r - off_b);
    const int64_t blk = pos / kPageSize;
    const int page = (pos >= 0 && blk < block_table_stride)
                         ? __ldg(block_table + static_cast<int64_t>(b) * block_table_stride + blk)
                         : -1;
    if (page < 0 || page >= num_pages) {
      if (lane == 0) atomicOr(status, MLA_DEVICE_BAD_PAGE);
      return nullptr;
    }
    return kvcache + (static_cast<int64_t>(page) * kPageSize + pos % kPageSize) * kFp8RowBytes;
  };
  for (int r = r0; r < r1; r += 2) {
    const bool two = r + 1 < r1;
    const uint16_t* s0 = x + static_cast<int64_t>(r) * kDqk;
    const uint16_t* s1 = s0 + kDqk;
    const uint4 a0 = ld_global_nc_v4(s0 + 16 * lane), c0 = ld_global_nc_v4(s0 + 16 * lane + 8);
    const uint4 p0 = lane < 8 ? ld_global_nc_v4(s0 + kDv + 8 * lane) : make_uint4(0, 0, 0, 0);
    uint4 a1 = make_uint4(0, 0, 0, 0), c1 = a1, p1 = a1;
    if (two) {
      a1 = ld_global_nc_v4(s1 + 16 * lane);
      c1 = ld_global_nc_v4(s1 + 16 * lane + 8);
      if (lane < 8) p1 = ld_global_nc_v4(s1 + kDv + 8 * lane);
    }
    uint8_t* d0 = dest(r);
    uint8_t* d1 = two ? dest(r + 1) : nullptr;
    if (d0) store_row(d0, a0, c0, p0, lane);
    if (d1) store_row(d1, a1, c1, p1, lane);
  }
}

}  // namespace

cudaError_t launch_fp8_cache_store(const uint16_t* x, int num_tokens, const int32_t* row_offsets,
                                   const int32_t* cache_lengths, int batch, const int32_t* block_table,
                                   int block_table_stride, uint8_t* kvcache, int num_pages, uint32_t* status,
                                   int sm_count, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int blocks_needed = (num_tokens + kStoreWarps - 1) / kStoreWarps;
  const int grid = blocks_needed < sm_count * 8 ? blocks_needed : sm_count * 8;
  fp8_store_kernel<<<grid, kStoreWarps * 32, 0, stream>>>(x, num_tokens, row_offsets, cache_lengths, batch,
                                                           block_table, block_table_stride, kvcache, num_pages,
                                                           status);
  return cudaGetLastError();
}

}  // namespace mla
