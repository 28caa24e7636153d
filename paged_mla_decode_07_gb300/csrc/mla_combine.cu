// K2 — merge split-KV partial results by their log-sum-exps.
//
// A problem whose keys were split over several parts has, per query row, one
// fp32 partial output o_i (already normalised by its own row sum) and its
// base-2 log-sum-exp lse_i.  The merged row is
//     L = log2 sum_i 2^{lse_i},   out = sum_i 2^{lse_i - L} o_i,   lse = L,
// the same rescaling that online softmax applies across tiles (Modular
// design-doc overview, section 6 "Matmul to Flash Attention"; the FlashMLA
// article, Design 5, pairs split-KV decode with a combine kernel launched
// with programmatic dependent launch).  Partials with lse = -inf contribute
// nothing; a problem with no keys at all gets out = 0, lse = -inf.
//
// One warp per output row; lane l owns dims [16l, 16l + 16).
#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kRowsPerBlock = 4;
constexpr int kFastSplits = 4;  // pieces merged with all loads in flight at once

__global__ void __launch_bounds__(kRowsPerBlock * 32) combine_kernel(const CombineParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int64_t grow = static_cast<int64_t>(blockIdx.x) * kRowsPerBlock + (threadIdx.x >> 5);
  if (grow >= static_cast<int64_t>(p.num_problems) * p.rows) return;
  const int prob = static_cast<int>(grow / p.rows);
  const int r = static_cast<int>(grow % p.rows);
  const int base = p.num_splits[prob];
  const int n = p.num_splits[prob + 1] - base;
  if (n == 0) {
    // a single piece wrote the output directly; a problem without any tile
    // (no keys) was touched by no part: its output is 0, its lse -inf
    if (problem_tiles(p.cache_seqlens, prob, p.s_q, p.topk) > 0) return;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + grow * kDv + lane * 16;
    const uint4 z = make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4*>(out)[0] = z;
    reinterpret_cast<uint4*>(out)[1] = z;
    if (lane == 0) p.lse[grow] = -__int_as_float(0x7f800000);
    return;
  }
  if (base < 0 || n < 2 || base + n > p.max_slots) {
    if (lane == 0) atomicOr(p.status, MLA_DEVICE_BAD_SCHEDULE);
    return;
  }
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + grow * kDv + lane * 16;

  if (n <= kFastSplits) {
    // few pieces (the common case): every load is issued before any is used,
    // so the merge costs two memory round trips instead of one per piece
    float l[kFastSplits];
#pragma unroll
    for (int i = 0; i < kFastSplits; ++i)
      l[i] = i < n ? p.lse_accum[static_cast<int64_t>(base + i) * p.rows + r] : -__int_as_float(0x7f800000);
    float4 x[kFastSplits][4];
#pragma unroll
    for (int i = 0; i < kFastSplits; ++i) {
      if (i < n) {
        const float4* src = reinterpret_cast<const float4*>(p.o_accum + (static_cast<int64_t>(base + i) * p.rows + r) * kDv +
                                                            lane * 16);
#pragma unroll
        for (int v = 0; v < 4; ++v) x[i][v] = src[v];
      }
    }
    float mxf = l[0];
#pragma unroll
    for (int i = 1; i < kFastSplits; ++i) mxf = fmaxf(mxf, l[i]);
    float acc[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[e] = 0.f;
    float Lf = -__int_as_float(0x7f800000);
    if (mxf != -__int_as_float(0x7f800000)) {
      float sum = 0.f;
#pragma unroll
      for (int i = 0; i < kFastSplits; ++i)
        if (i < n) sum += exp2f(l[i] - mxf);
      Lf = mxf + log2f(sum);
#pragma unroll
      for (int i = 0; i < kFastSplits; ++i) {
        if (i < n) {
          const float w = exp2f(l[i] - Lf);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            acc[4 * v + 0] += w * x[i][v].x;
            acc[4 * v + 1] += w * x[i][v].y;
            acc[4 * v + 2] += w * x[i][v].z;
            acc[4 * v + 3] += w * x[i][v].w;
          }
        }
      }
    }
    uint4 o0, o1;
    o0.x = pack_bf16x2(acc[0], acc[1]);
    o0.y = pack_bf16x2(acc[2], acc[3]);
    o0.z = pack_bf16x2(acc[4], acc[5]);
    o0.w = pack_bf16x2(acc[6], acc[7]);
    o1.x = pack_bf16x2(acc[8], acc[9]);
    o1.y = pack_bf16x2(acc[10], acc[11]);
    o1.z = pack_bf16x2(acc[12], acc[13]);
    o1.w = pack_bf16x2(acc[14], acc[15]);
    reinterpret_cast<uint4*>(out)[0] = o0;
    reinterpret_cast<uint4*>(out)[1] = o1;
    if (lane == 0) p.lse[grow] = Lf;
    return;
  }

  float mx = -__int_as_float(0x7f800000);
  for (int i = lane; i < n; i += 32) mx = fmaxf(mx, p.lse_accum[static_cast<int64_t>(base + i) * p.rows + r]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (n <= 0 || mx == -__int_as_float(0x7f800000)) {
    const uint4 z = make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4*>(out)[0] = z;
    reinterpret_cast<uint4*>(out)[1] = z;
    if (lane == 0) p.lse[grow] = -__int_as_float(0x7f800000);
    return;
  }
  float s = 0.f;
  for (int i = lane; i < n; i += 32) s += exp2f(p.lse_accum[static_cast<int64_t>(base + i) * p.rows + r] - mx);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const float L = mx + log2f(s);

  float acc[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) acc[e] = 0.f;
  for (int i = 0; i < n; ++i) {
    const int64_t slot_row = static_cast<int64_t>(base + i) * p.rows + r;
    const float w = exp2f(p.lse_accum[slot_row] - L);
    const float4* src = reinterpret_cast<const float4*>(p.o_accum + slot_row * kDv + lane * 16);
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const float4 x = src[v];
      acc[4 * v + 0] += w * x.x;
      acc[4 * v + 1] += w * x.y;
      acc[4 * v + 2] += w * x.z;
      acc[4 * v + 3] += w * x.w;
    }
  }
  uint4 o0, o1;
  o0.x = pack_bf16x2(acc[0], acc[1]);
  o0.y = pack_bf16x2(acc[2], acc[3]);
  o0.z = pack_bf16x2(acc[4], acc[5]);
  o0.w = pack_bf16x2(acc[6], acc[7]);
  o1.x = pack_bf16x2(acc[8], acc[9]);
  o1.y = pack_bf16x2(acc[10], acc[11]);
  o1.z = pack_bf16x2(acc[12], acc[13]);
  o1.w = pack_bf16x2(acc[14], acc[15]);
  reinterpret_cast<uint4*>(out)[0] = o0;
  reinterpret_cast<uint4*>(out)[1] = o1;
  if (lane == 0) p.lse[grow] = L;
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream, bool pdl) {
  const int64_t rows = static_cast<int64_t>(p.num_problems) * p.rows;
  const unsigned grid = static_cast<unsigned>((rows + kRowsPerBlock - 1) / kRowsPerBlock);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kRowsPerBlock * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, combine_kernel, p);
}

}  // namespace mla
