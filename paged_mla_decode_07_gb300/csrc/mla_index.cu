// K4 + K5 — FP8 top-k indexer (MAX kernels summary, MLA indexing kernels:
// mla_fp8_index_top_k scores FP8 queries against a quantised, paged key
// cache with their scales, aggregates over the index heads, masks, and keeps
// the top-k key ids per query token as int32, -1 in unused slots).
//
//   score(t, s) = sum_h w[t,h] * f(qs[t,h] * ks[s] * sum_d q[t,h,d] k[s,d])
//   f = ReLU or identity; query row j of element b (n_b new rows, the last
//   n_b positions of a cache of L_b) sees keys s <= L_b - n_b + j.
//
// K4 index_score_kernel: one CTA per (element, run of 128-key tiles).  The
// head dots of a tile are one tcgen05 kind::f8f6f4 contraction
//     D[key, row] = K[key, :] . Q[row, :]    M = 128 keys, N = n_b * h rows, K = 128
// with E4M3 operands in shared memory (128-byte rows, 128-byte swizzle,
// loaded by TMA) and the fp32 accumulator in TMEM (two buffers, so the
// epilogue of one tile overlaps the MMAs of the next).  The epilogue (one
// thread per key) applies the scales, f and the head weights and writes one
// fp32 score per (query row, key).  The contraction streams the key cache
// once per element; its arithmetic intensity (2 * N FLOP per 132-byte key)
// stays under the FP8 ridge, so the kernel is bounded by HBM.
//
// K5 index_topk_kernel: one CTA of 1024 threads per query row: radix select
// (four 8-bit passes over order-preserving integer images of the scores)
// finds the k-th largest score, the keys above it and the first ties in key
// order are collected, and a bitonic sort orders them by (score desc, id asc).
//
// Every mbarrier wait is bounded (watchdog); on expiry the CTA records
// MLA_DEVICE_TIMEOUT, drains its own copies and MMAs and frees TMEM.
#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kIdxDim = 128;                          // index head dimension (bytes per E4M3 row)
constexpr int kKeysPerTile = 128;                     // M of the MMA: two pages
constexpr int kStages = 4;                            // key tiles in flight
constexpr int kTileBytes = kKeysPerTile * kIdxDim;    // 16 KB
constexpr int kMaxRows = 256;                         // N of the MMA (query rows x heads of one element)
constexpr int kScoreThreads = 384;                    // warp 0 TMA, 1 MMA, 2 TMEM, 4..11 epilogue
constexpr int kEpiWarps = 8;                          // two per TMEM lane quarter: they split the query rows
constexpr int kQOff = kStages * kTileBytes;
constexpr int kBarOff = kQOff + kMaxRows * kIdxDim;
constexpr int kNumBars = 2 * kStages + 4 + 2;         // full, empty, d_full[2], d_empty[2], q_full, done
constexpr int kAuxOff = kBarOff + kNumBars * 8;       // qs[kMaxRows], w[kMaxRows], ints
constexpr int kScoreSmem = kAuxOff + 2 * kMaxRows * 4 + 64 + 1024;
static_assert(kAuxOff % 16 == 0, "w * qs must be 16-byte aligned for vector loads");

// kind::f8f6f4 instruction descriptor: D f32 (bits 4-5 = 1), A and B E4M3
// (format 0 in bits 7-9 and 10-12), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__device__ __forceinline__ uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void umma_e4m3_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Warp-uniform bounded wait: if any lane fails, every lane sees failure.
__device__ __forceinline__ bool warp_wait_any(uint64_t* bar, uint32_t parity, const Watchdog& wd) {
  const bool ok = mbar_wait(bar, parity, wd);
  return __all_sync(0xffffffffu, ok);
}

// Bounded wait that ignores the abort flag (used to drain own async work).
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > limit_ns) return false;
  return true;
}

// With positive scales (the quantiser's amax / 448, or 1) a head's term is
// w * f(qs * ks * dot) = ks * (w * qs) * f(dot), f = ReLU or identity: the
// epilogue multiplies each dot by the per-row factor w * qs (kept in shared
// memory) and the sum by the key's scale once.
template <bool RELU, bool H64>
__global__ void __launch_bounds__(kScoreThreads, 2)
    index_score_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const IndexParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint8_t* qs = smem + kQOff;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* full = bar;
  uint64_t* empty = bar + kStages;
  uint64_t* d_full = bar + 2 * kStages;
  uint64_t* d_empty = d_full + 2;
  uint64_t* q_full = d_empty + 2;
  uint64_t* done = q_full + 1;
  float* wq = reinterpret_cast<float*>(smem + kAuxOff);  // w * qs per query row x head (16-byte aligned)
  int* ints = reinterpret_cast<int*>(wq + 2 * kMaxRows);
  volatile int* abort_flag = ints;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ints + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.y;
  const int r0 = p.row_offsets[b];
  const int n_b = p.row_offsets[b + 1] - r0;
  const int L = p.cache_seqlens[b];
  const int nrows = n_b * p.h_idx;
  if (n_b <= 0 || L <= 0) return;
  if (n_b > p.max_new) {
    if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(p.status, MLA_DEVICE_BAD_SCHEDULE);
    return;
  }
  const int ntiles = (L + kKeysPerTile - 1) / kKeysPerTile;
  const int tb = blockIdx.x * p.tiles_per_cta;
  const int te = min(ntiles, tb + p.tiles_per_cta);
  if (tb >= te) return;
  const int N = (nrows + 15) & ~15;  // MMA N: a multiple of 16 (rows past nrows are ignored)

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(d_full + i, 1);
      mbar_init(d_empty + i, kEpiWarps);  // one arrival per epilogue warp
    }
    mbar_init(q_full, 1);
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  for (int i = threadIdx.x; i < nrows; i += kScoreThreads) {
    wq[i] = p.weights[static_cast<int64_t>(r0) * p.h_idx + i] * p.q_scales[static_cast<int64_t>(r0) * p.h_idx + i];
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t dcols = p.tmem_cols / 2;  // columns of one accumulator buffer
  Watchdog wd{abort_flag, p.status, p.timeout_ns};
  // the top-k kernel (a programmatic dependent of this one) may be scheduled
  // once every CTA of this grid has started: its blocks take the SMs that
  // the last wave frees and wait (griddepcontrol.wait) for this grid to end
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int32_t* bt = p.block_table + static_cast<int64_t>(b) * p.block_table_stride;

  if (warp == 0) {
    // ---- producer: Q rows of the element once, then the key tiles
    const uint64_t pol = l2_policy_evict_first();
    int uses[kStages] = {0, 0, 0, 0};
    bool q_armed = false;
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(p.n_box) * kIdxDim);
      tma_load_2d(qs, &tm_q, q_full, 0, r0 * p.h_idx, l2_policy_evict_normal());
    }
    q_armed = true;
    __syncwarp();
    for (int t = tb, i = 0; t < te; ++t, ++i) {
      const int st = i % kStages;
      if (i >= kStages && !warp_wait_any(empty + st, static_cast<uint32_t>((i / kStages) - 1) & 1u, wd)) break;
      int pages[2];
      uint32_t bytes = 0;
      for (int pg = 0; pg < 2; ++pg) {
        const int jp = 2 * t + pg;
        pages[pg] = -1;
        if (jp * kPageSize < L && jp < p.block_table_stride) {
          const int id = bt[jp];
          if (id >= 0 && id < p.num_pages) {
            pages[pg] = id;
            bytes += kPageSize * kIdxDim;
          } else if (lane == 0) {
            atomicOr(p.status, MLA_DEVICE_BAD_PAGE);
          }
        }
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(full + st, bytes);
        for (int pg = 0; pg < 2; ++pg)
          if (pages[pg] >= 0)
            tma_load_2d(ring + st * kTileBytes + pg * (kPageSize * kIdxDim), &tm_k, full + st, 0,
                        pages[pg] * kPageSize, pol);
      }
      ++uses[st];
      __syncwarp();
    }
    // drain (bounded): the latest armed phase of every stage and Q
    if (lane == 0) {
      for (int st = 0; st < kStages; ++st)
        if (uses[st] > 0) mbar_wait_drain(full + st, static_cast<uint32_t>(uses[st] - 1) & 1u, wd.limit_ns);
      if (q_armed) mbar_wait_drain(q_full, 0, wd.limit_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- MMA issuer (converged warp, elected lane)
    const uint32_t idesc = idesc_e4m3_f32(kKeysPerTile, N);
    const uint64_t hi = smem_desc_hi(16, 1024);
    const uint32_t ringb = smem_u32(ring), qb = smem_u32(qs);
    bool ok = warp_wait_any(q_full, 0, wd);
    tc_fence_after();
    for (int t = tb, i = 0; ok && t < te; ++t, ++i) {
      const int st = i % kStages, db = i & 1;
      if (i >= 2 && !warp_wait_any(d_empty + db, static_cast<uint32_t>((i >> 1) - 1) & 1u, wd)) break;
      if (!warp_wait_any(full + st, static_cast<uint32_t>(i / kStages) & 1u, wd)) break;
      tc_fence_after();
      const uint64_t a0 = hi | ((ringb + st * kTileBytes) >> 4);
      const uint64_t b0 = hi | (qb >> 4);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {  // K = 32 E4M3 values (32 bytes) per MMA
        if (elect_one()) umma_e4m3_ss(tmem + db * dcols, a0 + 2 * kk, b0 + 2 * kk, idesc, kk != 0);
        __syncwarp();
      }
      if (elect_one()) {
        umma_commit(empty + st);
        umma_commit(d_full + db);
      }
      __syncwarp();
    }
    // drain: every MMA issued by this warp has completed
    if (elect_one()) umma_commit(done);
    __syncwarp();
    if (lane == 0) mbar_wait_drain(done, 0, wd.limit_ns);
    __syncwarp();
  } else if (warp >= 4) {
    // ---- epilogue: thread = key of the tile (TMEM lane); the two warps of a
    // lane quarter take alternate query rows
    const int q4 = warp & 3;
    const int eg = (warp - 4) >> 2;
    const int kt = 32 * q4 + lane;  // key within the tile
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    // The key's page (block table) and scale: two dependent global reads,
    // software-pipelined three and two tiles ahead so that their latency is
    // not paid per tile.  -1: no page (past the keys or the table, or a bad
    // id, which the producer flags).
    auto page_of = [&](int tt) -> int {
      const int key = tt * kKeysPerTile + kt;
      const int jp = key >> 6;
      if (tt >= te || key >= L || jp >= p.block_table_stride) return -1;
      const int id = bt[jp];
      return (id >= 0 && id < p.num_pages) ? id : -1;
    };
    auto scale_of = [&](int id, int tt) -> float {
      return id >= 0 ? p.k_scales[static_cast<int64_t>(id) * kPageSize + ((tt * kKeysPerTile + kt) & 63)] : 0.f;
    };
    int pg0 = page_of(tb), pg1 = page_of(tb + 1), pg2 = page_of(tb + 2);
    float ks0 = scale_of(pg0, tb), ks1 = scale_of(pg1, tb + 1);
    for (int t = tb, i = 0; t < te; ++t, ++i) {
      const int db = i & 1;
      if (!warp_wait_any(d_full + db, static_cast<uint32_t>(i >> 1) & 1u, wd)) break;
      tc_fence_after();
      const int key = t * kKeysPerTile + kt;
      // this tile's page and scale were read ahead; start the reads for the
      // tiles two (scale) and three (page) ahead
      const int page = pg0;
      const float ks = ks0;
      pg0 = pg1;
      pg1 = pg2;
      ks0 = ks1;
      ks1 = scale_of(pg1, t + 2);
      pg2 = page_of(t + 3);
      const uint32_t dbase = tmem + lane_base + db * dcols;
      for (int j = eg; j < n_b; j += 2) {
        float acc = 0.f;
        if (H64) {
          // 64 heads: two full 32-column reads, factors read before the FMAs
          float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int h0 = 0; h0 < 64; h0 += 32) {
            float v[32];
            tmem_ld_x32(dbase + j * 64 + h0, v);
            const float4* w4 = reinterpret_cast<const float4*>(wq + j * 64 + h0);
            tmem_ld_wait();
#pragma unroll
            for (int g = 0; g < 2; ++g) {
              float4 w[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) w[k] = w4[4 * g + k];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const int c = 16 * g + 4 * k;
                a[0] = fmaf(w[k].x, RELU ? fmaxf(v[c], 0.f) : v[c], a[0]);
                a[1] = fmaf(w[k].y, RELU ? fmaxf(v[c + 1], 0.f) : v[c + 1], a[1]);
                a[2] = fmaf(w[k].z, RELU ? fmaxf(v[c + 2], 0.f) : v[c + 2], a[2]);
                a[3] = fmaf(w[k].w, RELU ? fmaxf(v[c + 3], 0.f) : v[c + 3], a[3]);
              }
            }
          }
          acc = (a[0] + a[1]) + (a[2] + a[3]);
        }
        for (int h0 = 0; !H64 && h0 < p.h_idx; h0 += 32) {
          // up to 32 columns per wait (h_idx is a multiple of 8)
          const int nc = min(32, p.h_idx - h0);
          float v[32];
          tmem_ld_x8(dbase + j * p.h_idx + h0, *reinterpret_cast<float(*)[8]>(v));
          if (nc > 8) tmem_ld_x8(dbase + j * p.h_idx + h0 + 8, *reinterpret_cast<float(*)[8]>(v + 8));
          if (nc > 16) tmem_ld_x8(dbase + j * p.h_idx + h0 + 16, *reinterpret_cast<float(*)[8]>(v + 16));
          if (nc > 24) tmem_ld_x8(dbase + j * p.h_idx + h0 + 24, *reinterpret_cast<float(*)[8]>(v + 24));
          tmem_ld_wait();
          const float4* w4 = reinterpret_cast<const float4*>(wq + j * p.h_idx + h0);
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            if (e < nc) {
              const float4 w = w4[e >> 2];
              acc = fmaf(w.x, RELU ? fmaxf(v[e], 0.f) : v[e], acc);
              acc = fmaf(w.y, RELU ? fmaxf(v[e + 1], 0.f) : v[e + 1], acc);
              acc = fmaf(w.z, RELU ? fmaxf(v[e + 2], 0.f) : v[e + 2], acc);
              acc = fmaf(w.w, RELU ? fmaxf(v[e + 3], 0.f) : v[e + 3], acc);
            }
          }
        }
        acc *= ks;
        const bool visible = page >= 0 && key <= L - n_b + j;
        if (key < p.width)
          p.scores[static_cast<int64_t>(r0 + j) * p.width + key] = visible ? acc : -__int_as_float(0x7f800000);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(d_empty + db);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
}

// ---------------------------------------------------------------------------
// K5: top-k per query row
// ---------------------------------------------------------------------------
constexpr int kTopkThreads = 512;                   // two CTAs per SM
constexpr int kBinsPerThread = 4096 / kTopkThreads;  // of the 12-bit digit histogram
constexpr int kVec = 8;        // float4 score loads in flight per thread (32 scores)
constexpr int kBatch = 8;      // scalar score loads in flight per thread (ordered tie collection)
constexpr int kRound = 4 * kVec * kTopkThreads;  // scores one round of loads covers
constexpr int kVecC = 4;       // float4 loads per thread and round of the collection pass
constexpr int kRoundC = 4 * kVecC * kTopkThreads;
constexpr int kCandCap = 4096;  // keys of the threshold's leading-digit bin kept in shared memory

// Descending bitonic sort of n (a power of two) keys in shared memory by the
// whole block.
__device__ void bitonic_desc(unsigned long long* a, int n) {
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n / 2; i += kTopkThreads) {
        const int x0 = 2 * i - (i & (stride - 1));
        const int x1 = x0 + stride;
        const bool desc = (x0 & size) == 0;
        const unsigned long long x = a[x0], y = a[x1];
        if ((x < y) == desc) {
          a[x0] = y;
          a[x1] = x;
        }
      }
      __syncthreads();
    }
  }
}

// Descending bitonic sort of n = E * kTopkThreads keys by the whole block,
// thread t holding keys [E t, E t + E) in registers: exchanges within a
// thread and between the lanes of a warp (shuffles) need no barrier; only
// the strides that cross warps go through shared memory.  a[0..n) is read
// at the start and written back sorted (the caller synchronised before).
template <int E>
__device__ void bitonic_desc_regs(unsigned long long* a, int n) {
  constexpr int kWarpSpan = 32 * E;
  const int tid = threadIdx.x;
  unsigned long long x[E];
#pragma unroll
  for (int k = 0; k < E; ++k) x[k] = a[E * tid + k];
  for (int size = 2; size <= n; size <<= 1) {
    int stride = size >> 1;
    if (stride >= kWarpSpan) {
#pragma unroll
      for (int k = 0; k < E; ++k) a[E * tid + k] = x[k];
      __syncthreads();
      for (; stride >= kWarpSpan; stride >>= 1) {
        for (int i = tid; i < n / 2; i += kTopkThreads) {
          const int x0 = 2 * i - (i & (stride - 1));
          const int x1 = x0 + stride;
          const bool desc = (x0 & size) == 0;
          const unsigned long long u = a[x0], w = a[x1];
          if ((u < w) == desc) {
            a[x0] = w;
            a[x1] = u;
          }
        }
        __syncthreads();
      }
#pragma unroll
      for (int k = 0; k < E; ++k) x[k] = a[E * tid + k];
    }
    // for strides and sizes of at least E the direction bits of key E t + k
    // are those of E t: one decision per thread and stage
    for (; stride >= E; stride >>= 1) {  // partner in lane ^ (stride / E), same slot k
      const bool take_max = (((E * tid) & stride) == 0) == (((E * tid) & size) == 0);
#pragma unroll
      for (int k = 0; k < E; ++k) {
        const unsigned long long y = __shfl_xor_sync(0xffffffffu, x[k], stride / E);
        x[k] = take_max ? (x[k] > y ? x[k] : y) : (x[k] < y ? x[k] : y);
      }
    }
    const bool desc_t = ((E * tid) & size) == 0;
#pragma unroll
    for (int sk = E / 2; sk > 0; sk >>= 1) {  // partner in the same thread (strides below E)
      if (sk < size) {
#pragma unroll
        for (int k = 0; k < E; ++k) {
          if ((k & sk) == 0) {
            const bool desc = size >= E ? desc_t : (k & size) == 0;
            const unsigned long long u = x[k], w = x[k + sk];
            if ((u < w) == desc) {
              x[k] = w;
              x[k + sk] = u;
            }
          }
        }
      }
    }
  }
#pragma unroll
  for (int k = 0; k < E; ++k) a[E * tid + k] = x[k];
  __syncthreads();
}

// Descending sort of n (a power of two) keys; a must have room for
// max(n, kTopkThreads) keys (shorter arrays are padded with 0, which sorts last).
__device__ void sort_desc(unsigned long long* a, int n) {
  if (n < kTopkThreads) {
    for (int i = n + threadIdx.x; i < kTopkThreads; i += kTopkThreads) a[i] = 0ull;
    __syncthreads();
    n = kTopkThreads;
  }
  if (n == kTopkThreads)
    bitonic_desc_regs<1>(a, n);
  else if (n == 2 * kTopkThreads)
    bitonic_desc_regs<2>(a, n);
  else if (n == 4 * kTopkThreads)
    bitonic_desc_regs<4>(a, n);
  else if (n == 8 * kTopkThreads)
    bitonic_desc_regs<8>(a, n);
  else
    bitonic_desc(a, n);
}

// Order-preserving image of a finite float (larger float -> larger unsigned);
// -0 is taken as +0.
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Sort key: score image in the high word, 0xFFFFFFFF - id in the low word,
// so a descending sort puts larger scores first and, among equal scores,
// smaller ids first.  0 = padding (sorts last).
__device__ __forceinline__ unsigned long long pack_key(uint32_t u, int id) {
  return (static_cast<unsigned long long>(u) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(id));
}

__global__ void __launch_bounds__(kTopkThreads, 2)
    index_topk_kernel(const IndexParams p, int topk, int sort_cap, int32_t* __restrict__ out) {
  extern __shared__ unsigned long long keys[];  // [max(sort_cap, kTopkThreads)], then candidates [kCandCap]
  unsigned long long* cand = keys + (sort_cap > kTopkThreads ? sort_cap : kTopkThreads);
  __shared__ __align__(16) uint32_t hist[4096];  // (also scratch for 2048 keys: 8-byte aligned)
  __shared__ uint32_t warp_cnt[kTopkThreads / 32];
  __shared__ uint32_t sh_prefix, sh_mask, sh_remaining, sh_gt, sh_eq_taken, sh_eq_total;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t t = blockIdx.x;
  // element of row t: the last b with row_offsets[b] <= t
  int lo = 0, hi = p.batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.row_offsets[mid] <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int b = lo;
  const int n_b = p.row_offsets[b + 1] - p.row_offsets[b];
  const int j = static_cast<int>(t - p.row_offsets[b]);
  const int L = p.cache_seqlens[b];
  int vis = min(L - n_b + j + 1, L);
  if (vis < 0 || n_b > p.max_new) vis = 0;
  if (vis > p.width) vis = static_cast<int>(p.width);
  const float* sc = p.scores + t * p.width;
  // launched as a programmatic dependent of the score kernel: the scores are
  // complete and visible from here on
  asm volatile("griddepcontrol.wait;" ::: "memory");
  int32_t* o = out + t * topk;

  if (vis <= topk) {
    for (int i = tid; i < sort_cap; i += kTopkThreads) keys[i] = i < vis ? pack_key(order_key(sc[i]), i) : 0ull;
  } else {
    // radix select of the topk-th largest image: digits of 12, 12 and 8 bits
    // from the top.  Twelve-bit leading digits (sign, exponent and three
    // mantissa bits) spread nearby scores over many bins, so plain shared
    // atomics rarely collide.
    if (tid == 0) {
      sh_prefix = 0;
      sh_mask = 0;
      sh_remaining = static_cast<uint32_t>(topk);
    }
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
      const int shift = pass == 0 ? 20 : (pass == 1 ? 8 : 0);
      const uint32_t dmask = pass == 2 ? 255u : 4095u;
      for (int i = tid; i < 4096; i += kTopkThreads) hist[i] = 0;
      __syncthreads();
      // read before any thread can update them (the digit search below)
      const uint32_t prefix = sh_prefix, mask = sh_mask, rem = sh_remaining;
      // kVec float4 loads per thread (independent, so they are all in
      // flight together), then the histogram updates
      for (int i0 = 0; i0 < vis; i0 += kRound) {
        float4 f[kVec];
#pragma unroll
        for (int k = 0; k < kVec; ++k) {
          const int i = i0 + 4 * (k * kTopkThreads + tid);
          f[k] = i < vis ? __ldcg(reinterpret_cast<const float4*>(sc + i)) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int k = 0; k < kVec; ++k) {
          const int i = i0 + 4 * (k * kTopkThreads + tid);
          const uint32_t u[4] = {order_key(f[k].x), order_key(f[k].y), order_key(f[k].z), order_key(f[k].w)};
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (i + c < vis && (u[c] & mask) == prefix) atomicAdd(&hist[(u[c] >> shift) & dmask], 1u);
        }
      }
      __syncthreads();
      // the digit holding the remaining-th largest: thread t owns bins
      // [kBinsPerThread * t, kBinsPerThread * (t + 1)); an exclusive suffix sum
      // over threads gives the count of keys in higher bins
      uint32_t c = 0;
#pragma unroll
      for (int q = 0; q < kBinsPerThread; ++q) c += hist[kBinsPerThread * tid + q];
      uint32_t x = c;  // inclusive suffix sum within the warp (lanes above)
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_down_sync(0xffffffffu, x, o);
        if (lane + o < 32) x += y;
      }
      if (lane == 0) warp_cnt[warp] = x;  // warp total
      __syncthreads();
      uint32_t above = x - c;  // bins of higher lanes in this warp
      for (int w = warp + 1; w < kTopkThreads / 32; ++w) above += warp_cnt[w];
      if (above < rem && above + c >= rem) {
        uint32_t acc = above;
        int d = kBinsPerThread * tid + kBinsPerThread - 1;
        for (; d > kBinsPerThread * tid; --d) {
          if (acc + hist[d] >= rem) break;
          acc += hist[d];
        }
        sh_remaining = rem - acc;
        sh_eq_total = hist[d];  // keys in the chosen bin (after the last pass: equal to T)
        sh_prefix = prefix | (static_cast<uint32_t>(d) << shift);
        sh_mask = mask | (dmask << shift);
      }
      __syncthreads();
      if (pass == 0 && sh_eq_total <= static_cast<uint32_t>(kCandCap)) break;  // uniform
    }
    if (sh_mask == (4095u << 20)) {
      // the bin of the leading digit holds few keys: one more pass over the
      // scores takes every key of a higher bin and copies that bin's keys to
      // shared memory, where a sort picks the rest (larger first, ties to the
      // smaller id)
      const uint32_t d1 = sh_prefix >> 20;
      const uint32_t rem1 = sh_remaining;
      const uint32_t n_cand = sh_eq_total;
      __syncthreads();
      if (tid == 0) {
        sh_gt = 0;
        sh_eq_taken = 0;
      }
      __syncthreads();
      for (int i0 = 0; i0 < vis; i0 += kRoundC) {
        float4 f[kVecC];
#pragma unroll
        for (int k = 0; k < kVecC; ++k) {
          const int i = i0 + 4 * (k * kTopkThreads + tid);
          f[k] = i < vis ? __ldcg(reinterpret_cast<const float4*>(sc + i)) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // each lane counts its keys above and in the bin, a warp scan of the
        // (packed) counts gives the lanes their slots: one atomic per list
        // and warp for the whole round
        uint32_t cnt = 0;  // above in the low half-word, in the bin in the high one
#pragma unroll
        for (int k = 0; k < kVecC; ++k) {
          const int i = i0 + 4 * (k * kTopkThreads + tid);
          const uint32_t u[4] = {order_key(f[k].x), order_key(f[k].y), order_key(f[k].z), order_key(f[k].w)};
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint32_t dig = u[c] >> 20;
            if (i + c < vis) cnt += dig > d1 ? 1u : (dig == d1 ? 0x10000u : 0u);
          }
        }
        uint32_t incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const uint32_t tot = __shfl_sync(0xffffffffu, incl, 31);
        uint32_t base_gt = 0, base_eq = 0;
        if (lane == 31) {
          if (tot & 0xffffu) base_gt = atomicAdd(&sh_gt, tot & 0xffffu);
          if (tot >> 16) base_eq = atomicAdd(&sh_eq_taken, tot >> 16);
        }
        uint32_t o_gt = __shfl_sync(0xffffffffu, base_gt, 31) + ((incl - cnt) & 0xffffu);
        uint32_t o_eq = __shfl_sync(0xffffffffu, base_eq, 31) + ((incl - cnt) >> 16);
#pragma unroll
        for (int k = 0; k < kVecC; ++k) {
          const int i = i0 + 4 * (k * kTopkThreads + tid);
          const uint32_t u[4] = {order_key(f[k].x), order_key(f[k].y), order_key(f[k].z), order_key(f[k].w)};
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint32_t dig = u[c] >> 20;
            if (i + c < vis && dig >= d1) {
              const unsigned long long key = pack_key(u[c], i + c);
              if (dig > d1)
                keys[o_gt++] = key;
              else
                cand[o_eq++] = key;
            }
          }
        }
      }
      const uint32_t n_gt1 = static_cast<uint32_t>(topk) - rem1;
      // The rem1 largest candidates, as a set (the final sort orders them):
      // one more radix step over the candidates in shared memory, on the next
      // twelve bits of the score image (bits 40..51 of the key); the keys of
      // higher sub-bins are taken, and the few keys of the chosen sub-bin are
      // sorted by one warp (by the block when there are many).
      __syncthreads();  // the collection pass is complete
      for (int i = tid; i < 4096; i += kTopkThreads) hist[i] = 0;
      if (tid == 0) {
        sh_gt = 0;
        sh_eq_taken = 0;
      }
      __syncthreads();
      for (uint32_t i = tid; i < n_cand; i += kTopkThreads)
        atomicAdd(&hist[static_cast<uint32_t>(cand[i] >> 40) & 4095u], 1u);
      __syncthreads();
      {
        uint32_t c = 0;
#pragma unroll
        for (int q = 0; q < kBinsPerThread; ++q) c += hist[kBinsPerThread * tid + q];
        uint32_t x = c;  // inclusive suffix sum within the warp
#pragma unroll
        for (int o2 = 1; o2 < 32; o2 <<= 1) {
          const uint32_t y = __shfl_down_sync(0xffffffffu, x, o2);
          if (lane + o2 < 32) x += y;
        }
        if (lane == 0) warp_cnt[warp] = x;
        __syncthreads();
        uint32_t above = x - c;
        for (int w = warp + 1; w < kTopkThreads / 32; ++w) above += warp_cnt[w];
        if (above < rem1 && above + c >= rem1) {
          uint32_t acc = above;
          int d = kBinsPerThread * tid + kBinsPerThread - 1;
          for (; d > kBinsPerThread * tid; --d) {
            if (acc + hist[d] >= rem1) break;
            acc += hist[d];
          }
          sh_prefix = static_cast<uint32_t>(d);
          sh_remaining = rem1 - acc;  // keys to take from sub-bin d
          sh_eq_total = hist[d];
        }
        __syncthreads();
      }
      const uint32_t d2 = sh_prefix, rem2 = sh_remaining, cnt2 = sh_eq_total;
      const uint32_t above2 = rem1 - rem2;  // keys of higher sub-bins, all taken
      unsigned long long* sub = reinterpret_cast<unsigned long long*>(hist);  // 2048 keys of scratch
      __syncthreads();  // every thread has read the histogram
      if (cnt2 <= 2048) {
        for (uint32_t i = tid; i < n_cand; i += kTopkThreads) {
          const unsigned long long key = cand[i];
          const uint32_t dd = static_cast<uint32_t>(key >> 40) & 4095u;
          if (dd > d2)
            keys[n_gt1 + atomicAdd(&sh_gt, 1u)] = key;
          else if (dd == d2)
            sub[atomicAdd(&sh_eq_taken, 1u)] = key;
        }
        __syncthreads();
        if (cnt2 <= 32) {
          if (warp == 0) {
            // descending bitonic sort of up to 32 keys, one per lane
            unsigned long long x = static_cast<uint32_t>(lane) < cnt2 ? sub[lane] : 0ull;
#pragma unroll
            for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
              for (int stride = size >> 1; stride > 0; stride >>= 1) {
                const unsigned long long y = __shfl_xor_sync(0xffffffffu, x, stride);
                const bool take_max = ((lane & stride) == 0) == ((lane & size) == 0);
                x = take_max ? (x > y ? x : y) : (x < y ? x : y);
              }
            }
            if (static_cast<uint32_t>(lane) < rem2) keys[n_gt1 + above2 + lane] = x;
          }
        } else {
          int c3 = 1;
          while (c3 < static_cast<int>(cnt2)) c3 <<= 1;
          for (int i = static_cast<int>(cnt2) + tid; i < c3; i += kTopkThreads) sub[i] = 0ull;
          __syncthreads();
          sort_desc(sub, c3);
          for (uint32_t k = tid; k < rem2; k += kTopkThreads) keys[n_gt1 + above2 + k] = sub[k];
        }
      } else {
        // (a sub-bin of more than 2048 keys: sort all candidates)
        int c2 = 1;
        while (c2 < static_cast<int>(n_cand)) c2 <<= 1;
        for (int i = static_cast<int>(n_cand) + tid; i < c2; i += kTopkThreads) cand[i] = 0ull;
        __syncthreads();
        sort_desc(cand, c2);
        for (uint32_t k = tid; k < rem1; k += kTopkThreads) keys[n_gt1 + k] = cand[k];
      }
      for (int i = topk + tid; i < sort_cap; i += kTopkThreads) keys[i] = 0ull;
      __syncthreads();
      sort_desc(keys, sort_cap);
      const int n_out1 = min(vis, topk);
      const unsigned long long ninf1 = static_cast<unsigned long long>(order_key(-__int_as_float(0x7f800000)));
      for (int k = tid; k < topk; k += kTopkThreads)
        o[k] = (k < n_out1 && (keys[k] >> 32) != ninf1)
                   ? static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(keys[k] & 0xFFFFFFFFull))
                   : -1;
      return;
    }
    const uint32_t T = sh_prefix;
    const uint32_t need_eq = sh_remaining;             // ties at T to take, in key order
    const uint32_t n_gt = static_cast<uint32_t>(topk) - need_eq;
    if (tid == 0) {
      sh_gt = 0;
      sh_eq_taken = 0;
    }
    __syncthreads();
    // when every key equal to T is taken their order does not matter: they
    // are appended like the larger ones; otherwise the first need_eq in key
    // order are taken (block-wide ordered compaction, chunk by chunk)
    const bool all_eq = sh_eq_total == need_eq;
    for (int i0 = 0; i0 < vis; i0 += kBatch * kTopkThreads) {
      uint32_t ub[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int i = i0 + k * kTopkThreads + tid;
        ub[k] = i < vis ? order_key(__ldcg(sc + i)) : 0u;
      }
#pragma unroll 1
      for (int k = 0; k < kBatch; ++k) {
        if (i0 + k * kTopkThreads >= vis) break;  // uniform across the block
        const int i = i0 + k * kTopkThreads + tid;
        const uint32_t u = ub[k];
        const bool gt = i < vis && (u > T || (all_eq && u == T));
        const uint32_t gbal = __ballot_sync(0xffffffffu, gt);
        uint32_t gbase = 0;
        if (lane == 0 && gbal) gbase = atomicAdd(&sh_gt, static_cast<uint32_t>(__popc(gbal)));
        gbase = __shfl_sync(0xffffffffu, gbase, 0);
        if (gt) keys[gbase + __popc(gbal & ((1u << lane) - 1u))] = pack_key(u, i);
        if (all_eq) continue;
        const bool eq = i < vis && u == T;
        const uint32_t bal = __ballot_sync(0xffffffffu, eq);
        if (lane == 0) warp_cnt[warp] = __popc(bal);
        const uint32_t taken_before = sh_eq_taken;
        __syncthreads();
        uint32_t before = 0;
        for (int w = 0; w < warp; ++w) before += warp_cnt[w];
        const uint32_t rank = taken_before + before + __popc(bal & ((1u << lane) - 1u));
        if (eq && rank < need_eq) keys[n_gt + rank] = pack_key(u, i);
        __syncthreads();
        if (tid == 0) {
          uint32_t tot = 0;
          for (int w = 0; w < kTopkThreads / 32; ++w) tot += warp_cnt[w];
          sh_eq_taken = taken_before + tot;
        }
        __syncthreads();
      }
    }
    for (int i = topk + tid; i < sort_cap; i += kTopkThreads) keys[i] = 0ull;
  }
  __syncthreads();
  sort_desc(keys, sort_cap);
  // keys of unusable pages carry -inf: sorted last, reported as unused slots
  const int n_out = min(vis, topk);
  const unsigned long long ninf = static_cast<unsigned long long>(order_key(-__int_as_float(0x7f800000)));
  for (int k = tid; k < topk; k += kTopkThreads)
    o[k] = (k < n_out && (keys[k] >> 32) != ninf)
               ? static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(keys[k] & 0xFFFFFFFFull))
               : -1;
}

}  // namespace

size_t index_score_smem_bytes() { return kScoreSmem; }

cudaError_t launch_index(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const IndexParams& p, int topk,
                         int32_t* out, cudaStream_t stream) {
  auto kern = p.h_idx == 64 ? (p.relu ? index_score_kernel<true, true> : index_score_kernel<false, true>)
                            : (p.relu ? index_score_kernel<true, false> : index_score_kernel<false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kScoreSmem);
  if (e != cudaSuccess) return e;
  const int max_tiles = static_cast<int>((p.width + kKeysPerTile - 1) / kKeysPerTile);
  dim3 grid((max_tiles + p.tiles_per_cta - 1) / p.tiles_per_cta, p.batch);
  kern<<<grid, kScoreThreads, kScoreSmem, stream>>>(tm_q, tm_k, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  int cap = 1;
  while (cap < topk) cap <<= 1;
  const size_t smem = static_cast<size_t>((cap > kTopkThreads ? cap : kTopkThreads) + kCandCap) * sizeof(unsigned long long);
  e = cudaFuncSetAttribute(index_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.num_tokens));
  cfg.blockDim = dim3(kTopkThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, index_topk_kernel, p, topk, cap, out);
}

}  // namespace mla
