// K0 — decode tile schedule ("get_mla_metadata").
//
// The FlashMLA article ("Why FlashMLA's decode kernel reaches 660 TFLOPS",
// Design 5) describes a tile scheduler that spreads requests and KV blocks
// evenly over the SMs, computed once per decode step and reused by every
// layer.  Here every problem (a batch element in dense mode, a (batch
// element, query token) pair in sparse mode) is a run of tiles (64 tokens, or
// 128 for the CTA-pair kernel) plus
// a fixed start-up cost; the concatenated cost line is cut into num_parts
// contiguous pieces of equal cost.  A piece may start or end inside a
// problem; such a problem is then split and its pieces are merged by the
// combine kernel.  num_splits is the exclusive prefix sum of the partial-result
// slots per problem: a split problem takes one slot per piece, a problem
// covered by a single piece takes none (its piece writes the output
// directly).  Split problems' part ranges overlap only at their end parts,
// so all problems together take at most 2 * num_parts slots, whatever the
// number of problems (and at most num_problems + num_parts: each part
// boundary adds one piece).
//
// Costs are in quarters of a 64-token bf16 tile: such a tile costs 4, a tile
// of FP8 rows (gathered and dequantised before its MMAs) 6, a 128-token tile
// twice that, and starting a problem segment (loading its queries, filling
// the pipeline, writing its rows) 8, so the cut weighs start-up against tiles
// as the decode kernels spend them.
//
// One CTA of 256 threads; per-problem prefix sums live in shared memory, and
// every step is a parallel pass or a block-wide scan (the kernel sits on the
// critical path of each decode step, before the decode kernel can start).
#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kThreads = 256;

struct Pos {
  int p, t;
};

__device__ __forceinline__ bool pos_less(Pos a, Pos b) { return a.p < b.p || (a.p == b.p && a.t < b.t); }

// Cost-line position x -> (problem, tile).  pre[q] = cost of problems < q,
// tiles[q] = tiles of problem q; a problem's line is its start-up cost
// followed by its tiles, tile_cost each.
__device__ Pos locate(const long long* pre, const int* tiles, int np, long long x, int tile_cost, int overhead) {
  if (x >= pre[np]) return Pos{np, 0};
  // largest p with pre[p] <= x (problems of zero cost share a prefix value; take the last)
  int lo = 0, hi = np - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= x)
      lo = mid;
    else
      hi = mid - 1;
  }
  long long o = x - pre[lo] - overhead;
  int t = o > 0 ? static_cast<int>(o / tile_cost) : 0;
  if (t >= tiles[lo]) return Pos{lo + 1, 0};
  return Pos{lo, t};
}

// Last part k (0 <= k < num_parts) whose start is at or before x.
__device__ int part_of(const Pos* starts, int num_parts, Pos x) {
  int lo = 0, hi = num_parts - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (!pos_less(x, starts[mid]))
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// In-place inclusive scan of v[0..n) by the whole block: each thread scans a
// contiguous run, warps scan their run totals with shuffles, one warp scans
// the warp totals.  warp_tot holds kThreads / 32 entries.
template <typename T>
__device__ void block_inclusive_scan(T* v, int n, T* warp_tot) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int per = (n + kThreads - 1) / kThreads;
  const int b = tid * per;
  const int e = min(n, b + per);
  T s = 0;
  for (int i = b; i < e; ++i) {
    s += v[i];
    v[i] = s;
  }
  T x = s;  // inclusive scan of run totals within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[w] = x;
  __syncthreads();
  if (w == 0) {
    T t = lane < kThreads / 32 ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const T y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < kThreads / 32) warp_tot[lane] = t;
  }
  __syncthreads();
  const T base = (x - s) + (w > 0 ? warp_tot[w - 1] : 0);
  for (int i = b; i < e; ++i) v[i] += base;
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads, 1)
    metadata_kernel(const int32_t* __restrict__ cache_seqlens, int np, int s_q, int topk, int num_parts,
                    int tile_tokens, int tile_cost, int overhead, int tag, int32_t* __restrict__ sched,
                    int32_t* __restrict__ num_splits) {
  extern __shared__ __align__(16) unsigned char smem[];
  long long* pre = reinterpret_cast<long long*>(smem);             // [np + 1]
  long long* warp_tot = pre + (np + 1);                            // [kThreads / 32]
  long long* cnt = pre;                                            // [np], reuses pre after step 2
  Pos* starts = reinterpret_cast<Pos*>(warp_tot + kThreads / 32);  // [num_parts + 1]
  int* tiles = reinterpret_cast<int*>(starts + num_parts + 1);     // [np]
  int* ne_pre = tiles + np;                                        // [num_parts + 1]
  const int tid = threadIdx.x;
  // the decode kernel may launch now (its prologue overlaps this kernel; it
  // waits for this kernel's results before reading the schedule)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // 1. problem tiles (one read of cache_seqlens), costs and their prefix sums
  for (int p = tid; p < np; p += kThreads) {
    const int n = problem_tiles(cache_seqlens, p, s_q, topk, tile_tokens);
    tiles[p] = n;
    pre[p + 1] = n > 0 ? static_cast<long long>(n) * tile_cost + overhead : 0;
  }
  if (tid == 0) pre[0] = 0;
  __syncthreads();
  block_inclusive_scan(pre + 1, np, warp_tot);
  const long long total = pre[np];

  // 2. cut the cost line into num_parts equal pieces.  A part shorter than
  // one tile may start where the next one does: such a part is empty (it
  // does no work and takes no partial-result slot).  With less work than
  // parts the surplus parts are empty.
  for (int k = tid; k <= num_parts; k += kThreads) {
    long long x = total >= num_parts ? total * static_cast<long long>(k) / num_parts
                                     : (static_cast<long long>(k) < total ? k : total);
    starts[k] = locate(pre, tiles, np, x, tile_cost, overhead);
  }
  __syncthreads();
  // ne_pre[k] = number of non-empty parts before part k
  for (int k = tid; k < num_parts; k += kThreads) ne_pre[k + 1] = pos_less(starts[k], starts[k + 1]) ? 1 : 0;
  if (tid == 0) ne_pre[0] = 0;
  __syncthreads();
  block_inclusive_scan(ne_pre + 1, num_parts, reinterpret_cast<int*>(warp_tot));

  // 3. pieces per problem.  Parts are contiguous, so the parts touching
  // problem p lie between first(p) = part(p, tile 0) and last(p) =
  // part(p, last tile), where part(x) = the last part starting at or before
  // x (always a non-empty part holding x); its pieces are the non-empty parts
  // of that range.  Slots: the piece count of a split problem, 0 for a single
  // piece.
  for (int p = tid; p < np; p += kThreads) {
    const int n = tiles[p];
    int pieces = 0;
    if (n > 0) {
      const int k0 = part_of(starts, num_parts, Pos{p, 0});
      const int k1 = part_of(starts, num_parts, Pos{p, n - 1});
      pieces = ne_pre[k1 + 1] - ne_pre[k0];
    }
    cnt[p] = pieces > 1 ? pieces : 0;
  }
  __syncthreads();
  block_inclusive_scan(cnt, np, warp_tot);
  for (int p = tid; p <= np; p += kThreads) num_splits[p] = p == 0 ? 0 : static_cast<int32_t>(cnt[p - 1]);

  // 4. schedule records; a part's split index in its first problem is its
  // rank among the non-empty parts touching that problem
  for (int k = tid; k < num_parts; k += kThreads) {
    Pos a = starts[k], b = starts[k + 1];
    int split0 = 0;
    if (pos_less(a, b) && a.p < np) split0 = ne_pre[k] - ne_pre[part_of(starts, num_parts, Pos{a.p, 0})];
    int32_t* r = sched + static_cast<size_t>(k) * kSchedInts;
    r[kSchedP0] = a.p;
    r[kSchedT0] = a.t;
    r[kSchedP1] = b.p;
    r[kSchedT1] = b.t;
    r[kSchedSplit0] = split0;
    r[kSchedParts] = num_parts;
    r[kSchedTag] = tag;
    r[7] = 0;
  }
}

}  // namespace

size_t metadata_smem_bytes(int np, int num_parts) {
  return sizeof(long long) * (np + 1) + sizeof(long long) * (kThreads / 32) + sizeof(int) * 2 * (num_parts + 1) +
         sizeof(int) * np + sizeof(int) * (num_parts + 1);
}

cudaError_t launch_metadata(const int32_t* cache_seqlens, int s_q, int topk, const Geometry& g, int32_t* sched,
                            int32_t* num_splits, cudaStream_t stream) {
  size_t smem = metadata_smem_bytes(g.num_problems, g.num_parts);
  cudaError_t e = cudaFuncSetAttribute(metadata_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  metadata_kernel<<<1, kThreads, smem, stream>>>(cache_seqlens, g.num_problems, s_q, topk, g.num_parts,
                                                 g.tile_tokens, g.tile_cost, g.overhead, g.tag, sched, num_splits);
  return cudaGetLastError();
}

}  // namespace mla
