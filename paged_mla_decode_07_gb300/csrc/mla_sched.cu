// K0 — decode tile schedule ("get_mla_metadata").
//
// The FlashMLA article ("Why FlashMLA's decode kernel reaches 660 TFLOPS",
// Design 5) describes a tile scheduler that spreads requests and KV blocks
// evenly over the SMs, computed once per decode step and reused by every
// layer.  Here every problem (a batch element in dense mode, a (batch
// element, query token) pair in sparse mode) is a run of 128-token tiles plus
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
// One CTA of 1024 threads; per-problem prefix sums live in shared memory.
#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kThreads = 1024;

struct Pos {
  int p, t;
};

__device__ __forceinline__ bool pos_less(Pos a, Pos b) { return a.p < b.p || (a.p == b.p && a.t < b.t); }

// Cost-line position x -> (problem, tile).  pre[q] = cost of problems < q,
// tiles[q] = tiles of problem q.
__device__ Pos locate(const long long* pre, const int* tiles, int np, long long x) {
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
  long long o = x - pre[lo] - kCostOverheadTiles;
  int t = o > 0 ? static_cast<int>(o) : 0;
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
__device__ void block_inclusive_scan(long long* v, int n, long long* warp_tot) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int per = (n + kThreads - 1) / kThreads;
  const int b = tid * per;
  const int e = min(n, b + per);
  long long s = 0;
  for (int i = b; i < e; ++i) {
    s += v[i];
    v[i] = s;
  }
  long long x = s;  // inclusive scan of run totals within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[w] = x;
  __syncthreads();
  if (w == 0) {
    long long t = lane < kThreads / 32 ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < kThreads / 32) warp_tot[lane] = t;
  }
  __syncthreads();
  const long long base = (x - s) + (w > 0 ? warp_tot[w - 1] : 0);
  for (int i = b; i < e; ++i) v[i] += base;
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads, 1)
    metadata_kernel(const int32_t* __restrict__ cache_seqlens, int np, int s_q, int topk, int num_parts,
                    int32_t* __restrict__ sched, int32_t* __restrict__ num_splits, uint32_t* status) {
  extern __shared__ __align__(16) unsigned char smem[];
  long long* pre = reinterpret_cast<long long*>(smem);             // [np + 1]
  long long* warp_tot = pre + (np + 1);                            // [kThreads / 32]
  long long* cnt = pre;                                            // [np], reuses pre after step 2
  Pos* starts = reinterpret_cast<Pos*>(warp_tot + kThreads / 32);  // [num_parts + 1]
  int* tiles = reinterpret_cast<int*>(starts + num_parts + 1);     // [np]
  const int tid = threadIdx.x;
  // the decode kernel may launch now (its prologue overlaps this kernel; it
  // waits for this kernel's results before reading the schedule)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // 1. problem tiles (one read of cache_seqlens), costs and their prefix sums
  for (int p = tid; p < np; p += kThreads) {
    const int n = problem_tiles(cache_seqlens, p, s_q, topk);
    tiles[p] = n;
    pre[p + 1] = n > 0 ? static_cast<long long>(n) + kCostOverheadTiles : 0;
  }
  if (tid == 0) pre[0] = 0;
  __syncthreads();
  block_inclusive_scan(pre + 1, np, warp_tot);
  const long long total = pre[np];

  // 2. cut the cost line into num_parts equal pieces.  Cut points are distinct
  // while k <= total (so equal part starts, i.e. empty parts, only arise inside
  // a problem's start-up cost, at its tile 0, or at the very end); with less
  // work than parts the surplus parts are empty.
  for (int k = tid; k <= num_parts; k += kThreads) {
    long long x = total >= num_parts ? total * static_cast<long long>(k) / num_parts
                                     : (static_cast<long long>(k) < total ? k : total);
    starts[k] = locate(pre, tiles, np, x);
  }
  __syncthreads();

  // 3. pieces per problem.  Parts are contiguous and empty parts can only sit
  // at a problem's tile 0, so the parts touching problem p are
  // first(p) .. last(p), where part(x) = the last part starting at or before x.
  // Slots: the piece count of a split problem, 0 for a single piece.
  for (int p = tid; p < np; p += kThreads) {
    const int n = tiles[p];
    const int pieces =
        n > 0 ? part_of(starts, num_parts, Pos{p, n - 1}) - part_of(starts, num_parts, Pos{p, 0}) + 1 : 0;
    cnt[p] = pieces > 1 ? pieces : 0;
  }
  __syncthreads();
  block_inclusive_scan(cnt, np, warp_tot);
  for (int p = tid; p <= np; p += kThreads) num_splits[p] = p == 0 ? 0 : static_cast<int32_t>(cnt[p - 1]);

  // 4. schedule records; a part's split index in its first problem is its
  // distance from the first part touching that problem
  for (int k = tid; k < num_parts; k += kThreads) {
    Pos a = starts[k], b = starts[k + 1];
    int split0 = 0;
    if (pos_less(a, b) && a.p < np) split0 = k - part_of(starts, num_parts, Pos{a.p, 0});
    int32_t* r = sched + static_cast<size_t>(k) * kSchedInts;
    r[kSchedP0] = a.p;
    r[kSchedT0] = a.t;
    r[kSchedP1] = b.p;
    r[kSchedT1] = b.t;
    r[kSchedSplit0] = split0;
    r[5] = 0;
    r[6] = 0;
    r[7] = 0;
  }
  (void)status;
}

}  // namespace

size_t metadata_smem_bytes(int np, int num_parts) {
  return sizeof(long long) * (np + 1) + sizeof(long long) * (kThreads / 32) + sizeof(int) * 2 * (num_parts + 1) +
         sizeof(int) * np;
}

cudaError_t launch_metadata(const int32_t* cache_seqlens, int batch, int s_q, int h_q, int topk,
                            const Geometry& g, int32_t* sched, int32_t* num_splits, uint32_t* status,
                            cudaStream_t stream) {
  (void)batch;
  (void)h_q;
  size_t smem = metadata_smem_bytes(g.num_problems, g.num_parts);
  cudaError_t e = cudaFuncSetAttribute(metadata_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  metadata_kernel<<<1, kThreads, smem, stream>>>(cache_seqlens, g.num_problems, s_q, topk, g.num_parts, sched,
                                                 num_splits, status);
  return cudaGetLastError();
}

}  // namespace mla
