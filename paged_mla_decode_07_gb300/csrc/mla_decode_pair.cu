// K1p — paged MLA decode on CTA pairs (tcgen05 cta_group::2) for problems of
// more than 64 query rows: dense over the bf16 cache, and sparse (top-k) over
// the FP8 cache or over bf16 rows (the bf16 cache, or the unpaged rows of
// sparse prefill).
//
// What is computed is the same as in the single-CTA kernel (mla_decode.cu):
// per query row, softmax(q K^T * sm_scale) V over the row's keys with
// V = K[:, :512] (the MQA form of MLA, Modular design-doc overview, section 9
// "Multi-Head Latent Attention"), with online softmax across tiles (overview,
// section 6 "Matmul to Flash Attention"), and a split-KV partial with its
// log-sum-exp where a part covers only some of a problem's tiles (FlashMLA
// article, Design 5; merged by the combine kernel).  In sparse mode the keys
// of a query token are the valid ids of its index row and each FP8 row is
// dequantised as bf16_rn(fp32(e4m3) * scale) before the MMAs (FlashMLA
// article, Design 2); bf16 rows are used as they are.
//
// Formulation.  The two CTAs of a cluster (one TPC) work together on 128
// query rows of a problem, 64 rows each, and on 128-token tiles, 64 tokens
// each (dense: one page per CTA; sparse: index slots 64c .. 64c + 63 of the
// tile for CTA c).  Both matrix products are pair MMAs issued by one thread
// of the even CTA: each CTA supplies half of A's rows and half of B's columns
// from its own shared memory and receives its half of the result rows in its
// own TMEM.  For an M = 128 pair result a CTA's row r lies in TMEM lane r for
// the first half of the columns and in lane 64 + r for the second half.
//     S[row, tok]  = Q[row, :] . K[tok, :]      M = 128 rows, N = 128 tokens, K = 576
//                    A: the CTA's 64 query rows, B: the CTA's 64 tokens
//     O[row, dv]  += P[row, tok] . V[tok, dv]    M = 128 rows, N = 256 dv (twice), K = 128 tokens
//                    A: the CTA's P rows, B: the CTA's share of the 256 dv
// An N = 256 pair MMA runs at the tensor pipe's full rate and an N = 128 one
// at 57 %, where a single-CTA M = 64 score MMA runs at 28 %.  Each CTA
// brings in its own 64 tokens per tile for the scores, and it keeps the
// running O of its own rows for all 512 value dims (64 rows x 512 fp32 = 256
// TMEM columns), so the online-softmax rescale and the epilogue stay inside
// the CTA.
//
// The value dims a CTA supplies to the PV product must sit at the same
// shared-memory address in both CTAs while holding different dims (dv 0-127
// and 256-383 for the even CTA, 128-255 and 384-511 for the odd one), so
// those dims of all 128 tokens of a tile live in a separate set of slots:
// loaded (dense), or (sparse) copied from the dequantised score operand of
// the CTA that owns the token: into its own slots by its gather warps, into
// its partner's by one bulk shared-memory copy per block.
//
// Shared memory (1024-byte aligned, identical in both CTAs):
//   Q    9 chunks [64 rows][64 dims] bf16, 128-byte swizzle         72 KB
//   KS   9 slots: dims chunk k of the CTA's 64 tokens (score operand) 72 KB
//   KV   8 slots: token half t of the tile, share s at slot 4t + s    64 KB
//   P    2 chunks [64 rows][64 tokens] bf16 (PV operand)             16 KB
//   barriers, row statistics, token-validity bits (sparse)
// TMEM (512 columns, allocated for the pair): O at [0, 256) (block m of 256
// dv at [128m, 128m + 128)), S double buffer at [256, 320) and [320, 384).
//
// Synchronisation.  Only the even CTA issues MMAs.  Dense: its producers arm
// its barriers with the bytes of both CTAs, and the odd CTA's copies
// (cta_group::2 TMA) complete on them directly; pages without tokens or with
// an unusable block-table entry are read past the end of the cache, as
// zeros.  Sparse: the softmax warps of both CTAs arrive on the even CTA's
// score-operand barriers once they have dequantised an item, and each CTA's
// value-slot copier once its slots of the tile are complete.  Sparse rows are
// copied with 16-byte cp.async by all lanes of the gather warps rather than
// with TMA row gathers: a warp issuing row gathers waits about 90 cycles per
// gather, which at 40 gathers per warp and tile was longer than the tile's
// MMAs.  The MMA warps commit to the barriers of both CTAs at once
// (multicast); the odd CTA's softmax warps arrive remotely on the even CTA's
// barriers.  Every wait is bounded by the
// watchdog; a CTA that gives up records MLA_DEVICE_TIMEOUT and unwinds, and
// its partner's waits then run out too.
//
// Roles:
//   warp 0      Q (and, dense, the score operand) producer (TMA), both CTAs
//   warp 1      score MMA issuer (even CTA)
//   warp 2      TMEM allocation, then the value-operand producer (dense: TMA
//               loads; sparse: bulk copies from the dequantised score slots)
//   warp 3      PV MMA issuer (even CTA)
//   warps 4-11  softmax + epilogue: warp w reads TMEM lane quarter w % 4, so
//               a thread owns one row and one half of the tile, and the two
//               warpgroups split that half's 64 tokens; sparse: also the
//               dequantisation of the next tile's score operand
//   warps 12-15 (sparse) row lookups, row copies, the own value share
#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {

// Pipeline tracing (built only with -DMLA_TRACE): clock64() stamps of the
// pipeline events of the first CTA pair, per (CTA, event, tile).
#ifdef MLA_TRACE
constexpr int kPairTrTiles = 256, kPairTrEvents = 16;
__device__ unsigned long long g_pair_trace[2 * kPairTrEvents * kPairTrTiles];
// per CTA (up to 1024): %globaltimer at the start of its work, at its end, and its tile count
__device__ unsigned long long g_pair_cta[3 * 1024];
#define PAIR_TR(rank, ev, idx)                                                                      \
  do {                                                                                              \
    if (blockIdx.x < 2 && (idx) < kPairTrTiles) g_pair_trace[((rank) * kPairTrEvents + (ev)) * kPairTrTiles + (idx)] = clock64(); \
  } while (0)
extern "C" int mla_pair_cta_read(unsigned long long* host) {
  return cudaMemcpyFromSymbol(host, g_pair_cta, sizeof(g_pair_cta)) == cudaSuccess ? 0 : -1;
}
extern "C" int mla_pair_trace_read(unsigned long long* host, size_t n) {
  const size_t total = sizeof(g_pair_trace) / sizeof(unsigned long long);
  if (n > total) n = total;
  if (cudaMemcpyFromSymbol(host, g_pair_trace, n * sizeof(unsigned long long)) != cudaSuccess) return -1;
  return static_cast<int>(n);
}
#else
#define PAIR_TR(rank, ev, idx) \
  do {                         \
  } while (0)
#endif

namespace {

constexpr int kPairRows = 64;            // query rows per CTA
constexpr int kPairTile = 128;           // tokens per tile (64 per CTA)
constexpr int kPairChunk = 8192;         // [64 rows or tokens][64 dims] bf16
constexpr int kPairQOff = 0;
constexpr int kPairKsOff = 9 * kPairChunk;
constexpr int kPairKvOff = 18 * kPairChunk;
constexpr int kPairPOff = 26 * kPairChunk;
constexpr int kPairAuxOff = 28 * kPairChunk;  // 229376
constexpr int kPairBarBytes = 320;
// aux: barriers, m[64], red[4][64] (partial row maxima / sums), ints (abort
// flag, TMEM base), token-validity bits of four tiles (sparse)
constexpr int kPairMOff = kPairBarBytes;
constexpr int kPairRedOff = kPairMOff + 64 * 4;
constexpr int kPairIntOff = kPairRedOff + 4 * 64 * 4;
constexpr int kPairFlagOff = kPairIntOff + 64;
// 16-byte slots the odd CTA's async signal copies write into (their contents
// are never read): 0..7 dequantised score blocks (per softmax warp), 8..9 the
// RoPE item, 10 P ready
constexpr int kPairSigOff = kPairFlagOff + 4 * 16;
constexpr int kPairSigSlots = 11;
constexpr int kPairAuxBytes = kPairSigOff + 16 * kPairSigSlots;
constexpr int kPairSmemBytes = kPairAuxOff + kPairAuxBytes + 1024;  // + alignment slack
static_assert(kPairSmemBytes <= 232448, "shared memory budget");
constexpr uint32_t kPairOCol = 0;
constexpr uint32_t kPairSCol = 256;
constexpr uint32_t kPairTmemCols = 512;
constexpr float kPairNegInf = -__builtin_huge_valf();
constexpr float kPairRescale = 8.0f;     // log2 units: P <= 2^8 before a max update is forced
constexpr uint32_t kPairSmBar = 1;       // named barrier of the 256 softmax threads
constexpr uint32_t kPairGatherBar = 2;   // named barrier of the 128 gather threads (sparse)
constexpr int kPairGatherWarp0 = 12;

// Dense: 384 threads, the score operand arrives in three copies of three
// chunks.  Sparse: 512 threads (four gather warps), the score operand is
// released and refilled by value block (chunks 2b, 2b + 1) and RoPE chunk.
// Registers: a kernel that uses setmaxnreg is compiled to the whole
// per-thread share of the register file; each role moves from it with .inc
// or .dec, and the shares add up to at most 65536.
template <bool SPARSE>
struct PairCfg {
  static constexpr int kThreads = SPARSE ? 512 : 384;
  static constexpr int kItems = SPARSE ? 5 : 3;
  static constexpr uint32_t kRegsCtl = SPARSE ? 64 : 88;
  static constexpr uint32_t kRegsSm = SPARSE ? 168 : 208;
  static constexpr uint32_t kRegsGather = 112;
  static constexpr uint32_t kLaunchRegs = SPARSE ? 128 : 168;
  static_assert(128 * kRegsCtl + 256 * kRegsSm + (SPARSE ? 128 * kRegsGather : 0) <= 65536, "register split");
  __device__ static constexpr int item_chunk0(int i) { return SPARSE ? 2 * i : 3 * i; }
  __device__ static constexpr int item_chunks(int i) { return SPARSE ? (i < 4 ? 2 : 1) : 3; }
};

enum PairBar {
  kBQFull = 0,    // Q of the segment loaded (both CTAs)
  kBQEmpty = 1,   // the segment's last score MMAs are done (Q reusable)
  kBKsFull = 2,   // [5] score-operand item i of both CTAs is in place
  kBKsEmpty = 7,  // [5] the score MMAs have read item i
  kBKvFull = 12,  // the tile's value-operand slots are in place
  kBKvEmpty = 13, // the tile's PV MMAs are done (value slots reusable)
  kBSFull = 14,   // [2] S of a tile is in TMEM
  kBSEmpty = 16,  // [2] (even) both CTAs' softmax warps have read an S buffer
  kBPFull = 18,   // (even) both CTAs' P of the tile is written, O rescaled
  kBPEmpty = 19,  // the tile's PV MMAs are done (P reusable, O current)
  kBOFull = 20,   // the segment's last PV MMAs are done
  kBOEmpty = 21,  // (even) both CTAs' epilogues have read O
  kBMmaDone = 22, // (even) drain of the MMA issuers
  kBRaw = 23,     // [5] (sparse) the rows of item i (block i, 4: RoPE) landed in this CTA
  kBFlags = 28,   // [4] (sparse) the validity bits of tile jt (barrier jt % 4) are written by the
                  // gather warps of both CTAs, which can run up to three tiles ahead of the softmax
  kBKsDone = 32,  // [2] (sparse) block 1 - rank + 2m of the tile's score operand is in place
  kBKsRead = 34,  // [2] (sparse) its copy to the partner's value slots has read it
  kBKvIn = 36,    // (sparse) this CTA's value slots of the tile are complete: its own share
                  // written by its gather warps, the partner's copies (transaction bytes)
  kBKsDoneOwn = 37,  // (sparse) blocks rank and rank + 2 of the tile's score operand are in place
  kBCount = 38
};
static_assert(kBCount * 8 <= kPairBarBytes, "barrier area");

// Segment iterator over the part's problems (128-token tiles); every role
// derives the identical sequence.
struct PairSeg {
  int p0, t0, p1, t1, np, s_q, topk;
  const int32_t* seqlens;
  __device__ int last() const { return p1 < np ? p1 : np - 1; }
  __device__ void range(int p, int& tb, int& te) const {
    const int n = problem_tiles(seqlens, p, s_q, topk, kPairTile);
    tb = (p == p0) ? t0 : 0;
    te = (p == p1) ? t1 : n;
    if (te > n) te = n;
  }
};

// Page of half h (0, 1) of tile j of element b: its id, or -1 when it holds
// no cached token or its block-table entry is unusable (flagged).
__device__ __forceinline__ int tile_page(const DecodeParams& p, int b, int L, int j, int h, bool flag) {
  const int pi = 2 * j + h;
  if (pi * kPageSize >= L) return -1;
  const int pg = pi < p.block_table_stride ? p.block_table[static_cast<int64_t>(b) * p.block_table_stride + pi] : -1;
  if (pg < 0 || pg >= p.num_pages) {
    if (flag) atomicOr(p.status, MLA_DEVICE_BAD_PAGE);
    return -1;
  }
  return pg;
}

__device__ __forceinline__ void tma3(uint32_t dst, const void* map, uint32_t bar, int c0, int c1, int c2,
                                     uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}

// The same copy, completing on an mbarrier of the even CTA (shared::cluster address).
__device__ __forceinline__ void tma3_to_even(uint32_t dst, const void* map, uint32_t bar_cluster, int c0, int c1, int c2,
                                             uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}

// Tile j of a problem of L tokens holds a page that straddles the length:
// its slots past the length may hold anything (e.g. NaN), so the value rows
// of those tokens are zeroed after the copy lands, before the PV MMAs.
__device__ __forceinline__ bool tail_tile(int L, int j) {
  return L > 0 && (L & (kPageSize - 1)) != 0 && j == (L - 1) / kPairTile;
}

// Prefetch a box of a tensor map into L2 (no shared memory involved).
__device__ __forceinline__ void tma_prefetch3(const void* map, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

// try_wait on a barrier of this CTA with acquire at cluster scope (the thread
// may be suspended until the phase completes or a time limit of the hardware
// passes).
__device__ __forceinline__ bool mbar_try_wait_cluster_u32(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Warp-uniform bounded wait on a barrier of this CTA (acquire at cluster
// scope: many phases are completed by the other CTA's arrivals).  The polls
// are try_waits, which may suspend the warp until the phase completes: hot
// test_wait loops of the waiting roles cost the score MMAs issue slots and
// shared-memory cycles (pair decode calls 2-3 % slower).
__device__ __forceinline__ bool pair_wait(uint32_t bar, uint32_t parity, const Watchdog& wd) {
  uint64_t t0 = 0;
  while (__shfl_sync(0xffffffffu, mbar_try_wait_cluster_u32(bar, parity) ? 1 : 0, 0) == 0) {
    if (t0 == 0) {
      t0 = global_timer_ns();
    } else if (__shfl_sync(0xffffffffu, wd.aborted() ? 1 : 0, 0)) {
      return false;
    } else if (__shfl_sync(0xffffffffu, global_timer_ns() - t0 > wd.limit_ns ? 1 : 0, 0)) {
      if ((threadIdx.x & 31) == 0) wd.trip(MLA_DEVICE_TIMEOUT);
      return false;
    }
  }
  return true;
}

// The same for one thread.
__device__ __forceinline__ bool pair_wait_thread(uint32_t bar, uint32_t parity, const Watchdog& wd) {
  if (mbar_test_wait_cluster_u32(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait_cluster_u32(bar, parity)) return true;
    if (wd.aborted()) return false;
    if (global_timer_ns() - t0 > wd.limit_ns) {
      wd.trip(MLA_DEVICE_TIMEOUT);
      return false;
    }
  }
}

// Bounded wait that ignores the abort flag (drain of own asynchronous work).
__device__ __forceinline__ void pair_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test_wait_u32(bar, parity))
    if (global_timer_ns() - t0 > limit_ns) return;
}

// One arrival of the calling warp on a barrier of the even CTA (remote from the odd CTA).
__device__ __forceinline__ void warp_arrive_even(int rank, uint32_t bar_local, uint32_t bar_even) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) {
    if (rank == 0)
      mbar_arrive(reinterpret_cast<uint64_t*>(__cvta_shared_to_generic(bar_local)));
    else
      mbar_arrive_cluster(bar_even);
  }
}

// ---------------------------------------------------------------------------
// warp 0: Q of each segment and (dense) the score operand: the CTA's own
// page of each tile
// ---------------------------------------------------------------------------
template <bool SPARSE>
__device__ void pair_producer_ks(const CUtensorMap* tm_q, const CUtensorMap* tm_ks, const DecodeParams& p,
                                 const PairSeg& sg, int g, int rank, uint32_t smem, uint32_t bars, uint32_t bars_even,
                                 const Watchdog& wd) {
  // The even CTA arms its Q and score-operand barriers with the bytes of
  // both CTAs; the odd CTA's copies complete on them directly.  A page that
  // holds no token or whose block-table entry is unusable is read at a row
  // past the end of the cache, which the copy fills with zeros.
  const int lane = threadIdx.x & 31;
  const uint64_t pol = l2_policy_evict_normal();
  const int oob_row = p.num_pages * kPageSize;
  uint32_t armed = 0, next_par = 0;  // ks_full barriers armed (bit per group), parity of their next phase
  int q_armed = 0, jt = 0;
  for (int prob = sg.p0; prob <= sg.last(); ++prob) {
    int tb, te;
    sg.range(prob, tb, te);
    if (tb >= te) continue;
    if (q_armed > 0 && !pair_wait(bars + 8 * kBQEmpty, (q_armed - 1) & 1, wd)) goto drain;
    {
      // this CTA's 64 query rows, all nine chunks, in one copy
      const int row0 = prob * p.rows + g * 2 * kPairRows + rank * kPairRows;
      if (lane == 0) {
        if (rank == 0) {
          mbar_arrive_expect_tx_u32(bars + 8 * kBQFull, 2 * kNumChunks * kPairChunk);
          tma3(smem + kPairQOff, tm_q, bars + 8 * kBQFull, 0, row0, 0, pol);
        } else {
          tma3_to_even(smem + kPairQOff, tm_q, bars_even + 8 * kBQFull, 0, row0, 0, pol);
        }
      }
      __syncwarp();
      ++q_armed;
    }
    if (SPARSE) continue;  // the gather warps fill the score operand
    {
      const int b = prob;
      const int L = sg.seqlens[b];
      for (int j = tb; j < te; ++j, ++jt) {
        const int pg = tile_page(p, b, L, j, rank, lane == 0);
        const int row = pg >= 0 ? pg * kPageSize : oob_row;
        if (lane == 0) PAIR_TR(rank, 0, jt);
        // the page two tiles ahead goes to L2 now, so that its copy into shared
        // memory (which must wait for this tile's score MMAs) hits L2
        if (j + 2 < te) {
          const int pg2 = tile_page(p, b, L, j + 2, rank, false);
          if (pg2 >= 0 && lane < 3) tma_prefetch3(tm_ks, 0, pg2 * kPageSize, 3 * lane);
        }
#pragma unroll 1
        for (int gr = 0; gr < 3; ++gr) {
          const uint32_t fb = bars + 8 * (kBKsFull + gr);
          if (jt > 0 && !pair_wait(bars + 8 * (kBKsEmpty + gr), (jt - 1) & 1, wd)) goto drain;
          if (lane == 0) {
            if (rank == 0) {
              mbar_arrive_expect_tx_u32(fb, 2 * 3 * kPairChunk);
              tma3(smem + kPairKsOff + 3 * gr * kPairChunk, tm_ks, fb, 0, row, 3 * gr, pol);
            } else {
              tma3_to_even(smem + kPairKsOff + 3 * gr * kPairChunk, tm_ks, bars_even + 8 * (kBKsFull + gr), 0, row,
                           3 * gr, pol);
            }
          }
          __syncwarp();
          armed |= 1u << gr;
          next_par ^= 1u << gr;
          if (lane == 0 && gr == 0) PAIR_TR(rank, 1, jt);
          if (lane == 0 && gr == 2) PAIR_TR(rank, 2, jt);
        }
      }
    }
  }
drain:
  // the even CTA waits (bounded) for the copies of both CTAs it armed; the
  // odd CTA's copies are covered by that wait and by the pause before exit
  if (lane == 0 && rank == 0) {
#pragma unroll 1
    for (int gr = 0; gr < 3; ++gr)
      if ((armed >> gr) & 1u) pair_drain(bars + 8 * (kBKsFull + gr), ((next_par >> gr) & 1u) ^ 1u, wd.limit_ns);
    if (q_armed > 0) pair_drain(bars + 8 * kBQFull, (q_armed - 1) & 1, wd.limit_ns);
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// warp 2 (dense, after the TMEM allocation): the value operand — for both
// pages of each tile, the two 128-dv blocks this CTA supplies (chunks
// 4m + 2 rank and 4m + 2 rank + 1 for m = 0, 1), into slots 4t + 2m, 4t + 2m + 1
// ---------------------------------------------------------------------------
__device__ void pair_producer_kv(const CUtensorMap* tm_kv, const DecodeParams& p, const PairSeg& sg, int rank,
                                 uint32_t smem, uint32_t bars, uint32_t bars_even, const Watchdog& wd) {
  // Every tile's value slots complete on the even CTA's kv_full (armed with
  // both CTAs' bytes), except on a tail tile, where each CTA's copies
  // complete on its own kv_full so that its softmax warps can zero the rows
  // past the length before they report P ready.  Each CTA arms its own
  // kv_full once per tile (the odd CTA with no bytes outside tail tiles).
  const int lane = threadIdx.x & 31;
  const uint64_t pol = l2_policy_evict_normal();
  const uint32_t fb = bars + 8 * kBKvFull;
  const int oob_row = p.num_pages * kPageSize;
  int jt = 0;
  bool armed = false;
  for (int prob = sg.p0; prob <= sg.last(); ++prob) {
    int tb, te;
    sg.range(prob, tb, te);
    if (tb >= te) continue;
    const int b = prob;
    const int L = sg.seqlens[b];
    for (int j = tb; j < te; ++j, ++jt) {
      const int pg0 = tile_page(p, b, L, j, 0, false);
      const int pg1 = tile_page(p, b, L, j, 1, false);
      const bool tail = tail_tile(L, j);
      if (jt > 0 && !pair_wait(bars + 8 * kBKvEmpty, (jt - 1) & 1, wd)) goto drain;
      if (lane == 0) {
        PAIR_TR(rank, 12, jt);
        const uint32_t own = 4 * kPairChunk * 2;  // two pages x two copies of two chunks
        if (rank == 0)
          mbar_arrive_expect_tx_u32(fb, tail ? own : 2 * own);
        else
          mbar_arrive_expect_tx_u32(fb, tail ? own : 0u);
      }
      __syncwarp();
      armed = true;
      if (lane < 4) {
        const int t = lane >> 1, m = lane & 1;
        const int pg = t ? pg1 : pg0;
        const int row = pg >= 0 ? pg * kPageSize : oob_row;
        const uint32_t dst = smem + kPairKvOff + (4 * t + 2 * m) * kPairChunk;
        if (rank == 0 || tail)
          tma3(dst, tm_kv, fb, 0, row, 4 * m + 2 * rank, pol);
        else
          tma3_to_even(dst, tm_kv, bars_even + 8 * kBKvFull, 0, row, 4 * m + 2 * rank, pol);
      }
      __syncwarp();
    }
  }
drain:
  if (lane == 0 && armed) pair_drain(fb, (jt - 1) & 1, wd.limit_ns);
  __syncwarp();
}

// ---------------------------------------------------------------------------
// sparse: E4M3 dequantisation, row copies
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t pair_dequant2(uint32_t codes16, float scale) {
  return e4m3x2_scaled_bf16x2(codes16, scale);
}

// Dequantise one token's 128 codes of a value block in place: the codes sit
// as a plain 128-byte row at row `tok` of chunk `hi_chunk`; values 0..63 go
// to row `tok` of `lo_chunk`, 64..127 to row `tok` of `hi_chunk`, in the
// 128-byte swizzle (16-byte unit u of row t at u ^ (t & 7)).  An invalid
// token's values become zeros.
__device__ __forceinline__ void dequant_block_row(uint32_t lo, uint32_t hi, uint32_t tsw, float scale, bool ok) {
  uint4 raw[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) raw[k] = ld_shared_v4(hi + ((k ^ tsw) << 4));
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t u = k ^ tsw;  // raw unit: codes 16u .. 16u + 15 of the block
    const uint32_t dst = (u & 4) ? hi : lo;
    const uint32_t k0 = (2 * (u & 3)) ^ tsw, k1 = (2 * (u & 3) + 1) ^ tsw;
    uint4 v = raw[k];
    if (!ok) v = make_uint4(0, 0, 0, 0);
    st_shared_v4(dst + (k0 << 4), pair_dequant2(v.x & 0xffffu, scale), pair_dequant2(v.x >> 16, scale),
                 pair_dequant2(v.y & 0xffffu, scale), pair_dequant2(v.y >> 16, scale));
    st_shared_v4(dst + (k1 << 4), pair_dequant2(v.z & 0xffffu, scale), pair_dequant2(v.z >> 16, scale),
                 pair_dequant2(v.w & 0xffffu, scale), pair_dequant2(v.w >> 16, scale));
  }
}

// Tile iterator of a role that runs ahead of the others.
struct PairIt {
  int prob, j, te;
  bool valid;
};
__device__ __forceinline__ PairIt pair_first_from(const PairSeg& sg, int prob) {
  for (; prob <= sg.last(); ++prob) {
    int tb, te;
    sg.range(prob, tb, te);
    if (tb < te) return PairIt{prob, tb, te, true};
  }
  return PairIt{0, 0, 0, false};
}
__device__ __forceinline__ PairIt pair_next(const PairSeg& sg, const PairIt& it) {
  if (!it.valid) return it;
  if (it.j + 1 < it.te) return PairIt{it.prob, it.j + 1, it.te, true};
  return pair_first_from(sg, it.prob + 1);
}

// Cache row of the token in index slot k of problem prob, or -1 for an
// invalid id (outside [0, length) or on an unusable page, flagged when asked).
__device__ __forceinline__ int sparse_row(const DecodeParams& p, const PairSeg& sg, int prob, int k, bool flag) {
  // (the length, the list length and the index are independent loads, in flight together)
  const int b = prob / p.s_q;
  const int L = p.flat_rows > 0 ? p.flat_rows : sg.seqlens[b];
  int tk = p.topk;
  if (p.topk_lengths) {
    const int len = p.topk_lengths[prob];
    tk = len < 0 ? 0 : (len < p.topk ? len : p.topk);
  }
  const int t = k < tk ? p.indices[static_cast<int64_t>(prob) * p.topk + k] : -1;
  if (t < 0 || t >= L) return -1;
  if (p.flat_rows > 0) return t;  // unpaged rows: the index is the row
  const int32_t* bt = p.block_table + static_cast<int64_t>(b) * p.block_table_stride;
  const int page = (t >> 6) < p.block_table_stride ? bt[t >> 6] : -1;
  if (page < 0 || page >= p.num_pages) {
    if (flag) atomicOr(p.status, MLA_DEVICE_BAD_PAGE);
    return -1;
  }
  return page * kPageSize + (t & 63);
}

// Prefetch `bytes` (a multiple of 16) from a 16-byte aligned address into L2.
__device__ __forceinline__ void l2_prefetch_bulk(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
               : "memory");
}

// 16-byte asynchronous copy global -> shared (L2 only); src_bytes 0 writes zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)),
               "r"(src_bytes)
               : "memory");
}
// One arrival on `bar` once every copy this thread has started is complete
// (the barrier's expected count includes it).
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// 4-byte asynchronous copy global -> shared (through L1); src_bytes 0 writes zeros.
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// Row copies of a gather warp.  Copy instruction i (0..7) of lane l moves the
// 16-byte unit l % 8 of warp token 4 i + l / 8, so that each instruction
// reads four 128-byte row segments whole.  rows[i] is that token's cache row
// (-1: invalid token).
struct WarpRows {
  int r[8];
  __device__ __forceinline__ void load(int my_row, int lane) {
#pragma unroll
    for (int i = 0; i < 8; ++i) r[i] = __shfl_sync(0xffffffffu, my_row, 4 * i + (lane >> 3));
  }
};

// The 128 codes of value block `blk` of the warp's 32 tokens, as plain 128-byte
// rows at rows wtok .. wtok + 31 of the chunk at `dst_chunk`.  An invalid
// token's codes are read from row 0 (its values are written as zeros later).
__device__ __forceinline__ void copy_block_codes(const DecodeParams& p, int row_bytes, const WarpRows& wr, int blk,
                                                 uint32_t dst_chunk, int wtok, int lane) {
  const int u = lane & 7;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = wr.r[i] < 0 ? 0 : wr.r[i];
    const int tk = wtok + 4 * i + (lane >> 3);
    cp_async16(dst_chunk + tk * 128 + 16 * u, p.kv_fp8 + static_cast<int64_t>(row) * row_bytes + 128 * blk + 16 * u,
               16);
  }
}

// Warps 12-15 (sparse): row lookups and row copies (FP8 rows: codes and
// scales, dequantised by the softmax warps; bf16 rows: both chunks of each
// block straight into the swizzle, to be handed over as they are).  Thread
// g (0..127) owns token tok = g % 64 of the CTA's half of each tile (index
// slot 64 rank + tok) and value blocks 2hh and 2hh + 1 (hh = g / 64); block
// bs = 2hh + rank is in this CTA's share of the value dims, block
// 2hh + 1 - rank in its partner's.
// Per tile:
//   * its warp copies those blocks for its 32 tokens into the score slots
//     (FP8: the codes of block b as plain rows in chunk 2b + 1, with the
//     token's scales in the first bytes of its row of chunk 2b; bf16: chunks
//     2b and 2b + 1 in the swizzle) as the score MMAs of the previous tile,
//     and for the partner's block the copier (pair_value_copier), release
//     them; the hh = 0 warps also copy the RoPE parts straight into the
//     128-byte swizzle of chunk 8 (zeros for invalid tokens).  The softmax
//     warps dequantise FP8 blocks in place and hand the blocks over to the
//     score MMAs (pair_softmax);
//   * once they have, and the PV MMAs of the previous tile are done, the
//     thread copies its token's row of block bs into this CTA's value slots
//     4 rank + 2hh, 4 rank + 2hh + 1.
// The hh = 0 warps write the tile's validity bits of their tokens to both
// CTAs, look the rows up three tiles ahead and prefetch them whole into L2,
// so that the copies on the tile's critical chain hit L2.
template <bool ROWS16>
__device__ void pair_gather(const DecodeParams& p, const PairSeg& sg, int rank, uint32_t smem, uint32_t bars,
                            const Watchdog& wd, uint32_t* flags) {
  const int g = threadIdx.x - 32 * kPairGatherWarp0;  // 0..127
  const int lane = g & 31;
  const int hh = g >> 6;
  const int tok = g & 63;
  const int wtok = tok & ~31;
  const uint32_t tsw = tok & 7;
  const int bs = 2 * hh + rank, bp = 2 * hh + 1 - rank;
  const int row_bytes = ROWS16 ? 2 * kDqk : (p.kv_scales ? 640 : kFp8RowBytes);
  const uint32_t peer = static_cast<uint32_t>(rank ^ 1);
  const uint32_t kv_own = smem + kPairKvOff + (4 * rank + 2 * hh) * kPairChunk + tok * 128;
  const uint32_t flags_here = static_cast<uint32_t>(__cvta_generic_to_shared(flags));
  const uint32_t flags_peer = mapa_shared(flags_here, peer);
  const uint32_t bars_peer = mapa_shared(bars, peer);
  uint32_t armed = 0, next_par = 0;  // raw barriers with copies of this thread (bit per item), parity of their next phase
  auto row_of = [&](const PairIt& it) {
    return it.valid ? sparse_row(p, sg, it.prob, it.j * kPairTile + 64 * rank + tok, hh == 0) : -1;
  };
  auto prefetch = [&](int row) {
    if (hh == 0 && row >= 0) l2_prefetch_bulk(p.kv_fp8 + static_cast<int64_t>(row) * row_bytes, row_bytes);
  };
  // this warp's items of tile jt into the score slots: bs, bp, (RoPE)
  auto issue = [&](int jt, int row) -> bool {
    WarpRows wr;
    wr.load(row, lane);
#pragma unroll 1
    for (int i = 0; i < (hh == 0 ? 3 : 2); ++i) {
      const int item = i == 0 ? bs : i == 1 ? bp : 4;
      if (jt > 0) {
        if (!pair_wait(bars + 8 * (kBKsEmpty + item), (jt - 1) & 1, wd)) return false;
        if (i == 1 && !pair_wait(bars + 8 * (kBKsRead + hh), (jt - 1) & 1, wd)) return false;
      }
      if (i == 0 && g == 0) PAIR_TR(rank, 0, jt);
      if (ROWS16 && item < 4) {
        // bf16 rows: the block's two chunks straight into the 128-byte swizzle
        // (zeros for invalid tokens)
        const uint32_t u = lane & 7;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const uint32_t cbase = smem + kPairKsOff + (2 * item + c) * kPairChunk;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int tk = wtok + 4 * k + (lane >> 3);
            const int r = wr.r[k];
            cp_async16(cbase + tk * 128 + ((u ^ (tk & 7)) << 4),
                       p.kv_fp8 + static_cast<int64_t>(r < 0 ? 0 : r) * row_bytes + 128 * (2 * item + c) + 16 * u,
                       r < 0 ? 0u : 16u);
          }
        }
      } else if (item < 4) {
        const uint32_t lo = smem + kPairKsOff + 2 * item * kPairChunk;
        copy_block_codes(p, row_bytes, wr, item, lo + kPairChunk, wtok, lane);
        // the token's scale(s), read by the dequantising thread before it writes its row of chunk 2b
        const uint32_t sdst = lo + tok * 128 + (tsw << 4);
        const int r0 = row < 0 ? 0 : row;
        if (p.kv_scales)
          cp_async4(sdst, p.kv_scales + r0, row < 0 ? 0u : 4u);
        else
          cp_async16(sdst, p.kv_fp8 + static_cast<int64_t>(r0) * row_bytes + kFp8ScaleOffset, row < 0 ? 0u : 16u);
      } else {
        const uint32_t u = lane & 7;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int tk = wtok + 4 * k + (lane >> 3);
          const int r = wr.r[k];
          cp_async16(smem + kPairKsOff + 8 * kPairChunk + tk * 128 + ((u ^ (tk & 7)) << 4),
                     p.kv_fp8 + static_cast<int64_t>(r < 0 ? 0 : r) * row_bytes + p.fp8_rope_off + 16 * u,
                     r < 0 ? 0u : 16u);
        }
      }
      cp_async_arrive(bars + 8 * (kBRaw + item));
      armed |= 1u << item;
      next_par ^= 1u << item;
    }
    if (g == 0) PAIR_TR(rank, 1, jt);
    return true;
  };

  // validity bits of this warp's tokens of tile t, to both CTAs (hh = 0 warps)
  auto put_flags = [&](int t, int row) {
    const uint32_t v = __ballot_sync(0xffffffffu, row >= 0);
    if (lane == 0) {
      const uint32_t word = 4 * (4 * (t & 3) + 2 * rank + (wtok >> 5));
      const uint32_t fb = 8 * (kBFlags + (t & 3));
      st_shared_u32(flags_here + word, v);
      st_cluster_u32(flags_peer + word, v);
      mbar_arrive(reinterpret_cast<uint64_t*>(__cvta_shared_to_generic(bars + fb)));
      mbar_arrive_cluster(bars_peer + fb);
    }
    __syncwarp();
  };

  PairIt it_c = pair_first_from(sg, sg.p0);
  PairIt it_1 = pair_next(sg, it_c);
  PairIt it_2 = pair_next(sg, it_1);
  int row_c = row_of(it_c), row_1 = row_of(it_1), row_2 = row_of(it_2);
  prefetch(row_1);
  prefetch(row_2);
  int jt = 0;
  if (hh == 0 && it_c.valid) put_flags(0, row_c);
  if (it_c.valid && !issue(0, row_c)) goto drain;
  for (; it_c.valid; ++jt) {
    // the bits of the next tile, a tile before its dequantisation needs them.
    // Their ring slot last held tile jt - 3's, which both CTAs' softmax warps
    // have read: issue(jt) waited for the score MMAs of tile jt - 1, which
    // follow the dequantisation of tile jt - 1, which each CTA's softmax warps
    // start after the softmax of tile jt - 2.
    if (hh == 0 && it_1.valid) put_flags(jt + 1, row_1);
    // rows of the tile three ahead (the lookup's dependent loads stall this warp)
    const PairIt it_3 = pair_next(sg, it_2);
    const int row_3 = row_of(it_3);
    const uint32_t par = static_cast<uint32_t>(jt) & 1u;
    // this CTA's value slots of block bs, once it is dequantised and the PV
    // MMAs of the previous tile are done (16-byte units in swizzled order:
    // the eight threads of a shared-memory wavefront touch eight banks)
    bool ok = pair_wait(bars + 8 * kBKsDoneOwn, par, wd);
    if (g == 0) PAIR_TR(rank, 2, jt);
    if (ok && jt > 0) ok = pair_wait(bars + 8 * kBKvEmpty, (jt - 1) & 1, wd);
    if (ok) {
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const uint32_t src = smem + kPairKsOff + (2 * bs + h2) * kPairChunk + tok * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint32_t off = (u ^ tsw) << 4;
          const uint4 v = ld_shared_v4(src + off);
          st_shared_v4(kv_own + h2 * kPairChunk + off, v.x, v.y, v.z, v.w);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(reinterpret_cast<uint64_t*>(__cvta_shared_to_generic(bars + 8 * kBKvIn)));
    }
    if (g == 0) PAIR_TR(rank, 3, jt);
    // every own-share copy of the tile is done before its score slots are
    // reloaded (every gather warp reaches this barrier: its waits are bounded)
    if (!named_bar_and(kPairGatherBar, 128, ok)) goto drain;
    prefetch(row_3);
    if (it_1.valid && !issue(jt + 1, row_1)) goto drain;
    it_c = it_1;
    it_1 = it_2;
    it_2 = it_3;
    row_c = row_1;
    row_1 = row_2;
    row_2 = row_3;
  }
  return;
drain:
  // abort: this thread's copies, then (bounded) the arrivals they trigger
  cp_async_wait_all();
#pragma unroll 1
  for (int k = 0; k < 5; ++k)
    if ((armed >> k) & 1u) pair_drain(bars + 8 * (kBRaw + k), ((next_par >> k) & 1u) ^ 1u, wd.limit_ns);
}

// 16-byte aligned bulk copy of `bytes` from this CTA's shared memory to shared
// memory of a CTA of the cluster, completing on a barrier of that CTA.
__device__ __forceinline__ void bulk_copy_s2c(uint32_t dst_cluster, uint32_t src, uint32_t bytes, uint32_t bar_cluster) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   dst_cluster),
               "r"(src), "r"(bytes), "r"(bar_cluster)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Warp 2 (sparse): the partner's value slots.  The value dims of block b of a
// token sit, dequantised, in score slots 2b and 2b + 1 of the CTA that owns
// the token (16 KB for its 64 tokens, the layout of a value-slot pair).  Per
// tile and m = 0, 1: once this CTA's gather warps have dequantised block
// 1 - rank + 2m (the partner's share) and the PV MMAs of the previous tile
// have released the slots, one thread copies it into the partner's value
// slots 4 rank + 2m, 4 rank + 2m + 1 with the bulk-copy engine, and releases
// the score slots to the gather warps once the copy has read them.  When
// this CTA's value slots of the tile are complete (its own share, written by
// its gather warps, and its partner's copies), the PV issuer of the even CTA
// is told.
__device__ void pair_value_copier(const PairSeg& sg, int rank, uint32_t smem, uint32_t bars, uint32_t bars_even,
                                  const Watchdog& wd) {
  const int lane = threadIdx.x & 31;
  const uint32_t peer = static_cast<uint32_t>(rank ^ 1);
  const uint32_t smem_peer = mapa_shared(smem, peer);
  const uint32_t kv_in_peer = mapa_shared(bars + 8 * kBKvIn, peer);
  bool pending = false;
  int jt = 0;
  for (int prob = sg.p0; prob <= sg.last(); ++prob) {
    int tb, te;
    sg.range(prob, tb, te);
    for (int j = tb; j < te; ++j, ++jt) {
      const uint32_t par = static_cast<uint32_t>(jt) & 1u;
#pragma unroll 1
      for (int m = 0; m < 2; ++m) {
        if (!pair_wait(bars + 8 * (kBKsDone + m), par, wd)) goto drain;
        if (m == 0) {
          if (jt > 0 && !pair_wait(bars + 8 * kBKvEmpty, (jt - 1) & 1, wd)) goto drain;
          // this CTA's slots receive the partner's two 16 KB copies
          if (lane == 0) mbar_arrive_expect_tx_u32(bars + 8 * kBKvIn, 2 * 2 * kPairChunk);
        }
        if (lane == 0) {
          if (m == 0) PAIR_TR(rank, 12, jt);
          const int b = 1 - rank + 2 * m;
          bulk_copy_s2c(smem_peer + kPairKvOff + (4 * rank + 2 * m) * kPairChunk, smem + kPairKsOff + 2 * b * kPairChunk,
                        2 * kPairChunk, kv_in_peer);
          bulk_commit();
          pending = true;
          bulk_wait_read_all();
          mbar_arrive(reinterpret_cast<uint64_t*>(__cvta_shared_to_generic(bars + 8 * (kBKsRead + m))));
        }
        __syncwarp();
      }
      if (!pair_wait(bars + 8 * kBKvIn, par, wd)) goto drain;
      if (lane == 0) {
        bulk_wait_all();
        pending = false;
        PAIR_TR(rank, 13, jt);
      }
      warp_arrive_even(rank, bars + 8 * kBKvFull, bars_even + 8 * kBKvFull);
    }
  }
  return;
drain:
  if (lane == 0 && pending) bulk_wait_all();
  __syncwarp();
}

// ---------------------------------------------------------------------------
// warp 1 of the even CTA: score MMAs, S = Q K^T over the pair
// ---------------------------------------------------------------------------
template <bool SPARSE>
__device__ void pair_s_issuer(const PairSeg& sg, uint32_t tmem, uint32_t smem, uint32_t bars, const Watchdog& wd) {
  using C = PairCfg<SPARSE>;
  constexpr uint32_t kIdS = idesc_bf16_f32(128, kPairTile, 0, 0);
  constexpr uint64_t kHiK = smem_desc_hi(16, 1024);
  const int lane = threadIdx.x & 31;
  int jt = 0, seg = 0;
  for (int prob = sg.p0; prob <= sg.last(); ++prob) {
    int tb, te;
    sg.range(prob, tb, te);
    if (tb >= te) continue;
    if (!pair_wait(bars + 8 * kBQFull, seg & 1, wd)) goto done;
    tc_fence_after();
    for (int j = tb; j < te; ++j, ++jt) {
      const int sb = jt & 1;
      if (jt >= 2 && !pair_wait(bars + 8 * (kBSEmpty + sb), ((jt >> 1) - 1) & 1, wd)) goto done;
      tc_fence_after();
      const uint32_t d = tmem + kPairSCol + sb * (kPairTile / 2);
#pragma unroll 1
      for (int it = 0; it < C::kItems; ++it) {
        if (!pair_wait(bars + 8 * (kBKsFull + it), jt & 1, wd)) goto done;
        tc_fence_after();
        if (lane == 0 && it == 0) PAIR_TR(0, 5, jt);
        if (lane == 0 && it == C::kItems - 1) PAIR_TR(0, 6, jt);
        const int k0 = C::item_chunk0(it), nk = C::item_chunks(it);
#pragma unroll 1
        for (int kc = 0; kc < nk; ++kc) {
          const int k = k0 + kc;
          const uint64_t a0 = kHiK | ((smem + kPairQOff + k * kPairChunk) >> 4);
          const uint64_t b0 = kHiK | ((smem + kPairKsOff + k * kPairChunk) >> 4);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            if (elect_one()) umma2_bf16_ss(d, a0 + 2 * kk, b0 + 2 * kk, kIdS, (k | kk) != 0);
            __syncwarp();
          }
        }
        if (elect_one()) umma2_commit_both(bars + 8 * (kBKsEmpty + it));
        __syncwarp();
      }
      if (elect_one()) {
        umma2_commit_both(bars + 8 * (kBSFull + sb));
        if (j == te - 1) umma2_commit_both(bars + 8 * kBQEmpty);
      }
      __syncwarp();
    }
    ++seg;
  }
done:
  if (elect_one()) umma2_commit_own(bars + 8 * kBMmaDone);
  __syncwarp();
  if (lane == 0) pair_drain(bars + 8 * kBMmaDone, 0, wd.limit_ns);
  __syncwarp();
}

// ---------------------------------------------------------------------------
// warp 3 of the even CTA: PV MMAs, O += P V over the pair
// ---------------------------------------------------------------------------
__device__ void pair_pv_issuer(const PairSeg& sg, uint32_t tmem, uint32_t smem, uint32_t bars, const Watchdog& wd) {
  constexpr uint32_t kIdO = idesc_bf16_f32(128, 256, 0, 1);  // A = P (K-major), B = V (MN-major)
  constexpr uint64_t kHiP = smem_desc_hi(16, 1024);
  constexpr uint64_t kHiV = smem_desc_hi(kPairChunk, 1024);
  const int lane = threadIdx.x & 31;
  int jt = 0, seg = 0;
  for (int prob = sg.p0; prob <= sg.last(); ++prob) {
    int tb, te;
    sg.range(prob, tb, te);
    if (tb >= te) continue;
    for (int j = tb; j < te; ++j, ++jt) {
      const bool first = (j == tb), last = (j == te - 1);
      if (!pair_wait(bars + 8 * kBPFull, jt & 1, wd)) goto done;
      if (!pair_wait(bars + 8 * kBKvFull, jt & 1, wd)) goto done;
      tc_fence_after();
      if (lane == 0) PAIR_TR(0, 10, jt);
      if (first && seg > 0) {
        if (!pair_wait(bars + 8 * kBOEmpty, (seg - 1) & 1, wd)) goto done;
        tc_fence_after();
      }
#pragma unroll
      for (int m = 0; m < 2; ++m) {
#pragma unroll
        for (int kk = 0; kk < kPairTile / 16; ++kk) {
          const int t = kk >> 2;
          const uint64_t a = kHiP | ((smem + kPairPOff + t * kPairChunk + 32 * (kk & 3)) >> 4);
          const uint64_t bdesc =
              kHiV | ((smem + kPairKvOff + (4 * t + 2 * m) * kPairChunk + 2048 * (kk & 3)) >> 4);
          if (elect_one()) umma2_bf16_ss(tmem + kPairOCol + 128 * m, a, bdesc, kIdO, !(first && kk == 0));
          __syncwarp();
        }
      }
      if (elect_one()) {
        umma2_commit_both(bars + 8 * kBPEmpty);
        umma2_commit_both(bars + 8 * kBKvEmpty);
        if (last) umma2_commit_both(bars + 8 * kBOFull);
      }
      __syncwarp();
      if (lane == 0) PAIR_TR(0, 11, jt);
    }
    ++seg;
  }
done:
  if (elect_one()) umma2_commit_own(bars + 8 * kBMmaDone);
  __syncwarp();
  if (lane == 0) pair_drain(bars + 8 * kBMmaDone, 0, wd.limit_ns);
  __syncwarp();
}

// ---------------------------------------------------------------------------
// warps 4-11: online softmax and epilogue
// ---------------------------------------------------------------------------
template <bool SPARSE, bool ROWS16>
__device__ void pair_softmax(const DecodeParams& p, const PairSeg& sg, int g, int rank, int split0, uint32_t tmem,
                             uint32_t smem, uint32_t bars, uint32_t bars_even, float* m_s, float* red,
                             const volatile uint32_t* flags, const Watchdog& wd) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int q = warp & 3;           // TMEM lane quarter
  const int h = q >> 1;             // half of the tile this thread's columns cover
  const int w = (warp - 4) >> 2;    // warpgroup: tokens [32w, 32w + 32) of the half
  const int r = (q & 1) * 32 + lane;  // row of this CTA (0..63)
  const int hw = 2 * h + w;         // which of the row's four partial statistics
  const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
  const int row0 = g * 2 * kPairRows + rank * kPairRows;
  const int grow = row0 + r;        // row within the problem
  const float sc = p.scale_log2;
  auto arrive_even = [&](int bar) { warp_arrive_even(rank, bars + 8 * bar, bars_even + 8 * bar); };
  auto all_ok = [&](bool ok) { return named_bar_and(kPairSmBar, 256, ok); };
  // signal slots of this CTA and of the even CTA (see the P-ready hand-over below)
  const uint32_t sig = smem + kPairAuxOff + kPairSigOff;
  const uint32_t sig_even = mapa_shared(sig, 0);
  // Hand-over of shared memory written by this warp's threads (after each
  // thread's proxy fence) to the pair's MMAs, on the even CTA's barrier
  // `bar`: the even CTA's two writing warps arrive (the first expecting the
  // odd CTA's 32 signal bytes); each of the odd CTA's two writing warps has
  // one lane issue a 16-byte async copy into the even CTA that completes on
  // the barrier -- no cluster-scope release stalls these warps.
  auto hand_over = [&](int bar, bool first, int slot) {
    __syncwarp();
    if (lane == 0) {
      if (rank == 0) {
        uint64_t* b = reinterpret_cast<uint64_t*>(__cvta_shared_to_generic(bars + 8 * bar));
        if (first)
          mbar_arrive_expect_tx(b, 32);
        else
          mbar_arrive(b);
      } else {
        bulk_copy_s2c(sig_even + 16 * slot, sig + 16 * slot, 16, bars_even + 8 * bar);
        bulk_commit();
      }
    }
  };
  auto wait_all = [&](int bar, uint32_t parity) { return all_ok(mbar_wait(
      reinterpret_cast<uint64_t*>(__cvta_shared_to_generic(bars + 8 * bar)), parity, wd)); };
  if (p.debug_stall) {
    // watchdog test: this barrier's first phase only completes when this role has finished
    if (!wait_all(kBMmaDone, 0)) return;
  }
  // Sparse: the score operand of tile t is dequantised here, one block row per
  // thread (warp 4 + 2b + k: block b, tokens 32k .. 32k + 31 of the CTA's
  // half), as soon as P of the previous tile is handed over: the softmax
  // warps are otherwise idle while the tile's rows arrive.  (Converting the
  // blocks one after the other with all eight warps, so that the score MMAs
  // of a block could start while the next is converted, measured slower: the
  // conversions are bound by the conversion pipe's rate, and the per-block
  // barriers of all 256 threads cost more than the overlap gave.)
  int tiles = 0;
  if (SPARSE) {
    for (int pr = sg.p0; pr <= sg.last(); ++pr) {
      int tb, te;
      sg.range(pr, tb, te);
      if (te > tb) tiles += te - tb;
    }
  }
  auto dequant_tile = [&](int t) -> bool {
    const int dw = warp - 4;
    const int blk = dw >> 1, tg = dw & 1;
    const int tok = 32 * tg + lane;
    const uint32_t tsw = tok & 7;
    if (!all_ok(pair_wait_thread(bars + 8 * (kBFlags + (t & 3)), (t >> 2) & 1, wd))) return false;
    if (warp == 4 && lane == 0) PAIR_TR(rank, 14, t);
    const bool ok = ((flags[4 * (t & 3) + 2 * rank + tg] >> lane) & 1u) != 0;
    if (!all_ok(pair_wait_thread(bars + 8 * (kBRaw + blk), t & 1, wd))) return false;
    if (warp == 4 && lane == 0) PAIR_TR(rank, 15, t);
    if (!ROWS16) {
      const uint32_t lo = smem + kPairKsOff + 2 * blk * kPairChunk + tok * 128;
      const float scale = ld_shared_f32(lo + (tsw << 4) + (p.kv_scales ? 0 : 4 * blk));
      dequant_block_row(lo, lo + kPairChunk, tsw, scale, ok);
    }
    // (bf16 rows were copied into place: only their hand-over to the MMAs)
    fence_proxy_async_smem();
    hand_over(kBKsFull + blk, tg == 0, dw);
    if (lane == 0)
      mbar_arrive(reinterpret_cast<uint64_t*>(
          __cvta_shared_to_generic(bars + 8 * ((blk & 1) == rank ? kBKsDoneOwn : kBKsDone + (blk >> 1)))));
    // the RoPE part landed in its final layout
    const bool rope_ok = dw < 2 ? pair_wait_thread(bars + 8 * (kBRaw + 4), t & 1, wd) : true;
    if (!all_ok(rope_ok)) return false;
    if (dw < 2) {
      fence_proxy_async_smem();
      hand_over(kBKsFull + 4, dw == 0, 8 + dw);
    }
    if (warp == 4 && lane == 0) PAIR_TR(rank, 4, t);
    return true;
  };
  if (SPARSE && tiles > 0 && !dequant_tile(0)) return;

  int jt = 0, seg = 0;
  for (int prob = sg.p0; prob <= sg.last(); ++prob) {
    int tb, te;
    sg.range(prob, tb, te);
    if (tb >= te) continue;
    const int b = SPARSE ? prob / p.s_q : prob;
    const int L = SPARSE ? 0 : sg.seqlens[b];  // (sparse: the validity bits, and no lengths for unpaged rows)
    // last visible key of this row (dense: bottom-right causal alignment)
    const int lim = (!SPARSE && p.is_causal) ? L - p.s_q + grow / p.h_q : L - 1;
    float l_part = 0.f;
    for (int j = tb; j < te; ++j, ++jt) {
      const int sb = jt & 1;
      // dense: the block-table entry of this thread's page, read before the
      // wait for S so that the load overlaps it
      const bool page_ok = SPARSE ? true : tile_page(p, b, L, j, h, false) >= 0;
      if (!wait_all(kBSFull + sb, (jt >> 1) & 1)) return;
      tc_fence_after();
      const bool tr = (warp == 4 && lane == 0);
      if (tr) PAIR_TR(rank, 7, jt);
      float x[32];
      tmem_ld_x32(tmem + lane_base + kPairSCol + sb * (kPairTile / 2) + 32 * w, x);
      tmem_ld_wait();
      tc_fence_before();
      // S read: the loads have completed (wait::ld) and the tcgen05 fence
      // orders them before the signal, which orders no memory access of its
      // own, so the odd CTA's arrival on the even CTA's barrier is relaxed (a
      // cluster-scope release would stall these warps for ~1k cycles per tile)
      __syncwarp();
      if (lane == 0) {
        if (rank == 0)
          mbar_arrive(reinterpret_cast<uint64_t*>(__cvta_shared_to_generic(bars + 8 * (kBSEmpty + sb))));
        else
          mbar_arrive_cluster_relaxed(bars_even + 8 * (kBSEmpty + sb));
      }
      // mask and scale (log2 units); tokens of this thread: h * 64 + 32 w + i
      uint32_t vbits = 0xffffffffu;
      if (SPARSE) {
        // the gather warps of this CTA wrote the tile's validity bits
        if (!all_ok(pair_wait_thread(bars + 8 * (kBFlags + (jt & 3)), (jt >> 2) & 1, wd))) return;
        vbits = flags[4 * (jt & 3) + 2 * h + w];
      }
      const int pos0 = j * kPairTile + h * 64 + 32 * w;
      float mx = kPairNegInf;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const bool ok = SPARSE ? ((vbits >> i) & 1u) != 0 : (page_ok && pos0 + i <= lim);
        x[i] = ok ? x[i] * sc : kPairNegInf;
        mx = fmaxf(mx, x[i]);
      }
      red[hw * 64 + r] = mx;
      named_bar_sync(kPairSmBar, 256);
      const float rmax = fmaxf(fmaxf(red[r], red[64 + r]), fmaxf(red[128 + r], red[192 + r]));
      const float m_old = (j == tb) ? kPairNegInf : m_s[r];
      const bool raise = (j == tb) || (rmax > m_old + kPairRescale);
      const float m_new = raise ? fmaxf(m_old, rmax) : m_old;
      // any row of either warpgroup raised its max (after the first tile): O needs a rescale
      const bool any = named_bar_or(kPairSmBar, 256, raise && j != tb);
      if (raise && hw == 0) m_s[r] = m_new;
      const float alpha = (m_old == kPairNegInf) ? 0.f : fast_exp2(m_old - m_new);
      if (raise) l_part *= alpha;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        x[i] = (x[i] == kPairNegInf) ? 0.f : fast_exp2(x[i] - m_new);
        l_part += x[i];
      }
      // P and O of the previous tile are free once its PV MMAs are done
      if (jt > 0 && !wait_all(kBPEmpty, (jt - 1) & 1)) return;
      tc_fence_after();
      if (tr) PAIR_TR(rank, 8, jt);
      if (any) {
        // rescale this thread's row of O (its lane's 128 columns of block w) by alpha
        const float a = raise ? alpha : 1.0f;
#pragma unroll 1
        for (int c = 0; c < 128; c += 16) {
          float v[16];
          const uint32_t ta = tmem + lane_base + kPairOCol + 128 * w + c;
          tmem_ld_x16(ta, v);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] *= a;
          tmem_st_x16(ta, v);
        }
        tmem_st_wait();
      }
      // P (bf16, K-major, 128-byte swizzle): row r, tokens 32w .. 32w + 31 of chunk h
      {
        const uint32_t prow = smem + kPairPOff + h * kPairChunk + r * 128;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int unit = 4 * w + u;
          st_shared_v4(prow + ((unit ^ (r & 7)) << 4), pack_bf16x2(x[8 * u], x[8 * u + 1]),
                       pack_bf16x2(x[8 * u + 2], x[8 * u + 3]), pack_bf16x2(x[8 * u + 4], x[8 * u + 5]),
                       pack_bf16x2(x[8 * u + 6], x[8 * u + 7]));
        }
      }
      // dense tail tile: this CTA's value slots are loaded (on its own
      // barrier); the rows of tokens past the length are zeroed (their P is
      // 0, but a slot may hold NaN, and 0 * NaN would poison O).  Unusable
      // pages were read as zeros.  (Sparse: invalid tokens were written as
      // zeros by the gather warps.)
      if (!SPARSE && tail_tile(L, j)) {
        if (!wait_all(kBKvFull, jt & 1)) return;
        const int tl = (q & 1) * 32 + lane;  // token of page h zeroed by this thread
        if (page_ok && j * kPairTile + h * 64 + tl >= L) {
#pragma unroll
          for (int s2 = 0; s2 < 2; ++s2) {
            const uint32_t rowa = smem + kPairKvOff + (4 * h + 2 * w + s2) * kPairChunk + tl * 128;
#pragma unroll
            for (int u = 0; u < 8; ++u) st_shared_v4(rowa + 16 * u, 0u, 0u, 0u, 0u);
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      // P ready.  Even CTA: one arrival per warp (the first also expects the
      // odd CTA's 16 signal bytes).  Odd CTA: its P (and any zeroed value rows)
      // were made visible to the async proxy by each thread's proxy fence; the
      // softmax threads meet, and one of them issues a 16-byte async copy into
      // the even CTA that completes on its P-ready barrier -- the hand-over of
      // data written by threads to the tensor core that TMA stores use, and it
      // does not stall the issuing warps as a cluster-scope release does.
      if (rank == 0) {
        __syncwarp();
        if (lane == 0) {
          uint64_t* pb = reinterpret_cast<uint64_t*>(__cvta_shared_to_generic(bars + 8 * kBPFull));
          if (warp == 4)
            mbar_arrive_expect_tx(pb, 16);
          else
            mbar_arrive(pb);
        }
      } else {
        named_bar_sync(kPairSmBar, 256);
        if (threadIdx.x == 128) {
          bulk_copy_s2c(sig_even + 16 * 10, sig + 16 * 10, 16, bars_even + 8 * kBPFull);
          bulk_commit();
        }
      }
      if (tr) PAIR_TR(rank, 9, jt);
      if (SPARSE && jt + 1 < tiles && !dequant_tile(jt + 1)) return;
    }

    // ---- epilogue: O / l -> out (single piece) or fp32 partial (split problem)
    if (!wait_all(kBOFull, seg & 1)) return;
    tc_fence_after();
    red[hw * 64 + r] = l_part;
    named_bar_sync(kPairSmBar, 256);
    const float lt = red[r] + red[64 + r] + red[128 + r] + red[192 + r];
    const float m_fin = m_s[r];
    named_bar_sync(kPairSmBar, 256);  // red and m_s are reused by the next segment
    const float inv = lt > 0.f ? 1.0f / lt : 0.f;
    const float lse = lt > 0.f ? m_fin + log2f(lt) : kPairNegInf;
    const int nsplit = p.num_splits[prob + 1] - p.num_splits[prob];
    const bool final_out = nsplit <= 1;
    const int slot = p.num_splits[prob] + (prob == sg.p0 ? split0 : 0);
    bool write_ok = grow < p.rows;
    if (!final_out && (slot < 0 || slot >= p.max_slots)) {
      write_ok = false;
      if (r == 0 && hw == 0) atomicOr(p.status, MLA_DEVICE_BAD_SCHEDULE);
    }
    const int dv0 = 256 * w + 128 * h;
    const int64_t orow = final_out ? static_cast<int64_t>(prob) * p.rows + grow
                                   : static_cast<int64_t>(slot) * p.rows + grow;
#pragma unroll 1
    for (int c = 0; c < 128; c += 16) {
      float v[16];
      tmem_ld_x16(tmem + lane_base + kPairOCol + 128 * w + c, v);
      tmem_ld_wait();
      if (write_ok) {
        if (final_out) {
          uint4 lo, hi;
          lo.x = pack_bf16x2(v[0] * inv, v[1] * inv);
          lo.y = pack_bf16x2(v[2] * inv, v[3] * inv);
          lo.z = pack_bf16x2(v[4] * inv, v[5] * inv);
          lo.w = pack_bf16x2(v[6] * inv, v[7] * inv);
          hi.x = pack_bf16x2(v[8] * inv, v[9] * inv);
          hi.y = pack_bf16x2(v[10] * inv, v[11] * inv);
          hi.z = pack_bf16x2(v[12] * inv, v[13] * inv);
          hi.w = pack_bf16x2(v[14] * inv, v[15] * inv);
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + orow * kDv + dv0 + c);
          dst[0] = lo;
          dst[1] = hi;
        } else {
          float4* dst = reinterpret_cast<float4*>(p.o_accum + orow * kDv + dv0 + c);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_float4(v[4 * e] * inv, v[4 * e + 1] * inv, v[4 * e + 2] * inv, v[4 * e + 3] * inv);
        }
      }
    }
    if (write_ok && hw == 0) {
      if (final_out)
        p.lse[orow] = lse;
      else
        p.lse_accum[orow] = lse;
    }
    tc_fence_before();
    arrive_even(kBOEmpty);
    ++seg;
  }
}

// ---------------------------------------------------------------------------
// kernel
// ---------------------------------------------------------------------------
template <bool SPARSE, bool ROWS16>
__global__ void __launch_bounds__(PairCfg<SPARSE>::kThreads, 1)
    mla_decode_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_ks,
                           const __grid_constant__ CUtensorMap tm_kv, const DecodeParams p) {
  using C = PairCfg<SPARSE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t smem = smem_u32(base);
  const uint32_t bars = smem + kPairAuxOff;
  float* m_s = reinterpret_cast<float*>(base + kPairAuxOff + kPairMOff);
  float* red = reinterpret_cast<float*>(base + kPairAuxOff + kPairRedOff);
  int* ints = reinterpret_cast<int*>(base + kPairAuxOff + kPairIntOff);
  uint32_t* flags = reinterpret_cast<uint32_t*>(base + kPairAuxOff + kPairFlagOff);
  volatile int* abort_flag = ints;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ints + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_ctarank());
  const int pair_id = blockIdx.x >> 1;
  const int part = pair_id / p.row_groups;
  const int g = pair_id % p.row_groups;

  if (threadIdx.x == 0) {
    uint64_t* bp = reinterpret_cast<uint64_t*>(base + kPairAuxOff);
    mbar_init(bp + kBQFull, 1);
    mbar_init(bp + kBQEmpty, 1);
    for (int it = 0; it < C::kItems; ++it) {
      // dense: the even producer's arrival plus both CTAs' bytes; sparse: the
      // two gather warps converting the item in each CTA
      // sparse: each item by two softmax warps of each CTA
      mbar_init(bp + kBKsFull + it, SPARSE ? 2 : 1);  // sparse: the even CTA's two writing warps (+ 32 bytes)
      mbar_init(bp + kBKsEmpty + it, 1);
    }
    mbar_init(bp + kBKvFull, SPARSE ? 2 : 1);  // sparse: the value-slot copier of each CTA
    mbar_init(bp + kBKvEmpty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bp + kBSFull + i, 1);
      mbar_init(bp + kBSEmpty + i, 16);  // 8 softmax warps in each CTA
    }
    mbar_init(bp + kBPFull, 8);  // the even CTA's 8 softmax warps (+ 16 bytes from the odd CTA)
    mbar_init(bp + kBPEmpty, 1);
    mbar_init(bp + kBOFull, 1);
    mbar_init(bp + kBOEmpty, 16);
    mbar_init(bp + kBMmaDone, 2);  // one commit per MMA-issuing warp
    if (SPARSE) {
      for (int k = 0; k < 5; ++k) mbar_init(bp + kBRaw + k, 64);   // the copies of the 64 threads of the item
      for (int k = 0; k < 4; ++k) mbar_init(bp + kBFlags + k, 4);  // the hh = 0 gather warps of both CTAs
      for (int k = 0; k < 2; ++k) {
        mbar_init(bp + kBKsDone + k, 2);  // the two softmax warps dequantising the block
        mbar_init(bp + kBKsRead + k, 1);  // the copier
      }
      mbar_init(bp + kBKsDoneOwn, 4);     // the four softmax warps dequantising blocks rank, rank + 2
      mbar_init(bp + kBKvIn, 5);  // the four gather warps and the copier's arming, plus the partner's bytes
    }
    for (int k = 0; k < 16; ++k) flags[k] = 0;
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    if (!SPARSE) tma_prefetch_desc(&tm_ks);
    if (!SPARSE) tma_prefetch_desc(&tm_kv);
  }
  if (warp == 2) {
    tmem_alloc_pair(tmem_slot, kPairTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  // both CTAs' barriers are initialised before any remote arrival or commit
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t bars_even = mapa_shared(bars, 0);

  Watchdog wd{abort_flag, p.status, p.timeout_ns};
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  PairSeg sg;
  int split0 = 0;
  if (p.sched[kSchedParts] == p.num_parts && p.sched[kSchedTag] == p.sched_tag) {
    const int32_t* sr = p.sched + static_cast<int64_t>(part) * kSchedInts;
    sg.p0 = sr[kSchedP0];
    sg.t0 = sr[kSchedT0];
    sg.p1 = sr[kSchedP1];
    sg.t1 = sr[kSchedT1];
    split0 = sr[kSchedSplit0];
  } else {
    sg.p0 = -1;
    sg.t0 = sg.p1 = sg.t1 = 0;
  }
  sg.np = p.num_problems;
  sg.s_q = p.s_q;
  sg.topk = SPARSE ? p.topk : 0;
  sg.seqlens = p.cache_seqlens;
  if (sg.p0 < 0 || sg.p0 > sg.np || sg.p1 < sg.p0 || sg.p1 > sg.np || sg.t0 < 0 || sg.t1 < 0) {
    if (threadIdx.x == 0) atomicOr(p.status, MLA_DEVICE_BAD_SCHEDULE);
    sg.p0 = sg.np;
    sg.p1 = sg.np;
  }

#ifdef MLA_TRACE
  if (threadIdx.x == 0 && blockIdx.x < 1024) {
    g_pair_cta[3 * blockIdx.x] = global_timer_ns();
    int n = 0;
    for (int pr = sg.p0; pr <= sg.last(); ++pr) {
      int tb, te;
      sg.range(pr, tb, te);
      if (te > tb) n += te - tb;
    }
    g_pair_cta[3 * blockIdx.x + 2] = n;
  }
#endif
  if (warp < 4) {
    regs_to<C::kRegsCtl, C::kLaunchRegs>();
    if (warp == 0) {
      pair_producer_ks<SPARSE>(&tm_q, &tm_ks, p, sg, g, rank, smem, bars, bars_even, wd);
    } else if (warp == 1) {
      if (rank == 0) pair_s_issuer<SPARSE>(sg, tmem, smem, bars, wd);
    } else if (warp == 2) {
      if (SPARSE)
        pair_value_copier(sg, rank, smem, bars, bars_even, wd);
      else
        pair_producer_kv(&tm_kv, p, sg, rank, smem, bars, bars_even, wd);
    } else if (rank == 0) {
      pair_pv_issuer(sg, tmem, smem, bars, wd);
    }
  } else if (warp < kPairGatherWarp0) {
    regs_to<C::kRegsSm, C::kLaunchRegs>();
    pair_softmax<SPARSE, ROWS16>(p, sg, g, rank, split0, tmem, smem, bars, bars_even, m_s, red, flags, wd);
    // the odd CTA's signal copies are complete before the pair's final sync
    if (rank == 1 && (threadIdx.x & 31) == 0) bulk_wait_all();
  } else if (SPARSE) {
    regs_to<C::kRegsGather, C::kLaunchRegs>();
    pair_gather<ROWS16>(p, sg, rank, smem, bars, wd, flags);
  }

  tc_fence_before();
  __syncthreads();
#ifdef MLA_TRACE
  if (threadIdx.x == 0 && blockIdx.x < 1024) g_pair_cta[3 * blockIdx.x + 1] = global_timer_ns();
#endif
  if (*abort_flag) {
    // after a timeout, copies the odd CTA issued may still be landing in its
    // shared memory (their completions go to the even CTA): give them time
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 50000) {
    }
  }
  // neither CTA leaves while its partner may still read its shared memory,
  // arrive on its barriers or run MMAs on its TMEM
  cluster_sync_all();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kPairTmemCols);
  }
}

template <bool SPARSE, bool ROWS16>
cudaError_t launch_pair(const CUtensorMap& tm_q, const CUtensorMap& tm_ks, const CUtensorMap& tm_kv,
                        const DecodeParams& p, cudaStream_t stream) {
  using C = PairCfg<SPARSE>;
  auto kern = mla_decode_pair_kernel<SPARSE, ROWS16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmemBytes);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != static_cast<int>(C::kLaunchRegs)) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * p.num_parts * p.row_groups);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = kPairSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, tm_q, tm_ks, tm_kv, p);
}

}  // namespace

int pair_cluster_capacity() {
  auto kern = mla_decode_pair_kernel<true, false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmemBytes) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(PairCfg<true>::kThreads);
  cfg.dynamicSmemBytes = kPairSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return 0;
  return n;
}

cudaError_t launch_decode_pair(const CUtensorMap& tm_q, const CUtensorMap& tm_ks, const CUtensorMap& tm_kv,
                               const DecodeParams& p, bool sparse, cudaStream_t stream) {
  if (!sparse) return launch_pair<false, false>(tm_q, tm_ks, tm_kv, p, stream);
  return p.rows16 ? launch_pair<true, true>(tm_q, tm_ks, tm_kv, p, stream)
                  : launch_pair<true, false>(tm_q, tm_ks, tm_kv, p, stream);
}

}  // namespace mla
