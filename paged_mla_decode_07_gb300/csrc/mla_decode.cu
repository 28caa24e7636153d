// K1 — split-KV paged MLA decode on sm_103a (tcgen05 tensor cores, TMEM
// accumulators, TMA), dense bf16 and sparse FP8 modes.
//
// What is computed (per query row r of a problem and a range of its keys):
// out = softmax(q K^T * sm_scale) V with V = K[:, :512] — the MQA form of MLA
// (Modular design-doc overview, section 9 "Multi-Head Latent Attention") —
// with online softmax across 64-token tiles (overview, section 6 "Matmul to
// Flash Attention": running row max, exp(old_max - new_max) correction of
// the running sum and output).  A CTA covering only part of a problem's keys
// writes an fp32 partial and its log-sum-exp for the combine kernel
// ("split-KV", FlashMLA article, Design 5; overview, section 6).
//
// Formulation: the MMAs run transposed, as proposed in the overview's section
// 8 "U/WGMMA Flash Decoding" (option 0: P goes back through shared memory):
//     S^T[tok, row] = K[tok, :] . Q[row, :]^T      M = 64 tokens, N = rows, K = 576
//     O^T[dv, row] += V^T[dv, tok] . P^T[tok, row]  M = 128 dv (x4), N = rows, K = 64 tokens
// A KV tile is one 64-token page.  An M = 64 MMA costs as many cycles as an
// M = 128 one at these N, but halving the tile lets shared memory hold two
// tiles beside Q, so the next tile loads while the current one is in the
// softmax and PV stages.  The fp32 accumulator O^T (4*rows TMEM columns) fits
// beside the two S^T buffers in 512 columns.  The same shared-memory K tile is
// the K-major A operand of the first MMA and (dims 0..511) the MN-major A
// operand of the second; no separate V load.
//
// Shared memory (1024-byte aligned):
//   KV ring : kNA pair slots (2 chunks of [64 tokens][64 dims] bf16, 128-byte
//             swizzle = one 128-dv block of V) + kNB RoPE-chunk slots
//   Q       : 9 chunks x [rows][64 dims] bf16, 128-byte swizzle  (rows*1152 B)
//   P       : per tile, bf16; in the tile's RoPE slot with 64 rows (dead once
//             S^T is computed), else a separate double buffer
//   barriers, row statistics
// TMEM: O^T at columns [0, 4*rows), S^T double buffer at [4*rows, 6*rows)
// (an M = 64 result fills lanes 0..15 of each 32-lane quarter).
//
// Pipeline: the MMA warp issues S^T of tile j+1 before the PV MMAs of tile j,
// so the tensor pipe computes scores while the softmax warps turn the
// previous scores into P; loads run up to two tiles ahead.
//
// Warp roles: warp 0 = TMA producer (Q; dense KV pages), warp 1 = MMA
// issuer, warp 2 = TMEM allocator, warps 4.. = softmax + epilogue (one or two
// warpgroups; lane l < 16 of warp q owns token 16q + l of the tile, and every
// lane a dv row of O^T in the epilogue), sparse only: four more warps gather
// the FP8 rows with TMA row gathers and dequantise them (two threads per token).
//
// The FP8 row (FlashMLA article, Design 2): 512 e4m3 codes, 4 fp32 scales
// (one per 128 dims), 64 bf16 RoPE values; dequantised value =
// bf16_rn(fp32(e4m3) * scale), computed here as e4m3x2 -> f16x2 (exact),
// f16 -> f32 (exact), one fp32 multiply, cvt.rn to bf16.
//
// Every wait is bounded (watchdog); on expiry the CTA records
// MLA_DEVICE_TIMEOUT, all roles unwind, in-flight copies and MMAs are drained
// with a bounded wait, and TMEM is freed.
#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {

// Pipeline tracing (built only with -DMLA_TRACE): clock64() stamps of the
// main pipeline events of CTA 0, one slot per (event, tile).
enum TraceEvent {
  kTrProdChunk0 = 0, kTrProdChunk8, kTrMmaKv0, kTrMmaKv8, kTrMmaSDone, kTrSmSFull, kTrSmVote, kTrSmPFull,
  kTrMmaPFull, kTrMmaODone, kTrGatherStart, kTrGatherDone, kTrEpiStart, kTrEpiEnd, kTrSmLoaded, kTrSmPStored,
  kTrMmaO1, kTrSmWaitS, kTrW1Loaded, kTrW2Loaded, kTrW3Loaded, kTrW0PreVote, kTrW1PreVote, kTrW2PreVote,
  kTrW3PreVote, kTrProdC = kTrW3PreVote + 1, kTrMmaC = kTrProdC + 9, kTrFine = kTrMmaC + 9, kTrNumEvents = kTrFine + 8
};
#ifdef MLA_TRACE
constexpr int kTraceTiles = 1024;
__device__ unsigned long long g_mla_trace[kTrNumEvents * kTraceTiles];
// per CTA (up to 1024): %globaltimer when its work starts and when it ends, its SM
__device__ unsigned long long g_mla_cta[3 * 1024];
#define MLA_TR(ev, idx)                                                                      \
  do {                                                                                       \
    if (blockIdx.x == 0 && (idx) < kTraceTiles) g_mla_trace[(ev) * kTraceTiles + (idx)] = clock64(); \
  } while (0)
#else
#define MLA_TR(ev, idx) \
  do {                  \
  } while (0)
#endif

namespace {

constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P <= 2^8 before a max update is forced
constexpr uint32_t kSoftmaxBar = 1;        // named barrier of the 128 softmax threads

// Kernel modes: dense decode over the bf16 cache, sparse (top-k) decode over
// the FP8 cache, dense decode over the FP8 cache, sparse over bf16 rows (the
// paged bf16 cache, or an unpaged KV for sparse prefill).
constexpr int kModeDense = 0, kModeSparse = 1, kModeDenseFp8 = 2, kModeSparseBf16 = 3;

template <int R, int MODE>
struct Cfg {
  // Rows other than whole bf16 pages are gathered by four extra warps (FP8
  // rows dequantised, bf16 rows put into the swizzled operand layout); sparse
  // problems are (batch element, query token) pairs with their own indices
  static constexpr bool kGather = MODE != kModeDense;
  static constexpr bool kIndexed = MODE == kModeSparse || MODE == kModeSparseBf16;
  static constexpr bool kFp8 = MODE == kModeSparse || MODE == kModeDenseFp8;
  // softmax warpgroups: with 64 rows two warpgroups split the rows
  static constexpr int kSmWG = (R == 64) ? 2 : 1;
  static constexpr int kGatherWarp0 = 4 + 4 * kSmWG;  // sparse: first FP8 gather warp
  static constexpr int kWarps = kGatherWarp0 + (kGather ? 4 : 0);
  // With two softmax warpgroups the producer/MMA warpgroup hands registers to
  // the others (setmaxnreg).  Gathered modes: 512 threads launched at 128
  // registers, 128*64 + 2*128*168 + 128*112 = 65536 (the softmax needs 168
  // to run without spilling).  Dense: 384 threads at 168, 128*88 + 2*128*208 = 64512.  The host checks the compiled register count
  // against kRegBudget before launching (an increase beyond the launch's total
  // would never be granted).
  static constexpr bool kRegSplit = kSmWG == 2;
  static constexpr uint32_t kRegsCtl = kGather ? 64 : 88, kRegsSoftmax = kGather ? 168 : 208, kRegsGather = 112;
  static constexpr int kRegBudget = 128 * kRegsCtl + 256 * kRegsSoftmax + (kGather ? 128 * kRegsGather : 0);
  // registers per thread at launch: a kernel that uses setmaxnreg is compiled
  // to the whole per-thread share of the register file (checked on the host);
  // each role then moves from this count to its own with .inc or .dec
  static constexpr uint32_t kLaunchRegs = (65536 / (kGatherWarp0 * 32 + (kGather ? 128 : 0))) & ~7u;
  static_assert(!kRegSplit || kRegBudget <= 65536, "register split exceeds the register file");
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kKvChunkBytes = kTileTokens * 128;  // 8 KB: [64 tokens][64 dims] bf16
  static constexpr int kPairBytes = 2 * kKvChunkBytes;    // chunks 2b, 2b+1: one 128-dv block of V
  static constexpr int kQChunkBytes = R * 128;
  static constexpr int kQBytes = kNumChunks * kQChunkBytes;
  static constexpr int kPBytes = R * kTileTokens * 2;     // P of one tile, bf16
  // KV staging ring: kNA pair slots + kNB RoPE-chunk slots; a tile occupies 4
  // pair slots and 1 RoPE slot.  The ring is sized to what shared memory holds
  // beside Q: with 64 rows exactly two tiles, P of a tile then living in its
  // RoPE slot once S^T has consumed the RoPE dims (kPAlias); with 16 or 32
  // rows 2.5-2.75 tiles plus a separate double-buffered P.
  static constexpr bool kPAlias = (R == 64);
  static constexpr int kNA = R == 64 ? 8 : (R == 32 ? 10 : 11);
  static constexpr int kNB = R == 64 ? 2 : (R == 32 ? 2 : 3);
  static constexpr int kPairOff = 0;
  static constexpr int kRopeOff = kNA * kPairBytes;
  static constexpr int kQOff = kRopeOff + kNB * kKvChunkBytes;
  static constexpr int kPOff = kQOff + kQBytes;                // separate P buffers (not kPAlias)
  static constexpr int kPBufBytes = kPAlias ? 0 : 2 * kPBytes;
  // With 64 rows P is stored MN-major ([64 tokens][64 rows], one 128-byte
  // swizzle atom per token): eight 16-byte stores per thread.
  static constexpr bool kPMnMajor = (R == 64);
  static constexpr int kAuxOff = (kPOff + kPBufBytes + 1023) / 1024 * 1024;
  // barriers: q_full, q_empty, chunk_full[2*kNA + kNB], pair_empty[kNA], rope_empty[kNB],
  // s_full[2], s_empty[2], p_full[2], o_full, o_empty, mma_done, o_done[2], raw_full[kNumRaw]
  // "tile full" barriers for the tiles in flight (at most three: the ring
  // holds under three tiles), used round robin: tile jt -> jt % 3, phase
  // jt / 3.  One per tile, or one per item of a tile (pairs 0..3, RoPE) where
  // the S MMAs start on each item as it is written: dense with 64 rows (the
  // tile loads are the chain there) and bf16 row gathers (the in-place
  // swizzle); both measured faster that way, the 16-row dense path and the
  // FP8 gathers slower.
  static constexpr bool kItemFull = (MODE == kModeSparseBf16) || (MODE == kModeDense && R == 64);
  static constexpr int kFullItems = kItemFull ? 5 : 1;
  static constexpr int kNumFull = 3 * kFullItems;
  // sparse: raw FP8 rows of a tile land by row gathers in the upper chunk of
  // each pair slot (codes) and in the RoPE slot; raw_full[5 * (jt & 1) + b]
  // (b = 0..3 pairs, 4 = RoPE) completes when tile jt's have arrived
  static constexpr int kNumRaw = kGather ? 10 : 0;  // two sets (tile parity) of five
  static constexpr int kNumBars = 2 + kNumFull + kNA + kNB + 4 + 2 + 5 + kNumRaw;
  // rounded to 128 bytes so the row statistics after the barriers are 16-byte
  // aligned (they are read with 16-byte vector loads)
  static constexpr int kBarBytes = (kNumBars * 8 + 127) / 128 * 128;
  // aux: floats m[R], alpha[R], inv_l[R], lse[R], red[4][R]; 16 ints (abort flag,
  // TMEM base); 512 bytes of per-tile token validity flags (a ring of four
  // tiles: a tile's flags are written once the slots of a tile at least two
  // back are free, when the softmax of the tile three back is surely done);
  // ints lim[R] (last visible key per row)
  static constexpr int kAuxBytes = kBarBytes + 8 * R * 4 + 64 + 512 + 4 * R;
  static constexpr int kSmemBytes = kAuxOff + kAuxBytes + 1024;  // + alignment slack
  static constexpr int kOCol = 0;
  static constexpr int kSCol = 4 * R;
  static constexpr int kTmemCols = (6 * R <= 128) ? 128 : ((6 * R <= 256) ? 256 : 512);

  // arrivals on a full barrier: dense 1 (the producer, + the TMA bytes);
  // gathered 4 per tile (each gather warp once it has written its part) or 2
  // per item (the two warps writing it)
  static constexpr int kFullArrivals = kGather ? (kItemFull ? 2 : 4) : 1;
  static_assert(kPBytes <= kKvChunkBytes || !kPAlias, "P must fit in the RoPE chunk");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(R == 16 || R == 32 || R == 64, "rows per CTA");
  static_assert((kAuxOff + kBarBytes) % 16 == 0, "row statistics must be 16-byte aligned");
  static_assert(kTileTokens == kPageSize, "one KV tile is one page");
};

struct Bars {
  uint64_t* q_full;
  uint64_t* q_empty;
  uint64_t* full;        // [3 * kFullItems]: tile jt's chunks (or one item of them) are in shared memory
  uint64_t* pair_empty;  // [kNA]
  uint64_t* rope_empty;  // [kNB]
  uint64_t* s_full;    // [2]
  uint64_t* s_empty;   // [2]
  uint64_t* p_full;    // [2]: tile jt's P is ready (barrier jt & 1)
  uint64_t* o_full;
  uint64_t* o_empty;
  uint64_t* mma_done;
  uint64_t* o_done;    // [2]: tile jt's PV MMAs are done (barrier jt & 1)
  uint64_t* raw_full;  // sparse: [10]
};

// Segment iterator shared by all roles: the part walks problems p0..p1 and,
// inside each, a tile range.  All roles derive the identical sequence.
struct Segments {
  int p0, t0, p1, t1, np, s_q, topk;
  const int32_t* seqlens;
  __device__ int last() const { return p1 < np ? p1 : np - 1; }
  __device__ void range(int p, int& tb, int& te) const {
    int n = problem_tiles(seqlens, p, s_q, topk);
    tb = (p == p0) ? t0 : 0;
    te = (p == p1) ? t1 : n;
    if (te > n) te = n;
  }
};

// Ring bookkeeping.  Tile number jt (counted over all of a CTA's segments)
// uses pair items 4*jt + b (b = 0..3) and RoPE item jt; item n of a ring of
// size k lives in slot n % k and is that slot's (n / k)-th use (the parity of
// its barriers' phases).
template <class C>
struct Ring {
  __device__ static int pair_slot(int jt, int b) { return (4 * jt + b) % C::kNA; }
  __device__ static uint32_t pair_use(int jt, int b) { return static_cast<uint32_t>((4 * jt + b) / C::kNA); }
  __device__ static int rope_slot(int jt) { return jt % C::kNB; }
  __device__ static uint32_t rope_use(int jt) { return static_cast<uint32_t>(jt / C::kNB); }
  // byte offset of chunk c (0..8) of tile jt in the KV region
  __device__ static uint32_t chunk_off(int jt, int c) {
    return c < 8 ? C::kPairOff + pair_slot(jt, c >> 1) * C::kPairBytes + (c & 1) * C::kKvChunkBytes
                 : C::kRopeOff + rope_slot(jt) * C::kKvChunkBytes;
  }
  __device__ static int full_index(int jt) { return jt % 3; }
  __device__ static uint32_t full_parity(int jt) { return static_cast<uint32_t>(jt / 3) & 1u; }
  // byte offset of the P buffer of tile jt
  __device__ static uint32_t p_off(int jt) {
    return C::kPAlias ? C::kRopeOff + rope_slot(jt) * C::kKvChunkBytes : C::kPOff + (jt & 1) * C::kPBytes;
  }
};

// Bounded wait that ignores the abort flag (used to drain own async work).
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > limit_ns) return false;
  return true;
}

// Warp-uniform bounded wait: if any lane fails, every lane sees failure.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const Watchdog& wd) {
  bool ok = mbar_wait(bar, parity, wd);
  return __all_sync(0xffffffffu, ok);
}

// ---------------------------------------------------------------------------
// producer: Q (always) and dense KV pages by TMA
// ---------------------------------------------------------------------------
template <int R, int MODE>
__device__ void producer(const CUtensorMap* tm_q, const CUtensorMap* tm_kv, const DecodeParams& p,
                         const Segments& sg, int g, uint8_t* kv, uint8_t* qs, const Bars& bars,
                         volatile uint8_t* flags, const Watchdog& wd) {
  // The whole producer warp runs this code converged; each copy is issued by
  // one elected lane (as for the MMAs, a lane issuing alone while its warp
  // waits elsewhere issues far more slowly).
  using C = Cfg<R, MODE>;

  const uint64_t pol_kv = p.evict_first ? l2_policy_evict_first() : l2_policy_evict_normal();
  const uint64_t pol_q = l2_policy_evict_normal();
  const int lane = threadIdx.x & 31;
  using RG = Ring<C>;
  // full barriers armed so far (bit per barrier) and the parity of each one's
  // next phase, for the drain
  uint32_t armed = 0, next_par = 0;
  int fidx = 0;  // this tile's full barrier (jt % 3)
  int q_armed = 0, jt = 0;
  for (int prob = sg.p0; prob <= sg.last(); ++prob) {
    int tb, te;
    sg.range(prob, tb, te);
    if (tb >= te) continue;
    if (q_armed > 0 && !warp_wait(bars.q_empty, (q_armed - 1) & 1, wd)) goto drain;
    {
      const int row0 = prob * p.rows + g * R;
      if (lane == 0) mbar_arrive_expect_tx(bars.q_full, kNumChunks * C::kQChunkBytes);
      __syncwarp();
      if (lane < kNumChunks) tma_load_3d(qs + lane * C::kQChunkBytes, tm_q, bars.q_full, 0, lane, row0, pol_q);
      __syncwarp();
      ++q_armed;
    }
    if (!C::kGather) {
      const int b = prob;
      const int32_t* bt = p.block_table + static_cast<int64_t>(b) * p.block_table_stride;
      for (int j = tb; j < te; ++j, ++jt) {
        // tile j is page j of the element
        const int pg = j < p.block_table_stride ? bt[j] : -1;
        const bool ok = pg >= 0 && pg < p.num_pages;
        if (!ok && lane == 0) atomicOr(p.status, MLA_DEVICE_BAD_PAGE);
        uint64_t* fb = bars.full + C::kFullItems * fidx;
        bool tile_armed = false;
        // RoPE chunk first when its slot frees at S^T (separate P); pairs first
        // when P lives in the RoPE slot until the PV MMAs are done
#pragma unroll 1
        for (int step = 0; step < 5; ++step) {
          const int item = C::kPAlias ? step : (step == 0 ? 4 : step - 1);  // 0..3 pairs, 4 RoPE
          int c0, nc;
          if (item < 4) {
            const uint32_t use = RG::pair_use(jt, item);
            if (use > 0 && !warp_wait(bars.pair_empty + RG::pair_slot(jt, item), (use - 1) & 1, wd)) goto drain;
            if (item == 0 && lane == 0) {
              // page flag of this tile for the softmax (its readers of two
              // tiles ago are done: their PV released this pair slot)
              flags[(jt & 3) * 128] = ok ? 1 : 0;
            }
            c0 = 2 * item;
            nc = 2;
          } else {
            const uint32_t use = RG::rope_use(jt);
            if (use > 0 && !warp_wait(bars.rope_empty + RG::rope_slot(jt), (use - 1) & 1, wd)) goto drain;
            c0 = 8;
            nc = 1;
          }
          // the tile's full barrier is armed with all its bytes before its first
          // copy (per item: the item's barrier with the item's bytes), after
          // that copy's slot wait (which implies the barrier's previous phase,
          // three tiles back, has completed); the item's chunks are issued by
          // one lane each
          uint64_t* ib = fb;
          if (C::kItemFull) {
            const int bi = C::kFullItems * fidx + item;
            ib = bars.full + bi;
            if (lane == 0) mbar_arrive_expect_tx(ib, ok ? static_cast<uint32_t>(nc * C::kKvChunkBytes) : 0u);
            __syncwarp();
            armed |= 1u << bi;
            next_par ^= 1u << bi;
          } else if (!tile_armed) {
            if (lane == 0) mbar_arrive_expect_tx(fb, ok ? static_cast<uint32_t>(kNumChunks * C::kKvChunkBytes) : 0u);
            __syncwarp();
            tile_armed = true;
            armed |= 1u << fidx;
            next_par ^= 1u << fidx;
          }
          if (ok && lane < nc)
            tma_load_3d(kv + RG::chunk_off(jt, c0 + lane), tm_kv, ib, 0, c0 + lane, pg * kPageSize, pol_kv);
          __syncwarp();
          if (lane == 0) {
            if (c0 == 0) MLA_TR(kTrProdChunk0, jt);
            if (c0 == 8) MLA_TR(kTrProdChunk8, jt);
          }
        }
        if (++fidx == 3) fidx = 0;
      }
    }
  }
drain:
  // wait (bounded) for this warp's own copies still in flight: the latest
  // armed phase of every full barrier (earlier phases of a barrier completed
  // before it was re-armed)
  if (lane == 0) {
    if (!C::kGather) {
#pragma unroll 1
      for (int k = 0; k < C::kNumFull; ++k)
        if ((armed >> k) & 1u) mbar_wait_drain(bars.full + k, ((next_par >> k) & 1u) ^ 1u, wd.limit_ns);
    }
    if (q_armed > 0) mbar_wait_drain(bars.q_full, (q_armed - 1) & 1, wd.limit_ns);
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// MMA issuers: warp 1 issues S^T, warp 3 issues PV
// ---------------------------------------------------------------------------
// Two warps feed the tensor pipe: one issues S^T(jt) as soon as tile jt is in
// shared memory, the other issues PV(jt) as soon as P(jt) is ready, so
// neither waits for the other's operands and the pipe receives both streams.
// Their MMAs write disjoint TMEM columns (S^T buffers, O^T).  Each warp runs
// converged and issues every MMA and commit from one elected lane (a lane
// issuing alone while its warp waits elsewhere feeds the pipe at well under
// half the rate).  Shared-memory addresses are 32-bit values in registers,
// ring positions advance by counters, descriptors are built once per pair
// slot and advanced by additions, and barrier tests are warp-uniform.

// Ring position of one tile: slot and use count of its first pair item and
// of its RoPE item.
template <class C>
struct RingPos {
  int pbase, puse, rslot, ruse;
  __device__ void advance() {
    pbase += 4;
    if (pbase >= C::kNA) {
      pbase -= C::kNA;
      ++puse;
    }
    if (++rslot == C::kNB) {
      rslot = 0;
      ++ruse;
    }
  }
  __device__ int pair_slot(int b) const { return pbase + b >= C::kNA ? pbase + b - C::kNA : pbase + b; }
};

// Warp-uniform barrier test (lane 0's result).
__device__ __forceinline__ bool warp_test_u32(uint32_t bar, uint32_t parity) {
  return __shfl_sync(0xffffffffu, mbar_test_wait_u32(bar, parity) ? 1 : 0, 0) != 0;
}

// Warp-uniform bounded wait.
__device__ __forceinline__ bool mbar_wait_u32(uint32_t bar, uint32_t parity, const Watchdog& wd) {
  uint64_t t0 = 0;
  while (!warp_test_u32(bar, parity)) {
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

// Commit from this warp's elected lane: arrive on `bar` when the MMAs this
// warp issued so far are done; then the drain of the CTA's end.
__device__ __forceinline__ void warp_commit(uint32_t bar) {
  if (elect_one()) umma_commit_u32(bar);
  __syncwarp();
}

template <int R, int MODE>
__device__ void s_issuer(const Segments& sg, uint32_t tmem, uint8_t* kv, uint8_t* qs, const Bars& bars,
                         const Watchdog& wd) {
  using C = Cfg<R, MODE>;
  constexpr uint32_t kIdS = idesc_bf16_f32(kTileTokens, R, 0, 0);  // A = K tile (K-major), B = Q (K-major)
  constexpr uint64_t kHiK = smem_desc_hi(16, 1024);
  const int lane = threadIdx.x & 31;
  const uint32_t kvb = smem_u32(kv), qb = smem_u32(qs);
  const uint32_t full = smem_u32(bars.full), s_full = smem_u32(bars.s_full), s_empty = smem_u32(bars.s_empty);
  const uint32_t rope_empty = smem_u32(bars.rope_empty);
  const uint32_t q_full = smem_u32(bars.q_full), q_empty = smem_u32(bars.q_empty);
  RingPos<C> cur{0, 0, 0, 0};
  int jt = 0, seg = 0;
  int fidx = 0, fphase = 0;  // full barrier of the next tile (jt % 3) and its phase (jt / 3)
  for (int prob = sg.p0; prob <= sg.last(); ++prob) {
    int tb, te;
    sg.range(prob, tb, te);
    if (tb >= te) continue;
    if (!mbar_wait_u32(q_full, seg & 1, wd)) goto done;
    tc_fence_after();
    for (int j = tb; j < te; ++j, ++jt) {
      const int sb = jt & 1;
      // the softmax has read S^T of tile jt-2 from this buffer
      if (jt >= 2 && !mbar_wait_u32(s_empty + 8 * sb, ((jt >> 1) - 1) & 1, wd)) goto done;
      tc_fence_after();
      const uint32_t fpar = static_cast<uint32_t>(fphase) & 1u;
      const uint32_t fbar = full + 8 * C::kFullItems * fidx;
      if (!C::kItemFull && !mbar_wait_u32(fbar, fpar, wd)) goto done;
      if (++fidx == 3) {
        fidx = 0;
        ++fphase;
      }
      const uint32_t d_s = tmem + C::kSCol + sb * R;
      // S^T = K Q^T over the nine chunks, 36 MMAs (pairs of chunks sit
      // together in a pair slot): back to back once the tile is in, or item
      // by item as each is written, in the order they are written (row
      // gathers: blocks 0 and 2, then 1 and 3, then RoPE)
#pragma unroll 1
      for (int q = 0; q < 5; ++q) {
        const int pb = (C::kGather && C::kItemFull) ? (q < 4 ? ((q & 1) << 1) | (q >> 1) : 4) : q;
        if (C::kItemFull && !mbar_wait_u32(fbar + 8 * pb, fpar, wd)) goto done;
        if (q == 0 && lane == 0) MLA_TR(kTrMmaKv0, jt);
        const uint32_t pa = pb < 4 ? kvb + C::kPairOff + cur.pair_slot(pb) * C::kPairBytes
                                   : kvb + C::kRopeOff + cur.rslot * C::kKvChunkBytes;
        const uint64_t a0 = kHiK | (pa >> 4);
        const uint64_t b0 = kHiK | ((qb + 2 * pb * C::kQChunkBytes) >> 4);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (pb == 4 && i >= 4) break;
          const int h = i >> 2, kk = i & 3;  // chunk 2pb+h, k step kk
          if (elect_one())
            umma_bf16_ss_fast(d_s, a0 + h * (C::kKvChunkBytes >> 4) + 2 * kk,
                              b0 + h * (C::kQChunkBytes >> 4) + 2 * kk, kIdS, (q | i) != 0);
          __syncwarp();
        }
      }
      if (elect_one()) {
        umma_commit_u32(s_full + 8 * sb);
        // with a separate P buffer the RoPE chunk is free once S^T is done
        if (!C::kPAlias) umma_commit_u32(rope_empty + 8 * cur.rslot);
        if (j == te - 1) umma_commit_u32(q_empty);
      }
      __syncwarp();
      if (lane == 0) MLA_TR(kTrMmaSDone, jt);
      cur.advance();
    }
    ++seg;
  }
done:
  warp_commit(smem_u32(bars.mma_done));
  if (lane == 0) mbar_wait_drain(bars.mma_done, 0, wd.limit_ns);
  __syncwarp();
}

template <int R, int MODE>
__device__ void pv_issuer(const Segments& sg, uint32_t tmem, uint8_t* kv, const Bars& bars, const Watchdog& wd) {
  using C = Cfg<R, MODE>;
  constexpr uint32_t kIdO = idesc_bf16_f32(128, R, 1, C::kPMnMajor ? 1 : 0);  // A = V^T (MN-major), B = P
  constexpr uint64_t kHiV = smem_desc_hi(C::kKvChunkBytes, 1024);
  constexpr uint64_t kHiP = smem_desc_hi(16, 1024);
  constexpr uint32_t kPStep = C::kPMnMajor ? (2048 >> 4) : (32 >> 4);  // 16 tokens of P
  const int lane = threadIdx.x & 31;
  const uint32_t kvb = smem_u32(kv);
  const uint32_t p_full = smem_u32(bars.p_full), o_empty = smem_u32(bars.o_empty), o_done = smem_u32(bars.o_done);
  const uint32_t o_full = smem_u32(bars.o_full), pair_empty = smem_u32(bars.pair_empty);
  const uint32_t rope_empty = smem_u32(bars.rope_empty);
  RingPos<C> cur{0, 0, 0, 0};
  int jt = 0, seg = 0;
  for (int prob = sg.p0; prob <= sg.last(); ++prob) {
    int tb, te;
    sg.range(prob, tb, te);
    if (tb >= te) continue;
    for (int j = tb; j < te; ++j, ++jt) {
      const bool first = (j == tb), last = (j == te - 1);
      if (!mbar_wait_u32(p_full + 8 * (jt & 1), (jt >> 1) & 1, wd)) goto done;
      tc_fence_after();
      if (lane == 0) MLA_TR(kTrMmaPFull, jt);
      if (first && seg > 0) {
        // the epilogue of the previous segment has read O^T
        if (!mbar_wait_u32(o_empty, (seg - 1) & 1, wd)) goto done;
        tc_fence_after();
      }
      const uint32_t p_addr = C::kPAlias ? kvb + C::kRopeOff + cur.rslot * C::kKvChunkBytes
                                         : kvb + C::kPOff + (jt & 1) * C::kPBytes;
      const uint64_t b0 = kHiP | (p_addr >> 4);
#pragma unroll
      for (int blk = 0; blk < 4; ++blk) {
        const int s = cur.pair_slot(blk);
        const uint64_t a0 = kHiV | ((kvb + C::kPairOff + s * C::kPairBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kTileTokens / 16; ++kk) {
          if (elect_one())
            umma_bf16_ss_fast(tmem + C::kOCol + blk * R, a0 + kk * (2048 >> 4), b0 + kk * kPStep, kIdO,
                              !(first && kk == 0));
          __syncwarp();
        }
        warp_commit(pair_empty + 8 * s);
        if (blk == 0 && lane == 0) MLA_TR(kTrMmaO1, jt);
      }
      if (elect_one()) {
        if (C::kPAlias) umma_commit_u32(rope_empty + 8 * cur.rslot);  // P lived in the RoPE slot
        umma_commit_u32(o_done + 8 * (jt & 1));
        if (last) umma_commit_u32(o_full);
      }
      __syncwarp();
      if (lane == 0) MLA_TR(kTrMmaODone, jt);
      cur.advance();
    }
    ++seg;
  }
done:
  warp_commit(smem_u32(bars.mma_done));
  if (lane == 0) mbar_wait_drain(bars.mma_done, 0, wd.limit_ns);
  __syncwarp();
}

// ---------------------------------------------------------------------------
// row gathers (128 threads, two per token): FP8 rows are dequantised, bf16
// rows only put into the swizzled operand layout
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t dequant2(uint32_t codes16, float scale) {
  return e4m3x2_scaled_bf16x2(codes16, scale);
}

// Permute one 128-byte row of a chunk, copied in plain order, into the
// 128-byte swizzle (unit u of row t goes to unit u ^ (t & 7)) in place; an
// invalid token's row becomes zeros.
__device__ __forceinline__ void swizzle_row_in_place(uint32_t row_addr, uint32_t tsw, bool ok) {
  uint4 raw[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) raw[k] = ld_shared_v4(row_addr + ((k ^ tsw) << 4));
  // raw[k] holds unit k ^ tsw, whose swizzled position is (k ^ tsw) ^ tsw = k
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint4 v = ok ? raw[k] : make_uint4(0, 0, 0, 0);
    st_shared_v4(row_addr + (k << 4), v.x, v.y, v.z, v.w);
  }
}

constexpr int kBf16RowBytes = kDqk * 2;  // a bf16 cache row: 576 dims

// 16-byte asynchronous copy global -> shared (src_bytes 0 writes zeros), and
// one arrival on `bar` once every copy this thread started has completed
// (the barrier's expected count includes it).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

template <int R, int MODE>
__device__ void gather_rows(const CUtensorMap* tm_rows, const DecodeParams& p, const Segments& sg, uint8_t* kv,
                            const Bars& bars, volatile uint8_t* flags, const Watchdog& wd) {
  using C = Cfg<R, MODE>;
  using RG = Ring<C>;
  // gathered bf16 rows (sparse over the bf16 cache, sparse prefill) are copied
  // by the threads, 16 bytes at a time, into their swizzled places
  constexpr bool kRowCopies = C::kIndexed && !C::kFp8;
  // 128 threads, two per token: half h = 0 (warps 0, 1) converts value blocks
  // 0 and 1 and the RoPE dims, half 1 (warps 2, 3) value blocks 2 and 3.
  // FP8 rows: a block's 128 codes land in the upper chunk of its pair slot
  // and are dequantised into both chunks.  bf16 rows: both chunks of a block
  // are copied as plain 128-byte rows and permuted into the swizzle in place.
  // Software-pipelined: the rows of tile jt+1 are looked up (dependent index
  // and block-table loads) before tile jt is dequantised, and tile jt+1's row
  // gathers are issued right after, so lookups overlap conversion and gather
  // latency overlaps the next lookup.  The raw barriers come in two sets
  // (tile parity) so two tiles' copies never share a phase.
  const int tid = threadIdx.x - 32 * C::kGatherWarp0;
  const int lane = tid & 31;
  const int h = tid >> 6;
  const int tok = tid & 63;           // token of the tile
  const int wtok = tok & ~31;         // first token of this warp
  const uint32_t tsw = tok & 7;
  const uint32_t kv_base = smem_u32(kv);
  const uint64_t pol = l2_policy_evict_normal();
  uint32_t armed = 0, next_par = 0;  // raw barriers armed by this warp (bit per barrier), next phase parity

  // tile iterator over the CTA's segments
  struct It {
    int prob, j, te;
    bool valid;
  };
  auto first_from = [&](int prob) -> It {
    for (; prob <= sg.last(); ++prob) {
      int tb, te;
      sg.range(prob, tb, te);
      if (tb < te) return It{prob, tb, te, true};
    }
    return It{0, 0, 0, false};
  };
  auto next_of = [&](const It& it) -> It {
    if (it.j + 1 < it.te) return It{it.prob, it.j + 1, it.te, true};
    return first_from(it.prob + 1);
  };
  // look up this thread's token of tile `it`: cache row (invalid -> row 0,
  // zeros written later), validity, this half's two scales
  auto lookup = [&](const It& it, int& row, bool& ok, uint2& sc) {
    if (C::kIndexed) {
      const int b = it.prob / p.s_q;
      const int L = p.flat_rows > 0 ? p.flat_rows : sg.seqlens[b];
      const int k = it.j * kTileTokens + tok;
      int tk = p.topk;  // index slots of this problem
      if (p.topk_lengths) {
        const int len = p.topk_lengths[it.prob];
        tk = len < 0 ? 0 : (len < p.topk ? len : p.topk);
      }
      const int t = k < tk ? p.indices[static_cast<int64_t>(it.prob) * p.topk + k] : -1;
      ok = t >= 0 && t < L;
      if (p.flat_rows > 0) {
        row = ok ? t : 0;  // unpaged KV: the index is the row
      } else {
        const int32_t* bt = p.block_table + static_cast<int64_t>(b) * p.block_table_stride;
        const int page = (ok && (t >> 6) < p.block_table_stride) ? bt[t >> 6] : -1;
        if (ok && (page < 0 || page >= p.num_pages)) {
          ok = false;
          if (h == 0) atomicOr(p.status, MLA_DEVICE_BAD_PAGE);
        }
        row = ok ? page * kPageSize + (t & 63) : 0;
      }
    } else {
      // dense: tile j is page j of the element; row = page * 64 + token, with
      // page 0 standing in for an unusable page (its tokens are written as zeros)
      const int b = it.prob;
      const int L = sg.seqlens[b];
      const int page = it.j < p.block_table_stride ? p.block_table[static_cast<int64_t>(b) * p.block_table_stride + it.j] : -1;
      const bool page_ok = page >= 0 && page < p.num_pages;
      if (!page_ok && tok == 0 && h == 0) atomicOr(p.status, MLA_DEVICE_BAD_PAGE);
      ok = page_ok && it.j * kTileTokens + tok < L;
      row = (page_ok ? page : 0) * kPageSize + tok;
    }
    if (C::kFp8 && p.kv_scales) {
      // one scale per token for all four blocks
      const uint32_t s1 = ok ? __float_as_uint(__ldg(p.kv_scales + row)) : 0u;
      sc = make_uint2(s1, s1);
    } else if (C::kFp8) {
      sc = ok ? __ldg(reinterpret_cast<const uint2*>(p.kv_fp8 + static_cast<int64_t>(row) * kFp8RowBytes +
                                                     kFp8ScaleOffset + 8 * h))
              : make_uint2(0, 0);
    } else {
      sc = make_uint2(0, 0);
    }
  };
  // issue the row gathers of tile jt (FP8: codes of this half's blocks into
  // the upper chunks of their pair slots; bf16: both chunks of each block;
  // half 0 also the RoPE bytes).  A 4-row gather covers tokens g4 .. g4 + 3.
  auto issue = [&](int jt, int row, bool ok) -> bool {
    if (kRowCopies) {
      // bf16 rows, copied in 16-byte units straight into the 128-byte swizzle
      // (unit u of a row goes to u ^ (token & 7)): per instruction the warp
      // copies one 128-byte chunk of four of its 32 tokens' rows, eight lanes
      // per row, so every row segment is one coalesced 128-byte request.  Half
      // h copies its two blocks and, half 0, the RoPE chunk; an unusable token
      // is zero-filled by the copies (source bytes 0)
      const int set = 5 * (jt & 1);
      const int u = lane & 7;
      int rs[8];
      uint32_t nbs[8];
#pragma unroll
      for (int st = 0; st < 8; ++st) {
        const int tl = 4 * st + (lane >> 3);
        const int r = __shfl_sync(0xffffffffu, row, tl);
        const bool o = __shfl_sync(0xffffffffu, ok ? 1 : 0, tl) != 0;
        rs[st] = o ? r : 0;
        nbs[st] = o ? 16u : 0u;
      }
      auto copy_chunk = [&](int c) {
        const uint32_t cbase = kv_base + RG::chunk_off(jt, c);
#pragma unroll
        for (int st = 0; st < 8; ++st) {
          const int tk = wtok + 4 * st + (lane >> 3);
          cp_async16(cbase + tk * 128 + ((u ^ (tk & 7)) << 4),
                     p.kv_fp8 + static_cast<int64_t>(rs[st]) * kBf16RowBytes + 128 * c + 16 * u, nbs[st]);
        }
      };
#pragma unroll 1
      for (int i = 0; i < 2; ++i) {
        const int blk = 2 * h + i;
        const uint32_t use = RG::pair_use(jt, blk);
        if (use > 0 && !warp_wait(bars.pair_empty + RG::pair_slot(jt, blk), (use - 1) & 1, wd)) return false;
        if (blk == 0) flags[(jt & 3) * 128 + tok] = ok ? 1 : 0;  // token validity for the softmax
        copy_chunk(2 * blk);
        copy_chunk(2 * blk + 1);
        cp_async_arrive(bars.raw_full + set + blk);
        armed |= 1u << (set + blk);
        next_par ^= 1u << (set + blk);
      }
      if (h == 0) {
        const uint32_t use = RG::rope_use(jt);
        if (use > 0 && !warp_wait(bars.rope_empty + RG::rope_slot(jt), (use - 1) & 1, wd)) return false;
        copy_chunk(8);
        cp_async_arrive(bars.raw_full + set + 4);
        armed |= 1u << (set + 4);
        next_par ^= 1u << (set + 4);
      }
      return true;
    }
    const int gl = lane & 7;
    const int g4 = wtok + 4 * gl;
    const int r0 = __shfl_sync(0xffffffffu, row, 4 * gl);
    const int r1 = __shfl_sync(0xffffffffu, row, 4 * gl + 1);
    const int r2 = __shfl_sync(0xffffffffu, row, 4 * gl + 2);
    const int r3 = __shfl_sync(0xffffffffu, row, 4 * gl + 3);
    const int set = 5 * (jt & 1);
#pragma unroll 1
    for (int i = 0; i < 2; ++i) {
      const int blk = 2 * h + i;
      const uint32_t use = RG::pair_use(jt, blk);
      if (use > 0 && !warp_wait(bars.pair_empty + RG::pair_slot(jt, blk), (use - 1) & 1, wd)) return false;
      if (blk == 0) flags[(jt & 3) * 128 + tok] = ok ? 1 : 0;  // token validity for the softmax
      if (lane == 0) mbar_arrive_expect_tx(bars.raw_full + set + blk, (C::kFp8 ? 1 : 2) * 32 * 128);
      armed |= 1u << (set + blk);
      next_par ^= 1u << (set + blk);
      __syncwarp();
      if (!C::kFp8) {
        // bf16 rows: lanes 0..7 chunk 2 blk, lanes 8..15 chunk 2 blk + 1
        if (lane < 16) {
          const int c = 2 * blk + (lane >> 3);
          uint8_t* dst = kv + RG::chunk_off(jt, c) + g4 * 128;
          tma_gather4(dst, tm_rows, bars.raw_full + set + blk, 128 * c, r0, r1, r2, r3, pol);
        }
      } else if (C::kIndexed) {
        if (lane < 8) {
          uint8_t* dst = kv + RG::chunk_off(jt, 2 * blk + 1) + g4 * 128;
          tma_gather4(dst, tm_rows, bars.raw_full + set + blk, 128 * blk, r0, r1, r2, r3, pol);
        }
      } else if (lane == 0) {
        // dense: this warp's 32 consecutive rows of the page in one box
        tma_load_2d(kv + RG::chunk_off(jt, 2 * blk + 1) + wtok * 128, tm_rows, bars.raw_full + set + blk,
                    128 * blk, row, pol);
      }
    }
    if (h == 0) {
      const uint32_t use = RG::rope_use(jt);
      if (use > 0 && !warp_wait(bars.rope_empty + RG::rope_slot(jt), (use - 1) & 1, wd)) return false;
      if (lane == 0) mbar_arrive_expect_tx(bars.raw_full + set + 4, 32 * 128);
      armed |= 1u << (set + 4);
      next_par ^= 1u << (set + 4);
      __syncwarp();
      if (C::kIndexed) {
        if (lane < 8) {
          uint8_t* dst = kv + RG::chunk_off(jt, 8) + g4 * 128;
          tma_gather4(dst, tm_rows, bars.raw_full + set + 4, C::kFp8 ? p.fp8_rope_off : 2 * kDv, r0, r1, r2, r3,
                      pol);
        }
      } else if (lane == 0) {
        tma_load_2d(kv + RG::chunk_off(jt, 8) + wtok * 128, tm_rows, bars.raw_full + set + 4, p.fp8_rope_off, row,
                    pol);
      }
    }
    return true;
  };

  It cur = first_from(sg.p0);
  int row_c = 0;
  bool ok_c = false;
  uint2 sc_c = make_uint2(0, 0);
  int jt = 0;
  if (cur.valid) {
    lookup(cur, row_c, ok_c, sc_c);
    if (!issue(0, row_c, ok_c)) goto drain;
  }
  for (; cur.valid; ++jt) {
    if (tid == 0) MLA_TR(kTrGatherStart, jt);
    // tile jt+1: look up its rows first (the loads overlap the conversion)
    const It nxt = next_of(cur);
    int row_n = 0;
    bool ok_n = false;
    uint2 sc_n = make_uint2(0, 0);
    if (nxt.valid) lookup(nxt, row_n, ok_n, sc_n);
    // dequantise tile jt in place: token tok's 128 code bytes of block b sit
    // at row tok of chunk 2b+1; they become row tok of chunks 2b and 2b+1
    // (bf16, 128-byte swizzle).  Units are read in a per-thread rotated order.
    // bf16 rows: each permuted block gets this warp's arrival on the block's
    // full barrier (after the proxy fence that orders it for the MMAs).
    {
      const int set = 5 * (jt & 1);
      const uint32_t par = static_cast<uint32_t>(jt >> 1) & 1u;  // phase of set (jt & 1) for tile jt
      uint64_t* fb = bars.full + C::kFullItems * RG::full_index(jt);
#pragma unroll 1
      for (int i = 0; i < 2; ++i) {
        const int blk = 2 * h + i;
        if (!warp_wait(bars.raw_full + set + blk, par, wd)) goto drain;
        if (!C::kFp8) {
          if (!kRowCopies) {
            swizzle_row_in_place(kv_base + RG::chunk_off(jt, 2 * blk) + tok * 128, tsw, ok_c);
            swizzle_row_in_place(kv_base + RG::chunk_off(jt, 2 * blk + 1) + tok * 128, tsw, ok_c);
          }
          if (C::kItemFull) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(fb + blk);
          }
          continue;
        }
        const float scale = __uint_as_float(i == 0 ? sc_c.x : sc_c.y);
        const uint32_t lo = kv_base + RG::chunk_off(jt, 2 * blk) + tok * 128;
        const uint32_t hi = kv_base + RG::chunk_off(jt, 2 * blk + 1) + tok * 128;
        uint4 raw[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) raw[k] = ld_shared_v4(hi + ((k ^ tsw) << 4));
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t u = k ^ tsw;  // raw unit: codes 16u..16u+15 of the block
          const uint32_t dst = ((u & 4) ? hi : lo);
          const uint32_t k0 = (2 * (u & 3)) ^ tsw, k1 = (2 * (u & 3) + 1) ^ tsw;
          uint4 v = raw[k];
          if (!ok_c) v = make_uint4(0, 0, 0, 0);
          st_shared_v4(dst + (k0 << 4), dequant2(v.x & 0xffffu, scale), dequant2(v.x >> 16, scale),
                       dequant2(v.y & 0xffffu, scale), dequant2(v.y >> 16, scale));
          st_shared_v4(dst + (k1 << 4), dequant2(v.z & 0xffffu, scale), dequant2(v.z >> 16, scale),
                       dequant2(v.w & 0xffffu, scale), dequant2(v.w >> 16, scale));
        }
      }
      if (h == 0) {
        // RoPE: already bf16; permute the 16-byte units into the swizzled order
        if (!warp_wait(bars.raw_full + set + 4, par, wd)) goto drain;
        if (!kRowCopies) swizzle_row_in_place(kv_base + RG::chunk_off(jt, 8) + tok * 128, tsw, ok_c);
        if (C::kItemFull) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(fb + 4);
        }
      }
      if (!C::kItemFull) {
        // this warp's part of the tile is written: one arrival on the tile's
        // full barrier (after the proxy fence that orders it for the MMAs)
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(fb);
      }
    }
    if (tid == 0) MLA_TR(kTrGatherDone, jt);
    // then tile jt+1's row gathers (their slots free once the PV of tile jt-1 is done)
    if (nxt.valid && !issue(jt + 1, row_n, ok_n)) goto drain;
    cur = nxt;
    row_c = row_n;
    ok_c = ok_n;
    sc_c = sc_n;
  }
  return;
drain:
  // abort: wait (bounded) for this warp's row gathers still in flight (the
  // latest armed phase of each raw barrier); row copies: this thread's own
  if (kRowCopies) asm volatile("cp.async.wait_all;" ::: "memory");
  if (lane == 0) {
#pragma unroll 1
    for (int k = 0; k < C::kNumRaw; ++k)
      if ((armed >> k) & 1u) mbar_wait_drain(bars.raw_full + k, ((next_par >> k) & 1u) ^ 1u, wd.limit_ns);
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// softmax + epilogue (128 threads; thread t -> token t of the tile, TMEM lane t)
// ---------------------------------------------------------------------------
// Reduce-scatter of N per-lane values over the 32 lanes of a warp (N a power
// of two, 16..64): at each step a lane keeps one half of its values, sends the
// other half to its partner and combines.  Afterwards lane l holds the
// reduction of values [k*l, k*l + k) in out[0..k) with k = max(N/32, 1) (for
// N < 32 lanes l and l ^ (32/N)... share a value).  Writes the results to
// dst[k*l + i] for the lanes that own distinct values.
template <int N, bool MAX>
__device__ __forceinline__ void warp_reduce_scatter(const float (&v)[N], float* dst, int lane) {
  constexpr int K = N >= 32 ? N / 32 : 1;
  float t[N / 2];
  // first step reads v directly (no copy of the N inputs)
  {
    const bool up = (lane & 16) != 0;
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      const float send = up ? v[i] : v[i + N / 2];
      const float keep = up ? v[i + N / 2] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
      t[i] = MAX ? fmaxf(keep, recv) : keep + recv;
    }
  }
  int n = N / 2;
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) {
    if (n > K) {
      const bool up = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < N / 4; ++i) {
        if (i < n / 2) {
          const float send = up ? t[i] : t[i + n / 2];
          const float keep = up ? t[i + n / 2] : t[i];
          const float recv = __shfl_xor_sync(0xffffffffu, send, o);
          t[i] = MAX ? fmaxf(keep, recv) : keep + recv;
        }
      }
      n >>= 1;
    } else {
      // fewer values than lanes left: plain butterfly on the remaining value
      const float recv = __shfl_xor_sync(0xffffffffu, t[0], o);
      t[0] = MAX ? fmaxf(t[0], recv) : t[0] + recv;
    }
  }
  // lane l now holds values [base, base + K) with base = (N >= 32 ? K * l : (l >> (5 - log2 N)) ...)
  if (N >= 32) {
#pragma unroll
    for (int i = 0; i < K; ++i) dst[K * lane + i] = t[i];
  } else {
    // N values over 32 lanes: after log2(N) keep-half steps lane l owns value (l >> (5 - log2N))
    constexpr int kShift = (N == 16) ? 1 : 0;
    if ((lane & ((1 << kShift) - 1)) == 0) dst[lane >> kShift] = t[0];
  }
}

// The same over the 16 lanes of each half warp (xor offsets 8..1; the two
// halves reduce independently).  N = 16: lane l of a half ends with value
// l & 15; N = 8: lanes 2k, 2k+1 of a half both hold value k.  Writes dst[i]
// for the lanes that own value i.
template <int N, bool MAX>
__device__ __forceinline__ void half_reduce_scatter(const float (&v)[N], float* dst, int lane) {
  static_assert(N == 8 || N == 16, "values per thread");
  float t[N / 2];
  {
    const bool up = (lane & 8) != 0;
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      const float send = up ? v[i] : v[i + N / 2];
      const float keep = up ? v[i + N / 2] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, 8);
      t[i] = MAX ? fmaxf(keep, recv) : keep + recv;
    }
  }
  int n = N / 2;
#pragma unroll
  for (int o = 4; o >= 1; o >>= 1) {
    if (n > 1) {
      const bool up = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < N / 4; ++i) {
        if (i < n / 2) {
          const float send = up ? t[i] : t[i + n / 2];
          const float keep = up ? t[i + n / 2] : t[i];
          const float recv = __shfl_xor_sync(0xffffffffu, send, o);
          t[i] = MAX ? fmaxf(keep, recv) : keep + recv;
        }
      }
      n >>= 1;
    } else {
      const float recv = __shfl_xor_sync(0xffffffffu, t[0], o);
      t[0] = MAX ? fmaxf(t[0], recv) : t[0] + recv;
    }
  }
  if (N == 16) {
    dst[lane & 15] = t[0];
  } else if ((lane & 1) == 0) {
    dst[(lane >> 1) & 7] = t[0];
  }
}

template <int R, int MODE>
__device__ void softmax_epilogue(const DecodeParams& p, const Segments& sg, int g, int split0, uint32_t tmem,
                                 uint8_t* kv, const Bars& bars, float* aux, volatile uint8_t* flags,
                                 const Watchdog& wd) {
  using C = Cfg<R, MODE>;
  constexpr int RW = R / C::kSmWG;  // rows owned by this warpgroup
  const int wg = (threadIdx.x - 128) >> 7;
  const int rb = wg * RW;           // first row of this warpgroup
  const int tid = (threadIdx.x - 128) & 127;  // TMEM lane (O^T: dv row of a block)
  const int warp_q = (threadIdx.x >> 5) & 3;
  const int lane = threadIdx.x & 31;
  // S^T of a 64-token tile (M = 64) occupies lanes 0..15 of each warp's
  // quarter of TMEM, token 16q + l in lane l of quarter q.  Both halves of a
  // warp work on the same 16 tokens: half hh = lane / 16 takes rows
  // [rb + hh*RH, rb + hh*RH + RH) of this warpgroup's RW rows.
  constexpr int RH = RW / 2;
  const int hh = lane >> 4;
  const int tl = 16 * warp_q + (lane & 15);  // token of the tile
  const int rh = rb + hh * RH;               // first row of this thread
  const uint32_t lane_base = static_cast<uint32_t>(warp_q * 32) << 16;
  const uint32_t bar_id = kSoftmaxBar + wg;
  float* m_s = aux;            // running row max (log2 units)
  float* alpha_s = aux + R;    // rescale factors
  float* inv_s = aux + 2 * R;  // 1 / row sum
  float* lse_s = aux + 3 * R;  // row lse
  float* red = aux + 4 * R;    // [4][R] cross-warp reduction
  // last visible key per row (causal), after the 16 ints and the 256 flag bytes
  int* lim_s = reinterpret_cast<int*>(aux + 8 * R) + 16 + 128;
  const uint32_t kv_base = smem_u32(kv);
  const uint32_t p_row_off = (tl & 7) * 2;  // K-major P: byte of this token inside its 16-byte unit
  const uint32_t p_chunk = tl >> 3;         // K-major P: 16-byte unit of this token
  // The 128 threads of a softmax warpgroup synchronise on their own hardware
  // named barrier.  Every bounded mbarrier wait is followed by a barrier AND
  // of its result, so on a timeout all four warps leave together and none is
  // left at a barrier.  Warpgroups own disjoint rows and never wait on each
  // other; consumers are signalled with one arrival per warp.
  auto group_ok = [&](bool ok) { return named_bar_and(bar_id, 128, ok); };
  auto gsync = [&]() { named_bar_sync(bar_id, 128); };
  auto warp_arrive = [&](uint64_t* b) {
    __syncwarp();
    if (lane == 0) mbar_arrive(b);
  };
  const bool tracer = (wg == 0 && tid == 0);
  int jt = 0, seg = 0;
  float l[RH];
  if (p.debug_stall) {
    // Watchdog test: mma_done only completes after this role has finished, so
    // this wait can only end by the watchdog limit.
    if (!group_ok(mbar_wait(bars.mma_done, 0, wd))) return;
  }

  for (int prob = sg.p0; prob <= sg.last(); ++prob) {
    int tb, te;
    sg.range(prob, tb, te);
    if (tb >= te) continue;
    const int b = C::kIndexed ? prob / p.s_q : prob;
    const int L = p.flat_rows > 0 ? p.flat_rows : sg.seqlens[b];
    // causal limit per row: query token i sees keys <= L - s_q + i (dense only)
    int lim_min = L - 1;
    if (!C::kIndexed && p.is_causal) {
      const int i_first = (g * R + rb) / p.h_q;
      lim_min = min(L - 1, L - p.s_q + i_first);
    }
    if (tid < RW) {
      m_s[rb + tid] = kNegInf;
      lim_s[rb + tid] = (!C::kIndexed && p.is_causal) ? L - p.s_q + (g * R + rb + tid) / p.h_q : L - 1;
    }
#pragma unroll
    for (int r = 0; r < RH; ++r) l[r] = 0.f;
    gsync();

    for (int j = tb; j < te; ++j, ++jt) {
      const int sb = jt & 1;
      if (tracer) MLA_TR(kTrSmWaitS, jt);
      // S^T of this tile is complete; the wait on the tile's (first) full
      // barrier (already complete) orders the loader's validity flags before
      // our reads
      {
        bool ok = mbar_wait(bars.s_full + sb, (jt >> 1) & 1, wd);
        ok = ok && mbar_wait(bars.full + C::kFullItems * Ring<C>::full_index(jt), Ring<C>::full_parity(jt), wd);
        if (!group_ok(ok)) return;
      }
      tc_fence_after();
      const int pos = j * kTileTokens + tl;  // dense: logical token of this thread
      // gathered modes: the gather warps' per-token flag (dense FP8: position
      // below the length and page usable); dense bf16: length and page flag
      const bool tok_ok = C::kGather ? flags[(jt & 3) * 128 + tl] != 0 : (pos < L && flags[(jt & 3) * 128] != 0);
      if (tracer) MLA_TR(kTrSmSFull, jt);

      // this thread's token, its RH rows of S^T (the two halves of the warp
      // read the two halves of the warpgroup's columns)
      float x[RH];
      {
        const uint32_t s_addr = tmem + lane_base + C::kSCol + sb * R + rb;
        if constexpr (RH == 16)
          tmem_ld_16x32bx2_x16<RH>(s_addr, x);
        else
          tmem_ld_16x32bx2_x8<RH>(s_addr, x);
        tmem_ld_wait();
      }
      tc_fence_before();
      warp_arrive(bars.s_empty + sb);  // S is in registers; the buffer can be rewritten
      if (tracer) MLA_TR(kTrSmLoaded, jt);
      if (wg == 0 && lane == 0 && warp_q == 1) MLA_TR(kTrW1Loaded, jt);

      // logits in log2 units; masked -> -inf.  Rows differ only where a causal
      // limit falls inside the tile: their limits come from shared memory.
      const bool all_rows = tok_ok && (C::kIndexed || pos <= lim_min);
      const float sc = p.scale_log2;
      if (all_rows) {
#pragma unroll
        for (int r = 0; r < RH; ++r) x[r] *= sc;
      } else if (C::kIndexed || !tok_ok) {
#pragma unroll
        for (int r = 0; r < RH; ++r) x[r] = kNegInf;
      } else {
#pragma unroll
        for (int r4 = 0; r4 < RH / 4; ++r4) {
          const int4 l4 = reinterpret_cast<const int4*>(lim_s + rh)[r4];
          x[4 * r4] = pos <= l4.x ? x[4 * r4] * sc : kNegInf;
          x[4 * r4 + 1] = pos <= l4.y ? x[4 * r4 + 1] * sc : kNegInf;
          x[4 * r4 + 2] = pos <= l4.z ? x[4 * r4 + 2] * sc : kNegInf;
          x[4 * r4 + 3] = pos <= l4.w ? x[4 * r4 + 3] * sc : kNegInf;
        }
      }

      // lazy max update: raise the running max only when some logit exceeds it
      // by more than the threshold (always on the first tile of a segment)
      bool need = (j == tb);
      if (!need) {
        float loc = kNegInf;
#pragma unroll
        for (int r4 = 0; r4 < RH / 4; ++r4) {
          const float4 m4 = reinterpret_cast<const float4*>(m_s + rh)[r4];
          loc = fmaxf(loc, fmaxf(fmaxf(x[4 * r4] - m4.x, x[4 * r4 + 1] - m4.y),
                                 fmaxf(x[4 * r4 + 2] - m4.z, x[4 * r4 + 3] - m4.w)));
        }
        if (wg == 0 && lane == 0 && warp_q > 0) MLA_TR(kTrW0PreVote + warp_q, jt);
        need = named_bar_or(bar_id, 128, loc > kRescaleThreshold);
        if (tracer) MLA_TR(kTrSmVote, jt);
      }
      if (need) {
        half_reduce_scatter<RH, true>(x, red + warp_q * R + rh, lane);
        gsync();
        if (tid < RW) {
          const int r = rb + tid;
          const float mx = fmaxf(fmaxf(red[r], red[R + r]), fmaxf(red[2 * R + r], red[3 * R + r]));
          const float mo = m_s[r];
          const float mn = fmaxf(mo, mx);
          alpha_s[r] = (mo == kNegInf) ? 0.f : fast_exp2(mo - mn);
          m_s[r] = mn;
        }
        gsync();
#pragma unroll
        for (int r = 0; r < RH; ++r) l[r] *= alpha_s[rh + r];
        if (j != tb) {
          // rescale this warpgroup's row columns of O^T by alpha once the PV
          // MMAs of the previous tile are done (those of earlier tiles are:
          // this tile's loads reused slots they released)
          if (!group_ok(mbar_wait(bars.o_done + ((jt - 1) & 1), ((jt - 1) >> 1) & 1, wd))) return;
          tc_fence_after();
#pragma unroll 1
          for (int blk = 0; blk < 4; ++blk) {
#pragma unroll
            for (int q = 0; q < RW / 16; ++q) {
              float v[16];
              const uint32_t ta = tmem + lane_base + C::kOCol + blk * R + rb + 16 * q;
              tmem_ld_x16(ta, v);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 16; ++e) v[e] *= alpha_s[rb + 16 * q + e];
              tmem_st_x16(ta, v);
            }
          }
          tmem_st_wait();
        }
      }

      // probabilities -> P (bf16) and row sums.  A separate P buffer was last
      // read by the PV of tile jt-2: wait for it (P in the RoPE slot needs no
      // wait: this tile's RoPE chunk was loaded there after that PV).
      if (!C::kPAlias && jt >= 2) {
        if (!group_ok(mbar_wait(bars.o_done + (jt & 1), ((jt - 2) >> 1) & 1, wd))) return;
      }
      const uint32_t p_base = kv_base + Ring<C>::p_off(jt);
#pragma unroll
      for (int r8 = 0; r8 < RH / 8; ++r8) {
        const float4 ma = reinterpret_cast<const float4*>(m_s + rh)[2 * r8];
        const float4 mb = reinterpret_cast<const float4*>(m_s + rh)[2 * r8 + 1];
        const float mr[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
        float pr[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int r = 8 * r8 + e;
          pr[e] = (x[r] == kNegInf) ? 0.f : fast_exp2(x[r] - mr[e]);
          l[r] += pr[e];
        }
        if (C::kPMnMajor) {
          // P^T as [token][R rows] (MN-major B operand): one 16-byte chunk per 8 rows
          const uint32_t ch = (rh >> 3) + r8;
          st_shared_v4(p_base + tl * 128 + ((ch ^ (tl & 7)) << 4), pack_bf16x2(pr[0], pr[1]),
                       pack_bf16x2(pr[2], pr[3]), pack_bf16x2(pr[4], pr[5]), pack_bf16x2(pr[6], pr[7]));
        } else {
          // P as [R rows][64 tokens] (K-major B operand)
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int r = rh + 8 * r8 + e;
            const uint32_t addr = p_base + p_row_off + r * 128 + ((p_chunk ^ (r & 7)) << 4);
            st_shared_u16(addr, __bfloat16_as_ushort(__float2bfloat16_rn(pr[e])));
          }
        }
      }
      if (!C::kGather && !tok_ok) {
        // a masked token's V row must be finite (0 * NaN would poison O): zero
        // it (the warpgroups and warp halves split the eight value chunks)
#pragma unroll 1
        for (int c = 2 * wg + hh; c < 8; c += 2 * C::kSmWG) {
          const uint32_t base = kv_base + Ring<C>::chunk_off(jt, c) + tl * 128;
#pragma unroll
          for (int q = 0; q < 8; ++q) st_shared_v4(base + 16 * q, 0u, 0u, 0u, 0u);
        }
      }
      if (tracer) MLA_TR(kTrSmPStored, jt);
      fence_proxy_async_smem();
      tc_fence_before();
      warp_arrive(bars.p_full + (jt & 1));
      if (tracer) MLA_TR(kTrSmPFull, jt);
      if (wg == C::kSmWG - 1 && tid == 96) MLA_TR(kTrW0PreVote, jt);  // last warp's arrival
    }

    // ---- epilogue: O / l -> out (single piece) or fp32 partial (split problem)
    if (!group_ok(mbar_wait(bars.o_full, seg & 1, wd))) return;
    tc_fence_after();
    if (tracer) MLA_TR(kTrEpiStart, seg);
    half_reduce_scatter<RH, false>(l, red + warp_q * R + rh, lane);
    gsync();
    if (tid < RW) {
      const int r = rb + tid;
      const float lt = red[r] + red[R + r] + red[2 * R + r] + red[3 * R + r];
      inv_s[r] = lt > 0.f ? 1.0f / lt : 0.f;
      lse_s[r] = lt > 0.f ? m_s[r] + log2f(lt) : kNegInf;
    }
    gsync();
    // partial-result slots of this problem: none when this piece is the whole problem
    const int nsplit = p.num_splits[prob + 1] - p.num_splits[prob];
    const bool final_out = nsplit <= 1;
    int slot = p.num_splits[prob] + (prob == sg.p0 ? split0 : 0);
    const int row0 = g * R + rb;
    bool write_ok = true;
    if (!final_out && (slot < 0 || slot >= p.max_slots)) {
      write_ok = false;  // schedule does not match this call: record it, write nothing
      if (tid == 0) atomicOr(p.status, MLA_DEVICE_BAD_SCHEDULE);
    }
#pragma unroll 1
    for (int blk = 0; blk < 4; ++blk) {
      const int dv = blk * 128 + tid;
#pragma unroll
      for (int q = 0; q < RW / 16; ++q) {
        float v[16];
        tmem_ld_x16(tmem + lane_base + C::kOCol + blk * R + rb + 16 * q, v);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int r = 16 * q + e;
          if (write_ok && row0 + r < p.rows) {
            const float o = v[e] * inv_s[rb + r];
            if (final_out) {
              __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
              out[(static_cast<int64_t>(prob) * p.rows + row0 + r) * kDv + dv] = __float2bfloat16_rn(o);
            } else {
              p.o_accum[(static_cast<int64_t>(slot) * p.rows + row0 + r) * kDv + dv] = o;
            }
          }
        }
      }
    }
    if (write_ok && tid < RW && row0 + tid < p.rows) {
      if (final_out)
        p.lse[static_cast<int64_t>(prob) * p.rows + row0 + tid] = lse_s[rb + tid];
      else
        p.lse_accum[static_cast<int64_t>(slot) * p.rows + row0 + tid] = lse_s[rb + tid];
    }
    tc_fence_before();
    warp_arrive(bars.o_empty);
    if (tracer) MLA_TR(kTrEpiEnd, seg);
    ++seg;
  }
}

// ---------------------------------------------------------------------------
// kernel
// ---------------------------------------------------------------------------
template <int R, int MODE>
__global__ void __launch_bounds__(Cfg<R, MODE>::kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
                      const DecodeParams p) {
  using C = Cfg<R, MODE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* kv = smem;
  uint8_t* qs = smem + C::kQOff;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::kAuxOff);
  float* aux = reinterpret_cast<float*>(smem + C::kAuxOff + C::kBarBytes);
  int* ints = reinterpret_cast<int*>(aux + 8 * R);
  volatile int* abort_flag = ints + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ints + 9);
  // flags[(jt & 3) * 128 + t]: sparse: token t of tile jt is valid (written by
  // the gather warps); dense: [0] = the tile's page is usable (written by the
  // producer)
  volatile uint8_t* flags = reinterpret_cast<volatile uint8_t*>(ints + 16);

  Bars bars;
  bars.q_full = bar + 0;
  bars.q_empty = bar + 1;
  bars.full = bar + 2;
  bars.pair_empty = bars.full + C::kNumFull;
  bars.rope_empty = bars.pair_empty + C::kNA;
  bars.s_full = bars.rope_empty + C::kNB;
  bars.s_empty = bars.s_full + 2;
  bars.p_full = bars.s_empty + 2;
  bars.o_full = bars.p_full + 2;
  bars.o_empty = bars.o_full + 1;
  bars.mma_done = bars.o_empty + 1;
  bars.o_done = bars.mma_done + 1;
  bars.raw_full = bars.o_done + 2;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int part = blockIdx.x / p.row_groups;
  const int g = blockIdx.x % p.row_groups;

  if (threadIdx.x == 0) {
    mbar_init(bars.q_full, 1);
    mbar_init(bars.q_empty, 1);
    for (int k = 0; k < C::kNumFull; ++k) mbar_init(bars.full + k, C::kFullArrivals);
    for (int k = 0; k < C::kNA; ++k) mbar_init(bars.pair_empty + k, 1);
    for (int k = 0; k < C::kNB; ++k) mbar_init(bars.rope_empty + k, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bars.s_full + i, 1);
      mbar_init(bars.s_empty + i, 4 * C::kSmWG);  // one arrival per softmax warp
      mbar_init(bars.p_full + i, 4 * C::kSmWG);
    }
    mbar_init(bars.o_done, 1);
    mbar_init(bars.o_done + 1, 1);
    mbar_init(bars.o_full, 1);
    mbar_init(bars.o_empty, 4 * C::kSmWG);
    mbar_init(bars.mma_done, 2);  // one commit per MMA-issuing warp
    // one arrive_expect_tx per issuing warp; bf16 row copies: one arrival per
    // copying thread (the 64 threads of a half)
    for (int k = 0; k < C::kNumRaw; ++k) mbar_init(bars.raw_full + k, (C::kIndexed && !C::kFp8) ? 64 : 2);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_kv);
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  Watchdog wd{abort_flag, p.status, p.timeout_ns};
  // launched as a programmatic dependent of the schedule kernel: everything
  // above overlapped it; its results (and any earlier kernel's) are visible
  // from here on
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the combine kernel (a programmatic dependent of this one) may be
  // scheduled from now on: its blocks wait (griddepcontrol.wait) for this
  // grid to complete, but are resident when it does
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#ifdef MLA_TRACE
  if (threadIdx.x == 0 && blockIdx.x < 1024) {
    g_mla_cta[3 * blockIdx.x] = global_timer_ns();
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    g_mla_cta[3 * blockIdx.x + 2] = smid;
  }
#endif
  Segments sg;
  int split0 = 0;
  // record 0 names the part count and geometry the schedule was made for;
  // only a matching schedule is read further
  if (p.sched[kSchedParts] == p.num_parts && p.sched[kSchedTag] == p.sched_tag) {
    const int32_t* sr = p.sched + static_cast<int64_t>(part) * kSchedInts;
    sg.p0 = sr[kSchedP0];
    sg.t0 = sr[kSchedT0];
    sg.p1 = sr[kSchedP1];
    sg.t1 = sr[kSchedT1];
    split0 = sr[kSchedSplit0];
  } else {
    sg.p0 = -1;  // reported and skipped below
    sg.t0 = sg.p1 = sg.t1 = 0;
  }
  sg.np = p.num_problems;
  sg.s_q = p.s_q;
  sg.topk = p.topk;
  sg.seqlens = p.cache_seqlens;
  if (sg.p0 < 0 || sg.p0 > sg.np || sg.p1 < sg.p0 || sg.p1 > sg.np || sg.t0 < 0 || sg.t1 < 0) {
    if (threadIdx.x == 0) atomicOr(p.status, MLA_DEVICE_BAD_SCHEDULE);
    sg.p0 = sg.np;  // nothing to do
    sg.p1 = sg.np;
  }

  if (warp < 4) {
    if (C::kRegSplit) regs_to<C::kRegsCtl, C::kLaunchRegs>();
    if (warp == 0) {
      producer<R, MODE>(&tm_q, &tm_kv, p, sg, g, kv, qs, bars, flags, wd);  // the whole warp, converged
    } else if (warp == 1) {
      s_issuer<R, MODE>(sg, tmem, kv, qs, bars, wd);  // the whole warp, converged
    } else if (warp == 3) {
      pv_issuer<R, MODE>(sg, tmem, kv, bars, wd);
    }
  } else if (warp < C::kGatherWarp0) {
    if (C::kRegSplit) regs_to<C::kRegsSoftmax, C::kLaunchRegs>();
    softmax_epilogue<R, MODE>(p, sg, g, split0, tmem, kv, bars, aux, flags, wd);
  } else if (C::kGather) {
    if (C::kRegSplit) regs_to<C::kRegsGather, C::kLaunchRegs>();
    gather_rows<R, MODE>(&tm_kv, p, sg, kv, bars, flags, wd);
  }

  tc_fence_before();
  __syncthreads();
#ifdef MLA_TRACE
  if (threadIdx.x == 0 && blockIdx.x < 1024) g_mla_cta[3 * blockIdx.x + 1] = global_timer_ns();
#endif
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int R, int MODE>
cudaError_t launch_one(const CUtensorMap& tm_q, const CUtensorMap& tm_kv, const DecodeParams& p,
                       cudaStream_t stream) {
  using C = Cfg<R, MODE>;
  auto kern = mla_decode_kernel<R, MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  if (C::kRegSplit) {
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs * C::kThreads < C::kRegBudget || fa.numRegs != static_cast<int>(C::kLaunchRegs))
      return cudaErrorInvalidConfiguration;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.num_parts * p.row_groups);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tm_q, tm_kv, p);
}

}  // namespace

size_t decode_smem_bytes(int rpc, int mode) {
  switch (mode * 100 + rpc) {
    case 16: return Cfg<16, kModeDense>::kSmemBytes;
    case 32: return Cfg<32, kModeDense>::kSmemBytes;
    case 64: return Cfg<64, kModeDense>::kSmemBytes;
    case 116: return Cfg<16, kModeSparse>::kSmemBytes;
    case 132: return Cfg<32, kModeSparse>::kSmemBytes;
    case 164: return Cfg<64, kModeSparse>::kSmemBytes;
    case 216: return Cfg<16, kModeDenseFp8>::kSmemBytes;
    case 232: return Cfg<32, kModeDenseFp8>::kSmemBytes;
    case 264: return Cfg<64, kModeDenseFp8>::kSmemBytes;
    case 316: return Cfg<16, kModeSparseBf16>::kSmemBytes;
    case 332: return Cfg<32, kModeSparseBf16>::kSmemBytes;
    case 364: return Cfg<64, kModeSparseBf16>::kSmemBytes;
  }
  return 0;
}

cudaError_t launch_decode(const CUtensorMap& tm_q, const CUtensorMap& tm_kv, const DecodeParams& p, int rpc,
                          int mode, cudaStream_t stream) {
  switch (mode * 100 + rpc) {
    case 16: return launch_one<16, kModeDense>(tm_q, tm_kv, p, stream);
    case 32: return launch_one<32, kModeDense>(tm_q, tm_kv, p, stream);
    case 64: return launch_one<64, kModeDense>(tm_q, tm_kv, p, stream);
    case 116: return launch_one<16, kModeSparse>(tm_q, tm_kv, p, stream);
    case 132: return launch_one<32, kModeSparse>(tm_q, tm_kv, p, stream);
    case 164: return launch_one<64, kModeSparse>(tm_q, tm_kv, p, stream);
    case 216: return launch_one<16, kModeDenseFp8>(tm_q, tm_kv, p, stream);
    case 232: return launch_one<32, kModeDenseFp8>(tm_q, tm_kv, p, stream);
    case 264: return launch_one<64, kModeDenseFp8>(tm_q, tm_kv, p, stream);
    case 316: return launch_one<16, kModeSparseBf16>(tm_q, tm_kv, p, stream);
    case 332: return launch_one<32, kModeSparseBf16>(tm_q, tm_kv, p, stream);
    case 364: return launch_one<64, kModeSparseBf16>(tm_q, tm_kv, p, stream);
  }
  return cudaErrorInvalidValue;
}

#ifdef MLA_TRACE
// Copies the trace buffer (kTrNumEvents x kTraceTiles clock64 stamps) to host memory.
extern "C" int mla_trace_read(unsigned long long* host, size_t n) {
  if (n > sizeof(g_mla_trace) / sizeof(unsigned long long)) n = sizeof(g_mla_trace) / sizeof(unsigned long long);
  if (cudaMemcpyFromSymbol(host, g_mla_trace, n * sizeof(unsigned long long)) != cudaSuccess) return -1;
  unsigned long long z[256] = {};
  for (size_t i = 0; i < sizeof(g_mla_trace); i += sizeof z)
    cudaMemcpyToSymbol(g_mla_trace, z, sizeof z, i);
  return static_cast<int>(n);
}
// Copies the per-CTA start/end stamps and SM ids (3 x 1024 values).
extern "C" int mla_trace_cta_read(unsigned long long* host) {
  return cudaMemcpyFromSymbol(host, g_mla_cta, sizeof(g_mla_cta)) == cudaSuccess ? 0 : -1;
}
#endif

}  // namespace mla
