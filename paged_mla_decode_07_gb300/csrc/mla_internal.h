// Internal definitions shared by the libmla translation units (host API and
// kernels).  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <string>

#include "../../include/mla.h"

namespace mla {

constexpr int kDqk = 576;          // latent (512 NoPE) + 64 RoPE dims per token
constexpr int kDv = 512;           // value dims = first 512 key dims
constexpr int kChunk = 64;         // dims per 128-byte swizzle atom row (bf16)
constexpr int kNumChunks = 9;      // 576 / 64
constexpr int kPageSize = 64;      // tokens per page
constexpr int kTileTokens = 64;    // tokens per KV tile (one page) = MMA M of S^T = K Q^T
constexpr int kFp8RowBytes = 656;  // 512 e4m3 + 4 fp32 scales + 64 bf16
constexpr int kFp8ScaleOffset = 512;
constexpr int kFp8RopeOffset = 528;
constexpr int kSchedInts = 8;      // ints per schedule record

// Schedule record of one part (a group of `row_groups` CTAs that walk the
// same tiles, one CTA per row group):
//   [0] first problem  [1] first tile in it  [2] last problem (inclusive bound)
//   [3] end tile in the last problem (exclusive)  [4] split index of the
//   part's piece of its first problem  [5] number of parts the schedule was
//   cut into  [6] geometry tag of the decode it was made for  [7] unused (0)
// The decode kernel compares [5] and [6] of record 0 with its own launch
// before it reads any other record, so a schedule made for another
// configuration (or another device) is reported, never followed.
enum SchedField { kSchedP0 = 0, kSchedT0 = 1, kSchedP1 = 2, kSchedT1 = 3, kSchedSplit0 = 4, kSchedParts = 5,
                  kSchedTag = 6 };

constexpr int kMaxProblems = 16384;    // metadata kernel keeps per-problem prefix sums in smem

// Number of tiles of problem p: dense covers the cached tokens [0, seqlen),
// sparse covers the topk index slots of the query token.  Tiles are 64
// tokens (one page) for the single-CTA kernel and 128 (two pages, one per
// CTA) for the CTA-pair kernel.
__host__ __device__ inline int problem_tiles(const int32_t* cache_seqlens, int p, int s_q, int topk,
                                             int tile_tokens = kTileTokens) {
  if (topk > 0) return (topk + tile_tokens - 1) / tile_tokens;
  int L = cache_seqlens[p];
  return L > 0 ? (L + tile_tokens - 1) / tile_tokens : 0;
}

// Rows per CTA for a problem with `rows` query rows sharing one key set.
inline int rows_per_cta(int rows) { return rows > 32 ? 64 : (rows > 16 ? 32 : 16); }

struct Geometry {
  int num_problems;  // dense: batch; sparse: batch * s_q
  int rows;          // query rows per problem: dense s_q*h_q; sparse h_q
  int rpc;           // rows per CTA (16, 32, 64)
  int row_groups;    // ceil(rows / rpc)
  int num_parts;     // schedule parts (each = row_groups CTAs)
  int sm_count;
  int mode;          // decode kernel mode: 0 dense bf16, 1 sparse FP8, 2 dense FP8, 3 sparse bf16 rows
  int pair;          // 1: CTA-pair kernel (128 rows and 128-token tiles per pair), 0: one CTA per row group
  int tile_tokens;   // tokens per schedule tile (64, or 128 for the pair kernel)
  int tile_cost;     // schedule cost of one tile (quarter units of a 64-token bf16 tile)
  int overhead;      // schedule cost of starting a problem segment (same units)
  int tag;           // geometry tag written into the schedule records
};

struct DecodeParams {
  const int32_t* block_table;
  const int32_t* cache_seqlens;
  const int32_t* indices;
  const int32_t* sched;
  const int32_t* num_splits;
  const uint8_t* kv_fp8;      // sparse: raw FP8 cache
  void* out;                  // bf16 [num_problems * rows, 512]
  float* lse;                 // [num_problems * rows]
  float* o_accum;             // [slots, rows, 512]
  float* lse_accum;           // [slots, rows]
  uint32_t* status;
  uint64_t timeout_ns;
  int batch, s_q, h_q, topk;
  int num_pages, block_table_stride;
  int num_problems, rows, row_groups, num_parts;
  int max_slots;              // partial-result slots the workspace holds
  int is_causal;
  int evict_first;
  int sched_tag;              // expected kSchedTag of the schedule records
  int debug_stall;            // test hook: the softmax role waits on a barrier nothing completes
  int flat_rows;              // > 0: sparse over an unpaged KV of this many rows (index = row; no
                              // block table or cache_seqlens); 0: paged cache
  const float* kv_scales;     // FP8 rows with one scale per token ([rows] fp32), else NULL
  const int32_t* topk_lengths;  // sparse: valid index slots per problem, else NULL
  int fp8_rope_off;           // byte offset of the RoPE dims in a row (FP8: 528, or 512 with kv_scales;
                              // bf16 rows: 1024)
  int rows16;                 // CTA-pair sparse decode: the rows are bf16 (1152 bytes, used as they
                              // are), 0: FP8 rows, dequantised

  float scale_log2;           // sm_scale * log2(e)
};

struct CombineParams {
  const int32_t* num_splits;
  const int32_t* cache_seqlens;  // problems without tiles get out = 0, lse = -inf (sparse: unused)
  int s_q, topk;
  const float* o_accum;
  const float* lse_accum;
  void* out;
  float* lse;
  int num_problems, rows;
  int max_slots;
  uint32_t* status;
};

struct IndexParams {
  const float* q_scales;      // [num_tokens, h_idx]
  const float* weights;       // [num_tokens, h_idx]
  const int32_t* row_offsets; // [batch + 1]
  const float* k_scales;      // [num_pages * 64]
  const int32_t* block_table;
  const int32_t* cache_seqlens;
  float* scores;              // [num_tokens, width]
  uint32_t* status;
  uint64_t timeout_ns;
  int64_t width;              // block_table_stride * 64: the longest possible key range
  int batch, num_tokens, h_idx, max_new, n_box, num_pages, block_table_stride, relu, tiles_per_cta;
  uint32_t tmem_cols;         // two accumulator buffers of tmem_cols / 2 >= n_box columns
};

// Kernel launchers (defined in the .cu files); return a CUDA error code.
cudaError_t launch_metadata(const int32_t* cache_seqlens, int s_q, int topk, const Geometry& g, int32_t* sched,
                            int32_t* num_splits, cudaStream_t stream);
// mode: 0 dense bf16 cache, 1 sparse FP8 cache, 2 dense FP8 cache, 3 sparse bf16 rows
cudaError_t launch_decode(const CUtensorMap& tm_q, const CUtensorMap& tm_kv, const DecodeParams& p, int rpc,
                          int mode, cudaStream_t stream);
// CTA pairs the pair decode kernel can keep resident at once on the current
// device (0 if the query fails)
int pair_cluster_capacity();
// CTA-pair decode for problems of more than 64 rows: dense over the bf16 cache
// (tm_q, tm_ks, tm_kv: chunk-major maps with boxes of 9 chunks (Q), 3 and 2
// chunks (cache)) or sparse over the FP8 cache (tm_q as before, tm_ks: the
// FP8 rows as 128-byte boxes of one row for row gathers, tm_kv unused)
cudaError_t launch_decode_pair(const CUtensorMap& tm_q, const CUtensorMap& tm_ks, const CUtensorMap& tm_kv,
                               const DecodeParams& p, bool sparse, cudaStream_t stream);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream, bool pdl);
size_t decode_smem_bytes(int rpc, int mode);
cudaError_t launch_fp8_cache_store(const uint16_t* x, int num_tokens, const int32_t* row_offsets,
                                   const int32_t* cache_lengths, int batch, const int32_t* block_table,
                                   int block_table_stride, uint8_t* kvcache, int num_pages, uint32_t* status,
                                   int sm_count, cudaStream_t stream);
cudaError_t launch_index(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const IndexParams& p, int topk,
                         int32_t* out, cudaStream_t stream);
// Sets the thread-local message returned by mla_last_error().
void set_error_message(const std::string& msg);

}  // namespace mla
