/*
 * libmla — paged Multi-head Latent Attention (MLA) decode for GB300 (sm_103a).
 *
 * C ABI.  Plain pointers and sizes only; every pointer named "device" must
 * point to memory of the current CUDA device.  The library never allocates
 * device memory: the caller sizes buffers with mla_metadata_size() and
 * mla_workspace_size() and passes them in.  All work is enqueued on the
 * caller's stream and is asynchronous; host-detectable errors return at once
 * with no launch, and mla_last_error() then names the offending argument.
 *
 * The two compute calls follow the decode API described in "Why FlashMLA's
 * decode kernel reaches 660 TFLOPS" (usage section): a scheduling-metadata
 * call made once per decode step and reused by every layer, then one decode
 * call per layer that returns the attention output and its log-sum-exp.
 *
 * Shapes (one KV head; the MQA form of MLA from the Modular design-doc
 * overview, section 9 "Multi-Head Latent Attention": a query row is 576-wide,
 * keys are 576-wide and the value is the first 512 dims of the key):
 *   q             bf16  [batch, s_q, h_q, 576], contiguous
 *   kvcache dense bf16  [num_pages, page_size, 1, 576], contiguous
 *   kvcache fp8   uint8 [num_pages, page_size, 1, 656], contiguous; per token
 *                 bytes [0,512) float8_e4m3 codes of dims 0..511, [512,528)
 *                 four float32 scales (scale k covers dims [128k,128k+128)),
 *                 [528,656) 64 bf16 RoPE values (FlashMLA article, Design 2)
 *   block_table   int32 [batch, block_table_stride]; logical token t of
 *                 element b lives in page block_table[b][t / page_size],
 *                 slot t % page_size (Modular overview, section 4
 *                 "PagedAttention")
 *   cache_seqlens int32 [batch]
 *   indices       int32 [batch, s_q, topk] logical token ids (sparse mode);
 *                 ids outside [0, cache_seqlens[b]) — e.g. -1 — are skipped,
 *                 repeated ids count once per occurrence
 *   out           bf16  [batch, s_q, h_q, 512]
 *   lse           fp32  [batch, s_q, h_q], base 2: log2(sum_j exp(s_j))
 *
 * out = softmax(q K^T * sm_scale) V over the key set of each query row:
 * dense mode = tokens [0, seqlen) (with is_causal: [0, seqlen - s_q + i] for
 * query token i), sparse mode = the valid ids of indices[b, i, :].  A row
 * with an empty key set gets out = 0 and lse = -inf.
 *
 * Supported modes (page_size 64): dense or sparse (top-k), each over a bf16
 * cache or an FP8 cache (is_fp8 selects the format); an FP8 cache may also
 * hold 640-byte rows (codes + RoPE) with one float32 scale per token in a
 * separate array (kv_scales).  Other page sizes return MLA_ERR_UNSUPPORTED.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The caller's CUDA stream (a cudaStream_t / CUstream); NULL = legacy default stream. */
typedef struct CUstream_st* mla_stream_t;

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,    /* null pointer, bad size or alignment; see mla_last_error() */
  MLA_ERR_UNSUPPORTED = 2,    /* valid request outside the supported modes/shapes */
  MLA_ERR_WORKSPACE = 3,      /* workspace missing or smaller than mla_workspace_size() */
  MLA_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed; message has the error */
  MLA_ERR_DEVICE_BOUNDS = 5,  /* device status: a block-table entry outside [0, num_pages) */
  MLA_ERR_DEVICE_TIMEOUT = 6  /* device status: a bounded wait inside a kernel gave up */
} mla_status;

/* Device status bits, reported by mla_get_device_status(). */
#define MLA_DEVICE_BAD_PAGE 0x1u     /* a page id outside [0, num_pages) was skipped (token masked) */
#define MLA_DEVICE_TIMEOUT 0x2u      /* a pipeline wait exceeded its limit; results are invalid */
#define MLA_DEVICE_BAD_SCHEDULE 0x4u /* the schedule did not match the arguments; results invalid */

/* ABI version of this header (incremented on incompatible change). */
#define MLA_ABI_VERSION 3
int mla_abi_version(void);

/* A decode configuration is the tuple (batch, h_q, s_q, topk, is_fp8), in the
 * order of the FlashMLA article's get_mla_metadata(cache_seqlens, ..., h_q,
 * is_fp8, topk) (usage section); topk = 0 selects dense mode, is_fp8 = 1 an
 * FP8 cache.  The three calls below and mla_decode must see the same tuple:
 * the schedule depends on it (rows per CTA, the kernel mode and the cost of a
 * tile in that mode) and on the current device's SM count, so a schedule
 * belongs to one configuration on one device. */

/* Sizes of the two metadata arrays for a decode configuration on the
 * current device (int32 element counts).  sched has one 8-int record per
 * scheduled work part; num_splits has one entry per problem plus one
 * (problem = batch element in dense mode, (batch element, query token) pair
 * in sparse mode). */
mla_status mla_metadata_size(int batch, int h_q, int s_q, int topk, int is_fp8, int* sched_elems,
                             int* num_splits_elems);

/* Scratch bytes that mla_decode needs for split-KV partial results
 * (fp32 partial outputs and their log-sum-exps): min(2 * parts,
 * problems + parts) slots of rows x 513 floats, bounded by the part count
 * whatever the batch size. */
mla_status mla_workspace_size(int batch, int h_q, int s_q, int topk, int is_fp8, size_t* bytes);

/* (1) Tile schedule for one decode step ("get_mla_metadata").
 * cache_seqlens: device int32 [batch]; sched, num_splits: device int32
 * buffers of the sizes above, written on `stream`.  The work of all problems
 * (64-token tiles of their key ranges, each tile weighted by the cost of its
 * mode, FP8 tiles 1.5 times a bf16 tile, plus a fixed start-up cost per
 * problem segment) is divided into contiguous ranges of near-equal cost,
 * one per part; num_splits holds the exclusive prefix sum of the split-KV
 * partial-result slots of each problem: as many as the parts touching it
 * when there are two or more, none when one part covers it (that part writes
 * the output directly).  Every sched record also holds the part count and a
 * tag of the configuration; mla_decode checks both on the device against its
 * own and, on a mismatch, sets MLA_DEVICE_BAD_SCHEDULE and computes nothing
 * (it reads only the first record before that check).  Reusable by every
 * layer of the step as long as cache_seqlens and the configuration are
 * unchanged. */
mla_status mla_get_metadata(const int32_t* cache_seqlens, int batch, int h_q, int s_q, int topk, int is_fp8,
                            int32_t* sched, int32_t* num_splits, mla_stream_t stream);

/* Arguments of mla_decode.  Pointers are device pointers unless noted. */
typedef struct {
  const void* q;                  /* bf16 [batch, s_q, h_q, 576] */
  int batch, s_q, h_q;
  const void* kvcache;            /* bf16 [num_pages,64,1,576], uint8 [num_pages,64,1,656], or with
                                     kv_scales uint8 [num_pages,64,1,640] */
  int num_pages, page_size;       /* page_size must be 64 */
  const int32_t* block_table;     /* int32 [batch, block_table_stride] */
  int block_table_stride;         /* >= ceil(max seqlen / page_size) */
  const int32_t* cache_seqlens;   /* int32 [batch] */
  float sm_scale;                 /* softmax scale applied to q.k */
  int is_causal;                  /* dense only: query token i sees keys <= seqlen - s_q + i */
  int is_fp8;                     /* 1: FP8 cache rows (656 bytes; 640 with kv_scales), 0: bf16
                                     576-value rows (either mode) */
  const int32_t* indices;         /* sparse: int32 [batch, s_q, topk]; NULL for dense */
  int topk;                       /* 0 for dense */
  const int32_t* sched;           /* from mla_get_metadata with the same batch/h_q/s_q/topk/is_fp8 */
  const int32_t* num_splits;
  void* workspace;                /* >= mla_workspace_size() bytes, 256-byte aligned */
  size_t workspace_bytes;
  void* out;                      /* bf16 [batch, s_q, h_q, 512] */
  float* lse;                     /* fp32 [batch, s_q, h_q] */
  /* ABI version 2 (zero when unused): */
  const float* kv_scales;         /* FP8 cache with one scale per token (MAX kernels summary, MLA section:
                                     the scaled decode's per-token KV scales and 640-byte FP8 + BF16 rows):
                                     fp32 [num_pages, 64]; the cache rows are then uint8 [.., 640] = 512
                                     E4M3 codes + 64 bf16 RoPE values, K[d] = bf16_rn(e4m3 * scale) for
                                     d < 512.  NULL: 656-byte rows with four scales each. */
  const int32_t* topk_lengths;    /* sparse, optional: int32 [batch, s_q]; row (b, i) reads only its first
                                     topk_lengths[b, i] index slots (clamped to [0, topk]); NULL: all topk
                                     slots, -1 marking unused ones */
} mla_decode_args;

/* (2) Decode ("flash_mla_with_kvcache"): split-KV attention kernel followed
 * by a log-sum-exp combine of the split partials, both on `stream`.
 * Alignment: q, kvcache and out 16-byte aligned, lse, block_table and
 * kv_scales 4-byte aligned, workspace 256-byte aligned.  Every wait inside
 * the kernels is bounded (2 s by default; the environment variable
 * MLA_WATCHDOG_NS sets another limit in nanoseconds): a wait that runs out
 * sets MLA_DEVICE_TIMEOUT and the kernel returns. */
mla_status mla_decode(const mla_decode_args* args, mla_stream_t stream);

/* Decode without any caller scratch, for callers that cannot allocate device
 * memory when they decode (for example code inside a runtime or plugin host
 * that owns no CUDA memory pool, or a latency-critical path where cudaMalloc
 * is not allowed).  The pages describe no such entry point; it is an addition
 * of this library.  Same arguments and results as mla_decode, except that
 * workspace/workspace_bytes are ignored: the split-KV partials go to a fixed
 * 32 MiB array in the library's device memory, which every GPU that loads
 * this part of the library keeps until exit.  A decode whose scratch (see
 * mla_workspace_size) exceeds 32 MiB returns MLA_ERR_WORKSPACE without
 * launching anything.  The first call on a device looks the array up (once
 * per device) and should come before any stream capture.  All calls share the
 * array, so calls that overlap on the GPU race; serialise them.  Nothing in
 * the array needs to start at zero. */
mla_status mla_decode_noalloc(const mla_decode_args* args, mla_stream_t stream);

/* FP8 cache write: quantise new tokens into the 656-byte FP8 cache row and
 * store them through the block table (the step before a sparse FP8 decode).
 *
 * Row format ("Why FlashMLA's decode kernel reaches 660 TFLOPS", Design 2):
 * dims 0..511 as float8_e4m3 codes in four 1 x 128 tiles, each tile with one
 * float32 scale = amax / 448 (1 for an all-zero tile), code = E4M3 of
 * x / scale (float32 division) rounded to nearest even and saturated at 448;
 * bytes [512, 528) the four scales; bytes [528, 656) dims 512..575 as bf16.
 * Placement (MAX kernels summary, KV-cache store section): the new tokens of
 * batch element b are rows input_row_offsets[b] .. input_row_offsets[b+1]-1
 * of x and go to positions cache_lengths[b] + i of element b, i.e. page
 * block_table[b * block_table_stride + pos / 64], slot pos % 64.
 *
 *   x                 bf16 [num_tokens, 576], device, 16-byte aligned
 *   input_row_offsets int32 [batch + 1], device, non-decreasing, from 0 to num_tokens
 *   cache_lengths     int32 [batch], device: tokens already cached per element
 *   block_table       int32 [batch, block_table_stride], device
 *   kvcache           uint8 [num_pages, 64, 1, 656], device, 16-byte aligned; written
 * The caller owns all memory; the call is asynchronous on `stream`.  A token
 * whose page entry lies past block_table_stride or outside [0, num_pages) is
 * not written and sets MLA_DEVICE_BAD_PAGE in the device status word.  Host-
 * side argument errors return MLA_ERR_INVALID_ARG / MLA_ERR_UNSUPPORTED
 * (page_size != 64) without launching.  num_tokens == 0 launches nothing. */
mla_status mla_fp8_cache_store(const void* x, int num_tokens, const int32_t* input_row_offsets,
                               const int32_t* cache_lengths, int batch, const int32_t* block_table,
                               int block_table_stride, void* kvcache, int num_pages, int page_size,
                               mla_stream_t stream);

/* Sparse prefill ("flash_mla_sparse_fwd(q, kv, indices, sm_scale)" of the
 * FlashMLA article's usage section): token-level sparse attention with no
 * batch dimension and an unpaged bf16 KV with one head.  For query token i
 * and head h the rows kv[indices[i, k]] are gathered (ids outside [0, s_kv)
 * are skipped, a repeated id counts once per occurrence), logits
 * s_k = sm_scale * q[i, h] . kv[id_k], and
 *   out[i, h] = sum_k softmax(s)_k kv[id_k][0:512],   lse[i, h] = log2 sum_k e^{s_k}
 * (base-2 log-sum-exp of the natural logits; no valid id: out = 0,
 * lse = -inf).  The same computation as sparse decode with one batch element
 * whose cache is the KV itself; the library runs its decode kernels on
 * chunks of at most 16384 query tokens. */
typedef struct {
  const void* q;                  /* bf16 [s_q, h_q, 576], 16-byte aligned */
  int s_q, h_q;                   /* h_q <= 1024 */
  const void* kv;                 /* bf16 [s_kv, 576] (the single KV head squeezed out), 16-byte aligned */
  int s_kv;
  const int32_t* indices;         /* int32 [s_q, topk] */
  int topk;                       /* >= 1 */
  float sm_scale;
  void* workspace;                /* >= mla_sparse_prefill_workspace_size() bytes, 256-byte aligned */
  size_t workspace_bytes;
  void* out;                      /* bf16 [s_q, h_q, 512], 16-byte aligned */
  float* lse;                     /* fp32 [s_q, h_q] */
} mla_sparse_prefill_args;

/* Scratch bytes for mla_sparse_prefill: one chunk's schedule and split-KV
 * partials (independent of s_q beyond the first 16384 tokens). */
mla_status mla_sparse_prefill_workspace_size(int s_q, int h_q, int topk, size_t* bytes);

/* Asynchronous on `stream`; all pointers are device pointers owned by the
 * caller.  Host-side argument errors return without launching; device-side
 * problems set bits in the device status word (mla_get_device_status). */
mla_status mla_sparse_prefill(const mla_sparse_prefill_args* args, mla_stream_t stream);

/* FP8 top-k indexer (MAX kernels summary, MLA indexing kernels:
 * mla_fp8_index_top_k): picks, per query token, the topk cached keys that
 * sparse attention will read.  The pages name its steps (FP8 scores with
 * scales, aggregation over the index heads, masking, int32 top-k with -1
 * fill) but give no formula; this library computes, for query row t of
 * element b (rows row_offsets[b] .. row_offsets[b+1]-1, the last n_b
 * positions of a cache of cache_seqlens[b] keys, so row j sees keys
 * s <= seqlen - n_b + j):
 *   score(t, s) = sum_h weights[t,h] * f(q_scales[t,h] * k_scales[s] * sum_d q[t,h,d] * k[s,d])
 * with E4M3 codes q, k (head dim 128), f = ReLU if relu != 0 else identity,
 * (q_scales and k_scales positive, as the amax / 448 quantiser makes them)
 * and writes the ids of the topk visible keys of largest score, in
 * descending score order (ties to the smaller id), -1 after the last visible
 * key.  Scores are computed in fp32 from the exact E4M3 products; keys whose
 * scores differ by less than that rounding may be ordered either way.  Key s
 * of element b is row block_table[b * block_table_stride + s / 64] * 64 + s % 64
 * of the key cache. */
typedef struct {
  const void* q_codes;            /* uint8 E4M3 [num_tokens, h_idx, 128], 16-byte aligned */
  const float* q_scales;          /* fp32 [num_tokens, h_idx] */
  const float* weights;           /* fp32 [num_tokens, h_idx] */
  int num_tokens, h_idx;          /* h_idx a multiple of 8, at most 256 */
  const int32_t* row_offsets;     /* int32 [batch + 1], non-decreasing, row_offsets[batch] = num_tokens */
  int batch;
  int max_new_tokens;             /* >= every element's row count; max_new_tokens * h_idx <= 256 */
  const void* k_codes;            /* uint8 E4M3 [num_pages, 64, 128], 16-byte aligned */
  const float* k_scales;          /* fp32 [num_pages, 64] */
  int num_pages, page_size;       /* page_size must be 64 */
  const int32_t* block_table;     /* int32 [batch, block_table_stride] */
  int block_table_stride;
  const int32_t* cache_seqlens;   /* int32 [batch], each <= block_table_stride * 64 */
  int relu;
  int topk;                       /* 1 .. 16384 */
  void* workspace;                /* >= mla_index_topk_workspace_size() bytes (fp32 scores) */
  size_t workspace_bytes;
  int32_t* indices;               /* out: int32 [num_tokens, topk] */
} mla_index_topk_args;

/* Scratch bytes for mla_index_topk: num_tokens x block_table_stride x 64 fp32 scores. */
mla_status mla_index_topk_workspace_size(int num_tokens, int block_table_stride, size_t* bytes);

/* Asynchronous on `stream`; device pointers owned by the caller.  Host-side
 * argument errors return without launching.  On the device, a block-table
 * entry outside [0, num_pages) sets MLA_DEVICE_BAD_PAGE (its keys are not
 * selected) and an element with more than max_new_tokens rows sets
 * MLA_DEVICE_BAD_SCHEDULE (its rows get -1). */
mla_status mla_index_topk(const mla_index_topk_args* args, mla_stream_t stream);

/* Test hooks, process-wide, for the library's own tests; production callers
 * never need them.  num_parts > 0 makes every later schedule (metadata,
 * workspace and decode geometry) use that many parts instead of the count
 * the SM count gives, to exercise split-KV paths on small inputs; 0 restores
 * the default.  debug_stall != 0 makes the decode kernel's softmax role wait
 * on a barrier that nothing completes, so that its bounded wait runs out and
 * MLA_DEVICE_TIMEOUT is reported; 0 restores normal operation.  The pages
 * describe no such call.  Returns MLA_ERR_INVALID_ARG for num_parts < 0. */
mla_status mla_test_hooks(int num_parts, int debug_stall);

/* Synchronises `stream`, returns the device status bits accumulated since the
 * last call in *flags (0 = clean) and clears them.  Returns
 * MLA_ERR_DEVICE_TIMEOUT / MLA_ERR_DEVICE_BOUNDS when the matching bit is set. */
mla_status mla_get_device_status(mla_stream_t stream, uint32_t* flags);

/* Thread-local description of the last error returned on this thread
 * (empty string if none).  The pointer stays valid until the next call. */
const char* mla_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H_ */
