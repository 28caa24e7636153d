// libmla host side: argument validation, geometry, TMA tensor maps, launches,
// device status and error reporting for the C ABI declared in include/mla.h.
//
// Error convention: each entry point checks every argument it can on the
// host and returns a status code without launching anything on failure; the
// thread-local message names the offending argument (the validation style of
// the MAX kernel wrappers, max.nn.kernels module overview).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "mla_internal.h"

namespace mla {

size_t metadata_smem_bytes(int np, int num_parts);

namespace {

thread_local std::string g_error;

mla_status fail(mla_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_error = buf;
  return s;
}

mla_status ok() {
  g_error.clear();
  return MLA_OK;
}

mla_status cuda_fail(cudaError_t e, const char* what) {
  return fail(MLA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// Device status word: one per device (a module global), its address fetched
// once per device.
__device__ uint32_t g_device_status;
constexpr int kMaxDevices = 64;
uint32_t* g_status_ptr[kMaxDevices];
int g_sm_count[kMaxDevices];
int g_pair_capacity[kMaxDevices];  // co-resident CTA pairs of the pair decode kernel
std::mutex g_mu;

mla_status device_info(uint32_t** status, int* sm_count, int* pair_capacity = nullptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(MLA_ERR_UNSUPPORTED, "device ordinal %d too large", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_device_status);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
    g_status_ptr[dev] = static_cast<uint32_t*>(ptr);
    g_sm_count[dev] = sms;
    const int cap = pair_cluster_capacity();
    g_pair_capacity[dev] = (cap > 0 && cap < sms / 2) ? cap : sms / 2;
  }
  if (status) *status = g_status_ptr[dev];
  if (sm_count) *sm_count = g_sm_count[dev];
  if (pair_capacity) *pair_capacity = g_pair_capacity[dev];
  return MLA_OK;
}

// The CTA-pair decode kernel for problems of more than 64 rows, dense over
// the bf16 cache or sparse over FP8 or bf16 rows (mla_decode_pair.cu).
constexpr bool kPairDecode = true;
// Sparse on CTA pairs.
constexpr bool kPairSparse = true;

// Test hooks (mla_test_hooks): a forced part count and a stalled softmax role.
std::atomic<int> g_test_num_parts{0};
std::atomic<int> g_test_debug_stall{0};

// Kernel mode of a decode: 0 dense over the bf16 cache, 1 sparse over the FP8
// cache, 2 dense over the FP8 cache, 3 sparse over bf16 rows.
int decode_mode(int topk, int is_fp8) { return topk > 0 ? (is_fp8 ? 1 : 3) : (is_fp8 ? 2 : 0); }

mla_status geometry(int batch, int h_q, int s_q, int topk, int is_fp8, Geometry* g) {
  if (batch < 1) return fail(MLA_ERR_INVALID_ARG, "batch must be >= 1 (got %d)", batch);
  if (s_q < 1) return fail(MLA_ERR_INVALID_ARG, "s_q must be >= 1 (got %d)", s_q);
  if (h_q < 1) return fail(MLA_ERR_INVALID_ARG, "h_q must be >= 1 (got %d)", h_q);
  if (topk < 0) return fail(MLA_ERR_INVALID_ARG, "topk must be >= 0 (got %d)", topk);
  const long long np = topk > 0 ? static_cast<long long>(batch) * s_q : batch;
  const long long rows = topk > 0 ? h_q : static_cast<long long>(s_q) * h_q;
  if (np > kMaxProblems)
    return fail(MLA_ERR_UNSUPPORTED, "%s = %lld exceeds the supported %d problems",
                topk > 0 ? "batch*s_q" : "batch", np, kMaxProblems);
  if (rows > 1024)
    return fail(MLA_ERR_UNSUPPORTED, "%s = %lld query rows per problem exceeds 1024",
                topk > 0 ? "h_q" : "s_q*h_q", rows);
  if (topk > (1 << 24)) return fail(MLA_ERR_UNSUPPORTED, "topk = %d too large", topk);
  if (is_fp8 != 0 && is_fp8 != 1) return fail(MLA_ERR_INVALID_ARG, "is_fp8 must be 0 or 1 (got %d)", is_fp8);
  int sms = 0, pairs = 0;
  mla_status st = device_info(nullptr, &sms, &pairs);
  if (st != MLA_OK) return st;
  g->num_problems = static_cast<int>(np);
  g->rows = static_cast<int>(rows);
  g->mode = decode_mode(topk, is_fp8);
  g->sm_count = sms;
  // problems of more than 64 rows, dense over the bf16 cache or sparse (FP8
  // or bf16 rows), run on CTA pairs (128 rows and 128-token tiles per pair);
  // everything else on single CTAs
  g->pair = (kPairDecode && (g->mode == 0 || (kPairSparse && (g->mode == 1 || g->mode == 3))) && g->rows > 64)
                ? 1
                : 0;
  g->rpc = g->pair ? 128 : rows_per_cta(g->rows);
  g->tile_tokens = g->pair ? 128 : kTileTokens;
  g->row_groups = (g->rows + g->rpc - 1) / g->rpc;
  // persistent grids: one CTA (or CTA pair) per SM (or per pair of SMs that
  // can hold one) for every row group of a part
  g->num_parts = (g->pair ? pairs : sms) / g->row_groups;
  const int forced = g_test_num_parts.load();
  if (forced > 0) g->num_parts = forced;
  if (g->num_parts < 1) g->num_parts = 1;
  // schedule costs in quarters of a 64-token bf16 tile: FP8 rows are
  // dequantised before their MMAs, so their tiles weigh more against the
  // fixed start-up of a segment
  g->tile_cost = (is_fp8 ? 6 : 4) * (g->tile_tokens / kTileTokens);
  g->overhead = 8;
  g->tag = g->rpc | (g->mode << 8) | ((g->tile_tokens / kTileTokens) << 12) | (g->pair << 15);
  return MLA_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Partial-result slots: only split problems take slots, at most two per part
// (see the metadata kernel), independent of the number of problems.
int max_slots(const Geometry& g) {
  // also at most one piece per problem plus one per part boundary
  return g.num_problems + g.num_parts < 2 * g.num_parts ? g.num_problems + g.num_parts : 2 * g.num_parts;
}

void workspace_layout(const Geometry& g, size_t* o_bytes, size_t* lse_bytes) {
  const size_t slots = static_cast<size_t>(max_slots(g));
  *o_bytes = align256(slots * g.rows * kDv * sizeof(float));
  *lse_bytes = align256(slots * g.rows * sizeof(float));
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 576-wide bf16 rows viewed as [rows][9 chunks][64]: dim0 = 64 elements
// (128 B, the swizzle atom width), dim1 = chunk (stride 128 B), dim2 = row
// (stride 1152 B).  A box of {64, 1, box_rows} lands in shared memory as
// box_rows x 128 B with the 128-byte swizzle, the canonical K-major operand
// layout of the tcgen05 MMAs.
mla_status encode_rows_map(CUtensorMap* map, const void* base, long long nrows, int box_rows, const char* what) {
  auto fn = encode_fn();
  if (!fn) return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  cuuint64_t dims[3] = {64, 9, static_cast<cuuint64_t>(nrows)};
  cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(kDqk * 2)};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with CUresult %d", what, (int)r);
  return MLA_OK;
}

// The same 576-wide bf16 rows viewed chunk-major: dim0 = 64 elements of a
// chunk, dim1 = row (stride 1152 B), dim2 = chunk (stride 128 B).  A box of
// {64, 64, n} copies n chunks of 64 consecutive rows in one instruction and
// lands as n x [64 rows][128 B] with the 128-byte swizzle: n consecutive
// K-major operand tiles of the tcgen05 MMAs.
mla_status encode_chunk_major_map(CUtensorMap* map, const void* base, long long nrows, int box_chunks,
                                  const char* what) {
  auto fn = encode_fn();
  if (!fn) return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(nrows), 9};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kDqk * 2), 128};
  cuuint32_t box[3] = {64, 64, static_cast<cuuint32_t>(box_chunks)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with CUresult %d", what, (int)r);
  return MLA_OK;
}

// Cache rows as raw bytes, [rows][row_bytes] (row = page * 64 + slot, or the
// row of an unpaged KV): FP8 rows (656 bytes) or bf16 rows (1152 bytes).  A
// box is 128 bytes of box_rows rows: one row for the sparse row gathers (as
// row gathers require), 32 consecutive rows of a page for dense decode over
// the FP8 cache; no swizzle: the rows land as plain 128-byte rows.
mla_status encode_byte_rows_map(CUtensorMap* map, const void* base, long long nrows, int row_bytes, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(nrows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
  cuuint32_t box[2] = {128, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled(kv rows) failed with CUresult %d", (int)r);
  return MLA_OK;
}

// E4M3 rows of 128 bytes, [rows][128], 128-byte swizzle: a box of box_rows
// rows lands as the canonical K-major operand of a kind::f8f6f4 MMA.
mla_status encode_e4m3_rows_map(CUtensorMap* map, const void* base, long long nrows, int box_rows, const char* what) {
  auto fn = encode_fn();
  if (!fn) return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(nrows)};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {128, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with CUresult %d", what, (int)r);
  return MLA_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

uint64_t watchdog_ns() {
  const char* s = getenv("MLA_WATCHDOG_NS");
  if (s) {
    unsigned long long v = strtoull(s, nullptr, 10);
    if (v > 0) return v;
  }
  return 2000000000ull;  // 2 s: far above any legitimate wait, short enough to unwind quickly
}

}  // namespace

void set_error_message(const std::string& msg) { g_error = msg; }

}  // namespace mla

using namespace mla;

// Sparse prefill runs the decode pipeline (schedule, attention, combine) on
// chunks of at most kMaxProblems query tokens; the workspace holds one
// chunk's schedule, slot prefix sums and split-KV partials.
namespace {
struct PrefillLayout {
  size_t sched, num_splits, o_accum, lse_accum, total;
};
mla_status prefill_layout(int s_q, int h_q, int topk, Geometry* g, PrefillLayout* L) {
  const int chunk = s_q < kMaxProblems ? s_q : kMaxProblems;
  mla_status st = geometry(1, h_q, chunk, topk, 0, g);
  if (st != MLA_OK) return st;
  size_t ob, lb;
  workspace_layout(*g, &ob, &lb);
  L->sched = 0;
  L->num_splits = align256(static_cast<size_t>(g->num_parts) * kSchedInts * sizeof(int32_t));
  L->o_accum = L->num_splits + align256(static_cast<size_t>(chunk + 1) * sizeof(int32_t));
  L->lse_accum = L->o_accum + ob;
  L->total = L->lse_accum + lb;
  return MLA_OK;
}
}  // namespace

extern "C" {

int mla_abi_version(void) { return MLA_ABI_VERSION; }

const char* mla_last_error(void) { return g_error.c_str(); }

mla_status mla_test_hooks(int num_parts, int debug_stall) {
  if (num_parts < 0) return fail(MLA_ERR_INVALID_ARG, "num_parts must be >= 0 (got %d)", num_parts);
  g_test_num_parts.store(num_parts);
  g_test_debug_stall.store(debug_stall != 0 ? 1 : 0);
  return ok();
}

mla_status mla_metadata_size(int batch, int h_q, int s_q, int topk, int is_fp8, int* sched_elems,
                             int* num_splits_elems) {
  if (!sched_elems) return fail(MLA_ERR_INVALID_ARG, "sched_elems is NULL");
  if (!num_splits_elems) return fail(MLA_ERR_INVALID_ARG, "num_splits_elems is NULL");
  Geometry g{};
  mla_status st = geometry(batch, h_q, s_q, topk, is_fp8, &g);
  if (st != MLA_OK) return st;
  *sched_elems = g.num_parts * kSchedInts;
  *num_splits_elems = g.num_problems + 1;
  return ok();
}

mla_status mla_workspace_size(int batch, int h_q, int s_q, int topk, int is_fp8, size_t* bytes) {
  if (!bytes) return fail(MLA_ERR_INVALID_ARG, "bytes is NULL");
  Geometry g{};
  mla_status st = geometry(batch, h_q, s_q, topk, is_fp8, &g);
  if (st != MLA_OK) return st;
  size_t ob, lb;
  workspace_layout(g, &ob, &lb);
  *bytes = ob + lb;
  return ok();
}

mla_status mla_get_metadata(const int32_t* cache_seqlens, int batch, int h_q, int s_q, int topk, int is_fp8,
                            int32_t* sched, int32_t* num_splits, mla_stream_t stream) {
  if (!cache_seqlens) return fail(MLA_ERR_INVALID_ARG, "cache_seqlens is NULL");
  if (!sched) return fail(MLA_ERR_INVALID_ARG, "sched is NULL");
  if (!num_splits) return fail(MLA_ERR_INVALID_ARG, "num_splits is NULL");
  Geometry g{};
  mla_status st = geometry(batch, h_q, s_q, topk, is_fp8, &g);
  if (st != MLA_OK) return st;
  cudaError_t e = launch_metadata(cache_seqlens, s_q, topk, g, sched, num_splits,
                                  reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "metadata kernel launch");
  return ok();
}

mla_status mla_decode(const mla_decode_args* a, mla_stream_t stream) {
  if (!a) return fail(MLA_ERR_INVALID_ARG, "args is NULL");
  const bool sparse = a->topk > 0;
  if (a->topk < 0) return fail(MLA_ERR_INVALID_ARG, "topk must be >= 0 (got %d)", a->topk);
  if (!a->q) return fail(MLA_ERR_INVALID_ARG, "q is NULL");
  if (!a->kvcache) return fail(MLA_ERR_INVALID_ARG, "kvcache is NULL");
  if (!a->block_table) return fail(MLA_ERR_INVALID_ARG, "block_table is NULL");
  if (!a->cache_seqlens) return fail(MLA_ERR_INVALID_ARG, "cache_seqlens is NULL");
  if (!a->sched) return fail(MLA_ERR_INVALID_ARG, "sched is NULL");
  if (!a->num_splits) return fail(MLA_ERR_INVALID_ARG, "num_splits is NULL");
  if (!a->out) return fail(MLA_ERR_INVALID_ARG, "out is NULL");
  if (!a->lse) return fail(MLA_ERR_INVALID_ARG, "lse is NULL");
  if (sparse && !a->indices) return fail(MLA_ERR_INVALID_ARG, "indices is NULL with topk = %d", a->topk);
  if (!sparse && a->indices) return fail(MLA_ERR_INVALID_ARG, "indices given with topk = 0");
  if (a->page_size != kPageSize)
    return fail(MLA_ERR_UNSUPPORTED, "page_size must be %d (got %d)", kPageSize, a->page_size);
  if (a->num_pages < 1) return fail(MLA_ERR_INVALID_ARG, "num_pages must be >= 1 (got %d)", a->num_pages);
  if (static_cast<long long>(a->num_pages) * kPageSize > (1ll << 31) - 1)
    return fail(MLA_ERR_UNSUPPORTED, "num_pages = %d exceeds 2^31 tokens", a->num_pages);
  if (a->block_table_stride < 1)
    return fail(MLA_ERR_INVALID_ARG, "block_table_stride must be >= 1 (got %d)", a->block_table_stride);
  if (a->is_causal && sparse) return fail(MLA_ERR_UNSUPPORTED, "is_causal applies to dense mode only");
  if (a->kv_scales && !a->is_fp8) return fail(MLA_ERR_INVALID_ARG, "kv_scales given with a bf16 cache (is_fp8 = 0)");
  if (a->topk_lengths && !sparse) return fail(MLA_ERR_INVALID_ARG, "topk_lengths given with topk = 0");
  if (a->kv_scales && !aligned(a->kv_scales, 4)) return fail(MLA_ERR_INVALID_ARG, "kv_scales is not 4-byte aligned");
  if (!std::isfinite(a->sm_scale)) return fail(MLA_ERR_INVALID_ARG, "sm_scale is not finite");
  if (!aligned(a->q, 16)) return fail(MLA_ERR_INVALID_ARG, "q is not 16-byte aligned");
  if (!aligned(a->kvcache, 16)) return fail(MLA_ERR_INVALID_ARG, "kvcache is not 16-byte aligned");
  if (!aligned(a->out, 16)) return fail(MLA_ERR_INVALID_ARG, "out is not 16-byte aligned");
  if (!aligned(a->lse, 4)) return fail(MLA_ERR_INVALID_ARG, "lse is not 4-byte aligned");
  if (!aligned(a->block_table, 4)) return fail(MLA_ERR_INVALID_ARG, "block_table is not 4-byte aligned");

  if (a->is_fp8 != 0 && a->is_fp8 != 1) return fail(MLA_ERR_INVALID_ARG, "is_fp8 must be 0 or 1 (got %d)", a->is_fp8);
  Geometry g{};
  mla_status st = geometry(a->batch, a->h_q, a->s_q, a->topk, a->is_fp8, &g);
  if (st != MLA_OK) return st;
  size_t ob, lb;
  workspace_layout(g, &ob, &lb);
  if (!a->workspace) return fail(MLA_ERR_WORKSPACE, "workspace is NULL (%zu bytes needed)", ob + lb);
  if (a->workspace_bytes < ob + lb)
    return fail(MLA_ERR_WORKSPACE, "workspace_bytes = %zu < %zu needed", a->workspace_bytes, ob + lb);
  if (!aligned(a->workspace, 256)) return fail(MLA_ERR_INVALID_ARG, "workspace is not 256-byte aligned");

  uint32_t* status = nullptr;
  st = device_info(&status, nullptr);
  if (st != MLA_OK) return st;

  CUtensorMap tm_q, tm_kv, tm_kv2;
  const long long qrows = static_cast<long long>(a->batch) * a->s_q * a->h_q;
  const long long cache_rows = static_cast<long long>(a->num_pages) * kPageSize;
  if (g.pair) {
    // chunk-major boxes: Q of a CTA in one copy; dense: a page's score operand
    // in three copies of three chunks, its value shares in copies of two
    // chunks.  Sparse: the rows are copied by the gather warps with cp.async
    // and the two cache maps go unused.
    st = encode_chunk_major_map(&tm_q, a->q, qrows, kNumChunks, "q");
    if (st == MLA_OK && g.mode == 0) st = encode_chunk_major_map(&tm_kv, a->kvcache, cache_rows, 3, "kvcache");
    if (st == MLA_OK && g.mode == 0) st = encode_chunk_major_map(&tm_kv2, a->kvcache, cache_rows, 2, "kvcache");
    if (st != MLA_OK) return st;
    if (g.mode == 1 || g.mode == 3) tm_kv = tm_kv2 = tm_q;
  } else {
    st = encode_rows_map(&tm_q, a->q, qrows, g.rpc, "q");
  }
  if (st != MLA_OK) return st;
  const int mode = g.mode;
  if (g.pair)
    ;  // maps encoded above
  else if (mode == 0)
    st = encode_rows_map(&tm_kv, a->kvcache, cache_rows, kPageSize, "kvcache");
  else if (mode == 3)
    st = encode_byte_rows_map(&tm_kv, a->kvcache, cache_rows, 2 * kDqk, 1);
  else
    st = encode_byte_rows_map(&tm_kv, a->kvcache, cache_rows, a->kv_scales ? 640 : kFp8RowBytes, mode == 1 ? 1 : 32);
  if (st != MLA_OK) return st;

  DecodeParams p;
  memset(&p, 0, sizeof p);
  p.block_table = a->block_table;
  p.cache_seqlens = a->cache_seqlens;
  p.indices = a->indices;
  p.sched = a->sched;
  p.num_splits = a->num_splits;
  p.kv_fp8 = static_cast<const uint8_t*>(a->kvcache);
  p.out = a->out;
  p.lse = a->lse;
  p.o_accum = static_cast<float*>(a->workspace);
  p.lse_accum = reinterpret_cast<float*>(static_cast<char*>(a->workspace) + ob);
  p.status = status;
  p.timeout_ns = watchdog_ns();
  p.batch = a->batch;
  p.s_q = a->s_q;
  p.h_q = a->h_q;
  p.topk = a->topk;
  p.num_pages = a->num_pages;
  p.block_table_stride = a->block_table_stride;
  p.num_problems = g.num_problems;
  p.rows = g.rows;
  p.row_groups = g.row_groups;
  p.num_parts = g.num_parts;
  p.max_slots = max_slots(g);
  p.is_causal = a->is_causal ? 1 : 0;
  p.evict_first = (g.row_groups == 1 && !g.pair) ? 1 : 0;
  p.sched_tag = g.tag;
  p.debug_stall = g_test_debug_stall.load();
  p.scale_log2 = a->sm_scale * 1.4426950408889634f;
  p.kv_scales = a->kv_scales;
  p.topk_lengths = a->topk_lengths;
  p.fp8_rope_off = mode == 3 ? 2 * kDv : (a->kv_scales ? kDv : kFp8RopeOffset);
  p.rows16 = mode == 3 ? 1 : 0;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = g.pair ? launch_decode_pair(tm_q, tm_kv, tm_kv2, p, g.mode == 1 || g.mode == 3, s)
                         : launch_decode(tm_q, tm_kv, p, g.rpc, mode, s);
  if (e != cudaSuccess) return cuda_fail(e, "decode kernel launch");

  CombineParams cp;
  cp.num_splits = a->num_splits;
  cp.cache_seqlens = a->cache_seqlens;
  cp.s_q = a->s_q;
  cp.topk = a->topk;
  cp.o_accum = p.o_accum;
  cp.lse_accum = p.lse_accum;
  cp.out = a->out;
  cp.lse = a->lse;
  cp.num_problems = g.num_problems;
  cp.rows = g.rows;
  cp.max_slots = p.max_slots;
  cp.status = status;
  e = launch_combine(cp, s, true);
  if (e != cudaSuccess) return cuda_fail(e, "combine kernel launch");
  return ok();
}

mla_status mla_fp8_cache_store(const void* x, int num_tokens, const int32_t* input_row_offsets,
                               const int32_t* cache_lengths, int batch, const int32_t* block_table,
                               int block_table_stride, void* kvcache, int num_pages, int page_size,
                               mla_stream_t stream) {
  if (batch < 1) return fail(MLA_ERR_INVALID_ARG, "batch = %d must be >= 1", batch);
  if (num_tokens < 0) return fail(MLA_ERR_INVALID_ARG, "num_tokens = %d must be >= 0", num_tokens);
  if (page_size != kPageSize) return fail(MLA_ERR_UNSUPPORTED, "page_size must be 64 (got %d)", page_size);
  if (num_pages < 1) return fail(MLA_ERR_INVALID_ARG, "num_pages = %d must be >= 1", num_pages);
  if (block_table_stride < 1)
    return fail(MLA_ERR_INVALID_ARG, "block_table_stride = %d must be >= 1", block_table_stride);
  if (num_tokens > 0 && !x) return fail(MLA_ERR_INVALID_ARG, "x is NULL");
  if (!input_row_offsets) return fail(MLA_ERR_INVALID_ARG, "input_row_offsets is NULL");
  if (!cache_lengths) return fail(MLA_ERR_INVALID_ARG, "cache_lengths is NULL");
  if (!block_table) return fail(MLA_ERR_INVALID_ARG, "block_table is NULL");
  if (!kvcache) return fail(MLA_ERR_INVALID_ARG, "kvcache is NULL");
  if (x && !aligned(x, 16)) return fail(MLA_ERR_INVALID_ARG, "x is not 16-byte aligned");
  if (!aligned(kvcache, 16)) return fail(MLA_ERR_INVALID_ARG, "kvcache is not 16-byte aligned");
  uint32_t* status = nullptr;
  int sms = 0;
  mla_status st = device_info(&status, &sms);
  if (st != MLA_OK) return st;
  cudaError_t e = launch_fp8_cache_store(static_cast<const uint16_t*>(x), num_tokens, input_row_offsets,
                                         cache_lengths, batch, block_table, block_table_stride,
                                         static_cast<uint8_t*>(kvcache), num_pages, status, sms, stream);
  if (e != cudaSuccess) return cuda_fail(e, "fp8 cache store launch");
  return ok();
}

mla_status mla_sparse_prefill_workspace_size(int s_q, int h_q, int topk, size_t* bytes) {
  if (!bytes) return fail(MLA_ERR_INVALID_ARG, "bytes is NULL");
  if (topk < 1) return fail(MLA_ERR_INVALID_ARG, "topk must be >= 1 (got %d)", topk);
  Geometry g{};
  PrefillLayout L{};
  mla_status st = prefill_layout(s_q, h_q, topk, &g, &L);
  if (st != MLA_OK) return st;
  *bytes = L.total;
  return ok();
}

mla_status mla_sparse_prefill(const mla_sparse_prefill_args* a, mla_stream_t stream) {
  if (!a) return fail(MLA_ERR_INVALID_ARG, "args is NULL");
  if (!a->q) return fail(MLA_ERR_INVALID_ARG, "q is NULL");
  if (!a->kv) return fail(MLA_ERR_INVALID_ARG, "kv is NULL");
  if (!a->indices) return fail(MLA_ERR_INVALID_ARG, "indices is NULL");
  if (!a->out) return fail(MLA_ERR_INVALID_ARG, "out is NULL");
  if (!a->lse) return fail(MLA_ERR_INVALID_ARG, "lse is NULL");
  if (a->s_q < 1) return fail(MLA_ERR_INVALID_ARG, "s_q must be >= 1 (got %d)", a->s_q);
  if (a->s_kv < 1) return fail(MLA_ERR_INVALID_ARG, "s_kv must be >= 1 (got %d)", a->s_kv);
  if (a->topk < 1) return fail(MLA_ERR_INVALID_ARG, "topk must be >= 1 (got %d)", a->topk);
  if (!std::isfinite(a->sm_scale)) return fail(MLA_ERR_INVALID_ARG, "sm_scale is not finite");
  if (!aligned(a->q, 16)) return fail(MLA_ERR_INVALID_ARG, "q is not 16-byte aligned");
  if (!aligned(a->kv, 16)) return fail(MLA_ERR_INVALID_ARG, "kv is not 16-byte aligned");
  if (!aligned(a->out, 16)) return fail(MLA_ERR_INVALID_ARG, "out is not 16-byte aligned");
  if (!aligned(a->lse, 4)) return fail(MLA_ERR_INVALID_ARG, "lse is not 4-byte aligned");
  if (!aligned(a->indices, 4)) return fail(MLA_ERR_INVALID_ARG, "indices is not 4-byte aligned");
  Geometry g{};
  PrefillLayout L{};
  mla_status st = prefill_layout(a->s_q, a->h_q, a->topk, &g, &L);
  if (st != MLA_OK) return st;
  if (!a->workspace) return fail(MLA_ERR_WORKSPACE, "workspace is NULL (%zu bytes needed)", L.total);
  if (a->workspace_bytes < L.total)
    return fail(MLA_ERR_WORKSPACE, "workspace_bytes = %zu < %zu needed", a->workspace_bytes, L.total);
  if (!aligned(a->workspace, 256)) return fail(MLA_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
  uint32_t* status = nullptr;
  st = device_info(&status, nullptr);
  if (st != MLA_OK) return st;

  char* ws = static_cast<char*>(a->workspace);
  int32_t* sched = reinterpret_cast<int32_t*>(ws + L.sched);
  int32_t* num_splits = reinterpret_cast<int32_t*>(ws + L.num_splits);
  CUtensorMap tm_kv;
  st = encode_byte_rows_map(&tm_kv, a->kv, a->s_kv, 2 * kDqk, 1);
  if (st != MLA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint64_t timeout = watchdog_ns();
  for (int c0 = 0; c0 < a->s_q; c0 += kMaxProblems) {
    const int chunk = a->s_q - c0 < kMaxProblems ? a->s_q - c0 : kMaxProblems;
    Geometry gc{};
    st = geometry(1, a->h_q, chunk, a->topk, 0, &gc);
    if (st != MLA_OK) return st;
    const char* q = static_cast<const char*>(a->q) + static_cast<size_t>(c0) * a->h_q * kDqk * 2;
    CUtensorMap tm_q;
    st = gc.pair ? encode_chunk_major_map(&tm_q, q, static_cast<long long>(chunk) * a->h_q, kNumChunks, "q")
                 : encode_rows_map(&tm_q, q, static_cast<long long>(chunk) * a->h_q, gc.rpc, "q");
    if (st != MLA_OK) return st;
    cudaError_t e = launch_metadata(nullptr, chunk, a->topk, gc, sched, num_splits, s);
    if (e != cudaSuccess) return cuda_fail(e, "metadata kernel launch");

    DecodeParams p;
    memset(&p, 0, sizeof p);
    p.indices = a->indices + static_cast<size_t>(c0) * a->topk;
    p.sched = sched;
    p.num_splits = num_splits;
    p.kv_fp8 = static_cast<const uint8_t*>(a->kv);
    p.out = static_cast<char*>(a->out) + static_cast<size_t>(c0) * a->h_q * kDv * 2;
    p.lse = a->lse + static_cast<size_t>(c0) * a->h_q;
    p.o_accum = reinterpret_cast<float*>(ws + L.o_accum);
    p.lse_accum = reinterpret_cast<float*>(ws + L.lse_accum);
    p.status = status;
    p.timeout_ns = timeout;
    p.batch = 1;
    p.s_q = chunk;
    p.h_q = a->h_q;
    p.topk = a->topk;
    p.num_pages = 1;
    p.block_table_stride = 1;
    p.num_problems = gc.num_problems;
    p.rows = gc.rows;
    p.row_groups = gc.row_groups;
    p.num_parts = gc.num_parts;
    p.max_slots = max_slots(gc);
    p.evict_first = (gc.row_groups == 1 && !gc.pair) ? 1 : 0;
    p.sched_tag = gc.tag;
    p.flat_rows = a->s_kv;
    p.scale_log2 = a->sm_scale * 1.4426950408889634f;
    p.fp8_rope_off = 2 * kDv;
    p.rows16 = 1;
    e = gc.pair ? launch_decode_pair(tm_q, tm_q, tm_q, p, true, s) : launch_decode(tm_q, tm_kv, p, gc.rpc, 3, s);
    if (e != cudaSuccess) return cuda_fail(e, "sparse prefill attention kernel launch");
    CombineParams cp;
    cp.num_splits = num_splits;
    cp.cache_seqlens = nullptr;
    cp.s_q = chunk;
    cp.topk = a->topk;
    cp.o_accum = p.o_accum;
    cp.lse_accum = p.lse_accum;
    cp.out = p.out;
    cp.lse = p.lse;
    cp.num_problems = gc.num_problems;
    cp.rows = gc.rows;
    cp.max_slots = p.max_slots;
    cp.status = status;
    e = launch_combine(cp, s, true);
    if (e != cudaSuccess) return cuda_fail(e, "combine kernel launch");
  }
  return ok();
}

mla_status mla_index_topk_workspace_size(int num_tokens, int block_table_stride, size_t* bytes) {
  if (!bytes) return fail(MLA_ERR_INVALID_ARG, "bytes is NULL");
  if (num_tokens < 0) return fail(MLA_ERR_INVALID_ARG, "num_tokens must be >= 0 (got %d)", num_tokens);
  if (block_table_stride < 1)
    return fail(MLA_ERR_INVALID_ARG, "block_table_stride must be >= 1 (got %d)", block_table_stride);
  *bytes = align256(static_cast<size_t>(num_tokens) * block_table_stride * kPageSize * sizeof(float));
  return ok();
}

mla_status mla_index_topk(const mla_index_topk_args* a, mla_stream_t stream) {
  if (!a) return fail(MLA_ERR_INVALID_ARG, "args is NULL");
  if (a->batch < 1) return fail(MLA_ERR_INVALID_ARG, "batch must be >= 1 (got %d)", a->batch);
  if (a->num_tokens < 0) return fail(MLA_ERR_INVALID_ARG, "num_tokens must be >= 0 (got %d)", a->num_tokens);
  if (a->h_idx < 8 || a->h_idx % 8 != 0 || a->h_idx > 256)
    return fail(MLA_ERR_UNSUPPORTED, "h_idx must be a multiple of 8 in [8, 256] (got %d)", a->h_idx);
  if (a->max_new_tokens < 1) return fail(MLA_ERR_INVALID_ARG, "max_new_tokens must be >= 1 (got %d)", a->max_new_tokens);
  if (static_cast<long long>(a->max_new_tokens) * a->h_idx > 256)
    return fail(MLA_ERR_UNSUPPORTED, "max_new_tokens * h_idx = %lld exceeds 256 rows per element",
                static_cast<long long>(a->max_new_tokens) * a->h_idx);
  if (a->topk < 1 || a->topk > 16384) return fail(MLA_ERR_UNSUPPORTED, "topk must be in [1, 16384] (got %d)", a->topk);
  if (a->page_size != kPageSize) return fail(MLA_ERR_UNSUPPORTED, "page_size must be 64 (got %d)", a->page_size);
  if (a->num_pages < 1) return fail(MLA_ERR_INVALID_ARG, "num_pages must be >= 1 (got %d)", a->num_pages);
  if (a->block_table_stride < 1)
    return fail(MLA_ERR_INVALID_ARG, "block_table_stride must be >= 1 (got %d)", a->block_table_stride);
  if (static_cast<long long>(a->block_table_stride) * kPageSize > (1ll << 31) - 1)
    return fail(MLA_ERR_UNSUPPORTED, "block_table_stride = %d exceeds 2^31 keys", a->block_table_stride);
  if (!a->q_codes) return fail(MLA_ERR_INVALID_ARG, "q_codes is NULL");
  if (!a->q_scales) return fail(MLA_ERR_INVALID_ARG, "q_scales is NULL");
  if (!a->weights) return fail(MLA_ERR_INVALID_ARG, "weights is NULL");
  if (!a->row_offsets) return fail(MLA_ERR_INVALID_ARG, "row_offsets is NULL");
  if (!a->k_codes) return fail(MLA_ERR_INVALID_ARG, "k_codes is NULL");
  if (!a->k_scales) return fail(MLA_ERR_INVALID_ARG, "k_scales is NULL");
  if (!a->block_table) return fail(MLA_ERR_INVALID_ARG, "block_table is NULL");
  if (!a->cache_seqlens) return fail(MLA_ERR_INVALID_ARG, "cache_seqlens is NULL");
  if (!a->indices) return fail(MLA_ERR_INVALID_ARG, "indices is NULL");
  if (!aligned(a->q_codes, 16)) return fail(MLA_ERR_INVALID_ARG, "q_codes is not 16-byte aligned");
  if (!aligned(a->k_codes, 16)) return fail(MLA_ERR_INVALID_ARG, "k_codes is not 16-byte aligned");
  size_t need = 0;
  mla_status st = mla_index_topk_workspace_size(a->num_tokens, a->block_table_stride, &need);
  if (st != MLA_OK) return st;
  if (a->num_tokens == 0) return ok();
  if (!a->workspace) return fail(MLA_ERR_WORKSPACE, "workspace is NULL (%zu bytes needed)", need);
  if (a->workspace_bytes < need) return fail(MLA_ERR_WORKSPACE, "workspace_bytes = %zu < %zu needed", a->workspace_bytes, need);
  if (!aligned(a->workspace, 16)) return fail(MLA_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
  uint32_t* status = nullptr;
  st = device_info(&status, nullptr);
  if (st != MLA_OK) return st;

  IndexParams p;
  memset(&p, 0, sizeof p);
  const int rows = a->max_new_tokens * a->h_idx;
  p.n_box = (rows + 15) & ~15;
  uint32_t cols = 32;
  while (cols < static_cast<uint32_t>(p.n_box)) cols <<= 1;
  p.tmem_cols = 2 * cols;
  CUtensorMap tm_q, tm_k;
  st = encode_e4m3_rows_map(&tm_q, a->q_codes, static_cast<long long>(a->num_tokens) * a->h_idx, p.n_box, "q_codes");
  if (st != MLA_OK) return st;
  st = encode_e4m3_rows_map(&tm_k, a->k_codes, static_cast<long long>(a->num_pages) * kPageSize, kPageSize, "k_codes");
  if (st != MLA_OK) return st;
  p.q_scales = a->q_scales;
  p.weights = a->weights;
  p.row_offsets = a->row_offsets;
  p.k_scales = a->k_scales;
  p.block_table = a->block_table;
  p.cache_seqlens = a->cache_seqlens;
  p.scores = static_cast<float*>(a->workspace);
  p.status = status;
  p.timeout_ns = watchdog_ns();
  p.width = static_cast<int64_t>(a->block_table_stride) * kPageSize;
  p.batch = a->batch;
  p.num_tokens = a->num_tokens;
  p.h_idx = a->h_idx;
  p.max_new = a->max_new_tokens;
  p.num_pages = a->num_pages;
  p.block_table_stride = a->block_table_stride;
  p.relu = a->relu ? 1 : 0;
  // key tiles per CTA: the run length that minimises the modelled time when
  // every element has the longest possible length -- whole waves of two CTAs
  // per SM, each costing its tiles plus about three tiles of set-up and
  // pipeline fill (a last, partly filled wave costs as much as a full one)
  {
    int sms = 0;
    st = device_info(nullptr, &sms);
    if (st != MLA_OK) return st;
    const long long max_tiles = (p.width + 127) / 128;
    const long long slots = 2ll * (sms > 0 ? sms : 1);
    long long best_cost = -1, best_tpc = 64;
    for (long long tpc = 4; tpc <= 64; ++tpc) {
      const long long ctas = static_cast<long long>(a->batch) * ((max_tiles + tpc - 1) / tpc);
      const long long waves = (ctas + slots - 1) / slots;
      const long long cost = waves * (tpc + 3);
      if (best_cost < 0 || cost < best_cost) {
        best_cost = cost;
        best_tpc = tpc;
      }
    }
    p.tiles_per_cta = static_cast<int>(best_tpc);
  }
  cudaError_t e = launch_index(tm_q, tm_k, p, a->topk, a->indices, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "indexer kernel launch");
  return ok();
}

mla_status mla_get_device_status(mla_stream_t stream, uint32_t* flags) {
  if (!flags) return fail(MLA_ERR_INVALID_ARG, "flags is NULL");
  uint32_t* status = nullptr;
  mla_status st = device_info(&status, nullptr);
  if (st != MLA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  uint32_t v = 0;
  e = cudaMemcpyAsync(&v, status, sizeof v, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(status, 0, sizeof v, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
  *flags = v;
  if (v & MLA_DEVICE_TIMEOUT) return fail(MLA_ERR_DEVICE_TIMEOUT, "a kernel wait exceeded its limit (status 0x%x)", v);
  if (v & MLA_DEVICE_BAD_PAGE)
    return fail(MLA_ERR_DEVICE_BOUNDS, "a block-table entry was outside [0, num_pages) (status 0x%x)", v);
  if (v & MLA_DEVICE_BAD_SCHEDULE)
    return fail(MLA_ERR_INVALID_ARG, "the schedule did not match the decode arguments (status 0x%x)", v);
  return ok();
}

}  // extern "C"
