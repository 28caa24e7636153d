// mla_decode_noalloc — decode for callers that cannot allocate device memory.
//
// Some callers have no way to obtain device scratch at the point where they
// decode: code running inside an allocator-less runtime or plugin host that
// owns no CUDA memory pool, or a real-time path where a cudaMalloc (which
// can synchronise the device and take unbounded time) is not allowed.  For
// them this entry point takes the split-KV scratch from a fixed array that
// lives in this library's device image instead of from a caller buffer.  The
// caller still passes every input and output buffer.
//
// Limits and behaviour:
//   * The scratch holds kNoallocScratchBytes (32 MiB).  A decode whose split
//     partials need more (see mla_workspace_size) is rejected with
//     MLA_ERR_WORKSPACE before anything is launched.
//   * Every GPU that loads this part of the library keeps the 32 MiB until
//     the process exits.
//   * The first call on a device looks up the array's device address (once
//     per device, with that device current); make that first call before any
//     stream capture.
//   * All calls share the one array and it keeps whatever the last call left
//     there.  Nothing in it needs to start at zero: every partial slot the
//     combine step reads is written earlier in the same call.  Two calls whose
//     work overlaps on the GPU (different streams, or different host threads
//     on one device) race on the array and corrupt each other's partials;
//     serialise them.
//   * args->workspace and args->workspace_bytes are ignored.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "mla_internal.h"

namespace mla {
namespace {

constexpr size_t kNoallocScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxNoallocDevices = 64;
void* g_noalloc_ptr[kMaxNoallocDevices];
std::mutex g_noalloc_mu;

// Device address of the scratch array on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxNoallocDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace mla

extern "C" mla_status mla_decode_noalloc(const mla_decode_args* args, mla_stream_t stream) {
  using namespace mla;
  if (!args) return mla_decode(args, stream);  // same argument error as the allocating entry point
  size_t need = 0;
  mla_status st = mla_workspace_size(args->batch, args->h_q, args->s_q, args->topk, args->is_fp8, &need);
  if (st != MLA_OK) return st;
  if (need > kNoallocScratchBytes) {
    set_error_message("mla_decode_noalloc: this decode needs " + std::to_string(need) +
                      " bytes of split-KV scratch, more than the fixed " + std::to_string(kNoallocScratchBytes) +
                      "-byte device scratch; use mla_decode with a caller workspace");
    return MLA_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) {
    set_error_message(std::string("mla_decode_noalloc: cudaGetSymbolAddress failed: ") + cudaGetErrorString(e));
    return MLA_ERR_CUDA;
  }
  mla_decode_args a = *args;
  a.workspace = scratch;
  a.workspace_bytes = kNoallocScratchBytes;
  return mla_decode(&a, stream);
}
