// Allocation-free entry point.
//
// Some callers cannot allocate device memory when they need the scores: a
// serving loop that reserves all device memory up front and forbids allocator
// calls on its hot path, or a host program that embeds this library through
// its C ABI without any device allocator of its own (no torch, no memory
// pool).  Such callers cannot provide the workspace that msa_index_score asks
// for, so this variant keeps the plan scratch in a fixed array that lives in
// the library itself.
//
// The array is a file-scope __device__ object of MSA_NOALLOC_WORKSPACE_BYTES
// bytes: every GPU that loads the library holds it until the process exits.
// In host code the array's name is only a host-side stand-in, so its device
// address is looked up with cudaGetSymbolAddress with the device current and
// cached per device, together with the id of the CUDA context it was looked
// up in: after a device reset, or in another context on the same device, the
// module is loaded afresh and the address is looked up again.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "msa_index_score.h"
#include "msa_common.cuh"

namespace {

constexpr size_t kScratchBytes = msa::workspace_bytes_for(MSA_NOALLOC_MAX_BATCH);
static_assert(kScratchBytes == MSA_NOALLOC_WORKSPACE_BYTES, "header constant out of date");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
struct Resolved {
  uint64_t ctx;   // context id the address belongs to (0: none yet)
  void* addr;
};
std::mutex g_mu;
Resolved g_scratch[kMaxDevices] = {};

msa_status_t cuda_error(cudaError_t e, const char* what) {
  char msg[256];
  snprintf(msg, sizeof msg, "%s: %s", what, cudaGetErrorString(e));
  msa::set_last_error_message(msg);
  return MSA_ERR_CUDA;
}

// Device address of the scratch array in the current device's context.
msa_status_t scratch_address(void** addr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) {
    msa::set_last_error_message("device ordinal beyond the no-alloc entry point's table");
    return MSA_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  const uint64_t ctx = msa::current_context_id();
  if (ctx == 0 || g_scratch[dev].ctx != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return cuda_error(e, "cudaGetSymbolAddress(no-alloc scratch)");
    // the lookup makes the device's primary context current if none was
    g_scratch[dev].ctx = msa::current_context_id();
    g_scratch[dev].addr = p;
  }
  *addr = g_scratch[dev].addr;
  return MSA_OK;
}

}  // namespace

extern "C" msa_status_t msa_index_score_noalloc(const msa_index_score_args* args, float* out,
                                                msa_stream_t stream) {
  if (!args) {
    msa::set_last_error_message("args is NULL");
    return MSA_ERR_INVALID_ARG;
  }
  if (args->B > MSA_NOALLOC_MAX_BATCH) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "msa_index_score_noalloc handles at most %d requests (got B = %d); use "
             "msa_index_score with a caller workspace",
             MSA_NOALLOC_MAX_BATCH, (int)args->B);
    msa::set_last_error_message(msg);
    return MSA_ERR_WORKSPACE;
  }
  void* ws = nullptr;
  msa_status_t st = scratch_address(&ws);
  if (st != MSA_OK) return st;
  return msa_index_score(args, out, ws, kScratchBytes, stream);
}

extern "C" msa_status_t msa_noalloc_device_error(int32_t* bits, msa_stream_t stream) {
  if (!bits) {
    msa::set_last_error_message("bits is NULL");
    return MSA_ERR_INVALID_ARG;
  }
  void* ws = nullptr;
  msa_status_t st = scratch_address(&ws);
  if (st != MSA_OK) return st;
  return msa_get_device_error(ws, bits, stream);
}
