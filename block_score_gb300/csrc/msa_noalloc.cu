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
// address is looked up with cudaGetSymbolAddress on the first call on each
// device (with that device current) and cached.
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
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (first use per
// device resolves it while that device is current).
msa_status_t scratch_address(void** addr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof msg, "cudaGetDevice: %s", cudaGetErrorString(e));
    msa::set_last_error_message(msg);
    return MSA_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    msa::set_last_error_message("device ordinal beyond the no-alloc entry point's table");
    return MSA_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      char msg[256];
      snprintf(msg, sizeof msg, "cudaGetSymbolAddress(no-alloc scratch): %s",
               cudaGetErrorString(e));
      msa::set_last_error_message(msg);
      return MSA_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
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
