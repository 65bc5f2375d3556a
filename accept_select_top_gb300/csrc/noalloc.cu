// noalloc.cu -- spec_verify_greedy_noalloc: greedy accept for callers that
// cannot allocate device memory.
//
// spec_verify_greedy needs a caller-provided workspace (per-request arrival
// counters, the error word, per-chunk argmax partials).  Some callers cannot
// allocate one: code that runs inside an engine whose allocator owns every byte
// of device memory, code on a latency-critical path where cudaMalloc's implicit
// device synchronisation is not acceptable, or plugins whose host forbids
// allocation after start-up.  This entry point uses a fixed scratch array that
// lives in the library's own device image instead.  Every GPU that loads the
// library holds the array (SPEC_NOALLOC_SCRATCH_BYTES) until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "accept_select_top.h"
#include "common.cuh"
#include "kernels.cuh"

namespace {

constexpr size_t kScratchBytes = SPEC_NOALLOC_SCRATCH_BYTES;

// The scratch memory.  In host code this name is only a host-side stand-in for
// the device symbol; kernels are given its device address, looked up below.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device, looked up once per device
// (with that device current) and kept for the life of the process.  The cache
// assumes the device's primary context lives as long as the process: after a
// cudaDeviceReset the module is reloaded and the kept address is stale, so a
// process that resets a device must not call these entry points afterwards.
int scratch_of_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPEC_ERR_LAUNCH;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return SPEC_ERR_LAUNCH;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SPEC_OK;
}

}  // namespace

extern "C" int spec_verify_greedy_noalloc(int b, int n, int S, int V, int dtype, const void* logits,
                                          const int32_t* draft_tokens, const int32_t* retrieve_index,
                                          const int32_t* next_token, const int32_t* next_sibling, int32_t* predict,
                                          int32_t* accept_index, int32_t* accept_lens, int32_t* accepted_tokens,
                                          int32_t* next_root, void* stream) {
  if (b < 0 || n < 1 || n > spec::kMaxN || S < 1 || V < 1) return SPEC_ERR_ARG;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (b == 0) return SPEC_OK;
  // every check that can reject the call comes before anything is enqueued
  if (!logits || !draft_tokens || !retrieve_index || !next_token || !next_sibling || !predict || !accept_index ||
      !accept_lens)
    return SPEC_ERR_ARG;
  const size_t need = spec::greedy_compact_bytes(b, n, V);
  if (need > kScratchBytes) return SPEC_ERR_WORKSPACE;  // too large for the fixed scratch
  void* ws = nullptr;
  if (int rc = scratch_of_current_device(&ws)) return rc;
  // The array keeps the previous call's contents.  The arrival counters must
  // start at zero (a call that completes leaves them zero; this also clears
  // what an interrupted call left).  The error word is not cleared: device
  // index errors accumulate until spec_noalloc_last_error reads them.  The
  // partials are always written before they are read.
  unsigned char* counters = static_cast<unsigned char*>(ws) + spec::kHeaderBytes;
  if (cudaMemsetAsync(counters, 0, spec::counters_bytes(b), static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SPEC_ERR_LAUNCH;
  return spec::verify_greedy_compact(b, n, S, V, dtype, logits, draft_tokens, retrieve_index, next_token,
                                     next_sibling, predict, accept_index, accept_lens, accepted_tokens, next_root,
                                     ws, kScratchBytes, stream);
}

extern "C" int spec_noalloc_last_error(void* stream) {
  void* ws = nullptr;
  if (int rc = scratch_of_current_device(&ws)) return rc;
  // the error word is the first word of the array, as in a caller workspace
  return spec_last_error(ws, stream);
}
