// common.cuh -- device helpers shared by the verify/accept kernels (sm_103a).
//
// Workspace layout (all offsets 256-byte aligned):
//   [0, 256)                 header: uint32 error word at offset 0
//   [256, 256 + counters)    uint32 per-request arrival counters (zero between calls)
//   [.., ..)                 per-operation partial results
// A kernel that splits a row over several CTAs writes its partial result, then
// the CTA that arrives last for a request (atomic counter) merges the partials
// and finishes the request, and puts the counter back to zero.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <climits>
#include <cmath>

#include "accept_select_top.h"

namespace spec {

constexpr int kThreads = 256;       // threads of every row-scan CTA
constexpr int kTargetCtas = 608;    // 152 SMs x 4 resident CTAs: the grid size a vocab scan aims for
constexpr int kMaxChunks = 32;      // row splits per row
constexpr int kMaxK = 16;           // largest topk
constexpr int kMaxN = 64;           // largest tree (one uint64 mask word per row)

constexpr size_t kHeaderBytes = 256;

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

__host__ __device__ inline size_t counters_bytes(int b) { return align256(size_t(b + 1) * 4); }

struct WsView {
  uint32_t* error;
  uint32_t* counters;
  unsigned char* partials;
};

inline WsView ws_view(void* ws, int b) {
  unsigned char* base = static_cast<unsigned char*>(ws);
  return WsView{reinterpret_cast<uint32_t*>(base), reinterpret_cast<uint32_t*>(base + kHeaderBytes),
                base + kHeaderBytes + counters_bytes(b)};
}

__device__ inline void raise_error(uint32_t* err, uint32_t bit) { atomicOr(err, bit); }

// a ranks before b: larger value, or equal value and smaller index
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <typename T>
struct LogitTraits;
template <>
struct LogitTraits<float> {
  static constexpr int kVec = 4;  // elements per 16-byte load
  __device__ static float load(const float* p, size_t i) { return __ldg(p + i); }
  __device__ static void unpack(const uint4& x, float (&f)[4]) {
    f[0] = __uint_as_float(x.x);
    f[1] = __uint_as_float(x.y);
    f[2] = __uint_as_float(x.z);
    f[3] = __uint_as_float(x.w);
  }
};
template <>
struct LogitTraits<uint16_t> {  // bf16 bit patterns
  static constexpr int kVec = 8;
  __device__ static float load(const uint16_t* p, size_t i) {
    return __uint_as_float(uint32_t(__ldg(p + i)) << 16);
  }
  __device__ static void unpack(const uint4& x, float (&f)[8]) {
    f[0] = bf16_lo(x.x); f[1] = bf16_hi(x.x);
    f[2] = bf16_lo(x.y); f[3] = bf16_hi(x.y);
    f[4] = bf16_lo(x.z); f[5] = bf16_hi(x.z);
    f[6] = bf16_lo(x.w); f[7] = bf16_hi(x.w);
  }
};

// Streaming 16-byte load: the logits are read once per step.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) { return __ldcs(p); }

// (value, index) argmax across a warp; every lane ends with the winner.
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float ov = __shfl_xor_sync(0xffffffffu, v, o);
    int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (better(ov, oi, v, i)) {
      v = ov;
      i = oi;
    }
  }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Returns true in every thread of the CTA that arrives last among `total` CTAs
// sharing `counter`.  Call after the CTA's partial result is written.  The last
// CTA must reset the counter (counter_reset) once it is done.
__device__ __forceinline__ bool arrive_last(uint32_t* counter, uint32_t total) {
  __shared__ int s_last;
  __threadfence();  // every thread's partial writes are ordered before the arrival
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t prev = atomicAdd(counter, 1u);
    s_last = prev == total - 1;
  }
  __syncthreads();
  if (s_last) __threadfence();
  return s_last;
}

__device__ __forceinline__ void counter_reset(uint32_t* counter) {
  if (threadIdx.x == 0) atomicExch(counter, 0u);
}

// How a row of V logits is split over CTAs.
struct RowSplit {
  int chunks;
  int chunk_elems;
};

inline RowSplit pick_split(long rows, int V, int vec, int max_chunks = kMaxChunks) {
  long want = (kTargetCtas + rows - 1) / rows;
  if (want < 1) want = 1;
  if (want > max_chunks) want = max_chunks;
  long by_size = V / 2048;  // at least ~2K elements per chunk
  if (by_size < 1) by_size = 1;
  if (want > by_size) want = by_size;
  int per = int((V + want - 1) / want);
  per = (per + vec - 1) / vec * vec;
  int chunks = (V + per - 1) / per;
  return RowSplit{chunks, per};
}

// The split select_topk uses: as pick_split, but never more than 8192 logits
// (32 per thread) per CTA, so a thread's share of a chunk fits in registers.
// More than kMaxChunks chunks (a vocabulary above 262144) is not supported.
constexpr int kSelectChunkMax = kThreads * 32;

inline RowSplit select_split(long rows, int V, int vec) {
  long want = (kTargetCtas + rows - 1) / rows;
  if (want < 1) want = 1;
  if (want > kMaxChunks) want = kMaxChunks;
  long by_size = V / 2048;
  if (by_size < 1) by_size = 1;
  if (want > by_size) want = by_size;
  const long need = (long(V) + kSelectChunkMax - 1) / kSelectChunkMax;
  if (want < need) want = need;
  int per = int((V + want - 1) / want);
  per = (per + vec - 1) / vec * vec;
  return RowSplit{(V + per - 1) / per, per};
}

}  // namespace spec
