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

#include <cuda_bf16.h>

#include "accept_select_top.h"

namespace spec {

constexpr int kThreads = 256;       // threads of every row-scan CTA
constexpr int kTargetCtas = 608;    // 152 SMs x 4 resident CTAs: the grid size a vocab scan aims for
constexpr int kMaxChunks = 32;      // row splits per row
constexpr int kMaxK = 16;           // largest topk
constexpr int kMaxN = 64;           // largest tree (one uint64 mask word per row)

constexpr size_t kHeaderBytes = 256;

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// at least 256 words: the attention merge counts arrivals per CTA (<= 192)
// Arrival counters: words [0, max(256, 2b+3)) serve every call (the
// attention's merge counters take up to 256; the select's two halves take 2b
// request counters from word 1 and one unit queue each at 2b+1 and 2b+2);
// greedy accept counts at greedy_counter_base(b) + request, a range no other
// call uses, so that its scan may overlap the attention before it; the word
// after them is the sampling accept's unit queue.
__host__ __device__ inline size_t greedy_counter_base(int b) { return size_t(2 * b + 3 > 256 ? 2 * b + 3 : 256); }
__host__ __device__ inline size_t sampling_queue_word(int b) { return greedy_counter_base(b) + size_t(b); }
__host__ __device__ inline size_t counters_bytes(int b) { return align256((sampling_queue_word(b) + 1) * 4); }

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

// Order-preserving key of a float for the unsigned warp reductions: a larger
// key is a larger value; -0 counts as +0 (they compare equal) and NaN ranks
// below everything.
__device__ __forceinline__ uint32_t order_key(float v) {
  v = v + 0.0f;  // -0 -> +0
  const uint32_t b = __float_as_uint(v);
  if (v != v) return 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// (value, index) argmax across a warp, in the order of better(); every lane
// ends with the winner.  Two warp reductions (redux.sync): the largest key,
// then the smallest index among the lanes that hold it.
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
  const uint32_t key = order_key(v);
  const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
  const uint32_t imin = __reduce_min_sync(0xffffffffu, key == kmax ? uint32_t(i) : 0xffffffffu);
  v = key_value(kmax);
  i = int(imin);
}
// Programmatic dependent launch.  Every kernel of the library is launched
// with programmatic stream serialisation (launch_pdl).  A kernel waits for the
// grid before it -- its completion and its memory -- before reading anything
// (pdl_wait), and only then lets the grid after it be scheduled
// (pdl_trigger).  So only a kernel's prologue overlaps the kernel before it.
// Two kernels may do work before their wait, and only when the caller has
// allowed overlap on the workspace: the select's chunk pass when the kernel
// before it is the previous select (the two use different halves of the
// select's area) or the KV commit on the same workspace, and greedy accept's
// scan when the kernel before it is the verify attention.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// 2^x by the hardware approximation: relative error about 2^-22, results
// below 2^-126 flushed to zero.  For sums of exponentials whose total is at
// least 1 (a softmax denominator), far below fp32's own accumulated rounding.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float warp_max(float v) {
  return key_value(__reduce_max_sync(0xffffffffu, order_key(v)));
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
// counter += 1 with acquire-release order at GPU scope; returns the old value
__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t* counter) {
  uint32_t prev;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(prev) : "l"(counter) : "memory");
  return prev;
}
__device__ __forceinline__ bool arrive_last(uint32_t* counter, uint32_t total) {
  __shared__ int s_last;
  // The barrier orders every thread's partial writes before thread 0's
  // arrival, an acquire-release atomic at GPU scope: the CTA that sees the
  // count complete also sees every other CTA's partials (read after the
  // second barrier).
  __syncthreads();
  if (threadIdx.x == 0) s_last = atom_add_acq_rel(counter) == total - 1;
  __syncthreads();
  return s_last;
}

__device__ __forceinline__ void counter_reset(uint32_t* counter) {
  if (threadIdx.x == 0) atomicExch(counter, 0u);
}

// Batches of a row chunk row[begin, end).  In each batch every thread holds
// U = 32 / E raw 16-byte vectors (vector v of the batch = v0 + tid + u *
// blockDim, E logits each) in registers; fn(x, v0) is called once per batch
// with absent vectors filled with -inf.  Logit (u, e) of the batch has index
// (v0 + tid + u * blockDim) * E + e, so each thread sees its logits in
// increasing index order.  Used only when rows are 16-byte aligned.
constexpr int kBatch = 32;

template <typename T>
struct VecOps;
template <>
struct VecOps<uint16_t> {
  static constexpr int E = 8;
  __device__ static uint4 neg_inf() { return make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u); }
  // maximum of the 8 bf16 values (packed bf16x2 max)
  __device__ static float vmax(const uint4& x) {
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&x.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&x.y);
    const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&x.z);
    const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&x.w);
    const __nv_bfloat162 m = __hmax2(__hmax2(a, b), __hmax2(c, d));
    return fmaxf(__low2float(m), __high2float(m));
  }
  __device__ static float at(const uint4& x, int e) {
    const uint32_t w = e < 2 ? x.x : e < 4 ? x.y : e < 6 ? x.z : x.w;
    return (e & 1) ? bf16_hi(w) : bf16_lo(w);
  }
};
template <>
struct VecOps<float> {
  static constexpr int E = 4;
  __device__ static uint4 neg_inf() {
    const uint32_t n = 0xFF800000u;
    return make_uint4(n, n, n, n);
  }
  __device__ static float vmax(const uint4& x) {
    return fmaxf(fmaxf(__uint_as_float(x.x), __uint_as_float(x.y)), fmaxf(__uint_as_float(x.z), __uint_as_float(x.w)));
  }
  __device__ static float at(const uint4& x, int e) {
    return __uint_as_float(e == 0 ? x.x : e == 1 ? x.y : e == 2 ? x.z : x.w);
  }
};

template <typename T, typename Fn>
__device__ __forceinline__ void for_each_vec_batch(const T* row, int begin, int end, Fn&& fn) {
  constexpr int E = VecOps<T>::E;
  constexpr int U = kBatch / E;
  const int nt = blockDim.x, tid = threadIdx.x;
  const uint4* p = reinterpret_cast<const uint4*>(row);
  const int ve = end / E;
  for (int v0 = begin / E; v0 < ve; v0 += U * nt) {
    uint4 x[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + tid + u * nt;
      x[u] = v < ve ? ld_stream(p + v) : VecOps<T>::neg_inf();
    }
    fn(x, v0);
  }
}

// Argmax (lowest index among equals) of this thread's logits of
// row[begin, end), plus an online softmax when `soft` (running max m and
// sum s of exp2((x - m) * c)), rescaled once per batch.
template <typename T>
__device__ __forceinline__ void scan_row_stats(const T* row, int begin, int end, bool vec, bool soft, float c,
                                               float& bv, int& bi, float& m, float& s) {
  using Tr = LogitTraits<T>;
  constexpr int E = VecOps<T>::E;
  constexpr int U = kBatch / E;
  if (vec) {
    const int nt = blockDim.x;
    for_each_vec_batch<T>(row, begin, end, [&](const uint4 (&x)[U], int v0) {
      float bm = VecOps<T>::vmax(x[0]);
#pragma unroll
      for (int u = 1; u < U; ++u) bm = fmaxf(bm, VecOps<T>::vmax(x[u]));
      if (bm > bv || (bm == bv && bi == INT_MAX)) {
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const float f = VecOps<T>::at(x[u], e);
            const int i = (v0 + int(threadIdx.x) + u * nt) * E + e;
            if (better(f, i, bv, bi)) {
              bv = f;
              bi = i;
            }
          }
      }
      if (soft) {
        const float mb = fmaxf(m, bm);
        float sb = 0.f;
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int e = 0; e < E; ++e) sb += fast_exp2((VecOps<T>::at(x[u], e) - mb) * c);
        s = s * exp2f((m - mb) * c) + sb;
        m = mb;
      }
    });
  } else {
    for (int i = begin + threadIdx.x; i < end; i += blockDim.x) {
      const float f = Tr::load(row, i);
      if (better(f, i, bv, bi)) {
        bv = f;
        bi = i;
      }
      if (soft) {
        if (f > m) {
          s *= exp2f((m - f) * c);
          m = f;
        }
        s += fast_exp2((f - m) * c);
      }
    }
  }
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

// The split greedy accept uses: one wave of 8 CTAs of 256 threads per SM
// (a 32-register kernel), so that a thread's share of a chunk is about one
// batch of 16-byte loads in flight (one round trip instead of two).
inline RowSplit greedy_split(long rows, int V, int vec) {
  long want = (2 * kTargetCtas) / rows;
  if (want < 1) want = 1;
  if (want > kMaxChunks) want = kMaxChunks;
  long by_size = V / 2048;
  if (by_size < 1) by_size = 1;
  if (want > by_size) want = by_size;
  int per = int((V + want - 1) / want);
  per = (per + vec - 1) / vec * vec;
  return RowSplit{(V + per - 1) / per, per};
}

// The split of the terminal row in the second sampling pass: fixed
// 4096-token chunks (16 tokens per thread of a 256-thread CTA, so the
// in-order search of one chunk is a single pass); at most kMaxChunks2 chunks.
constexpr int kMaxChunks2 = 64;
inline RowSplit terminal_split(int V) {
  const int per = V < 4096 ? V : 4096;
  return RowSplit{(V + per - 1) / per, per};
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
