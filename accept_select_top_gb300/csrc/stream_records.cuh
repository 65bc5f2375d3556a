// stream_records.cuh -- the logits streaming pass shared by the select and
// the sampling accept, and the device helpers their request steps use.
//
// One pass over the flattened [rows, V] logits (16-byte vectors, rows
// contiguous), cut into units of 256 vectors (4 KB).  Every warp of a
// persistent grid (two CTAs a SM) works on its own: it takes units in chunks
// of 2 to 16 consecutive ones (about four chunks a warp), the first two
// chunks fixed by its index, the rest from a queue (an atomic counter, asked
// two chunks ahead so that its latency stays hidden), so that warps the memory
// serves faster take more.  Lane l holds vectors l, l + 32,
// ..., l + 224 of a unit in a private ring of 16-byte cp.async copies, three
// units deep, and waits for its own copies with cp.async.wait_group: no barrier
// and no wait on another warp.  A lane's vectors of one unit inside one row
// form a group; for each group it writes one record: the group's maximum g and
// s = sum over the group of 2^((x - g) c), c = log2(e) / T of the row (s = -1
// where the lane has no vector in that row of the unit; s = 1 in a greedy
// row, T = 0, which needs no sum).  A unit spans at most two rows, so the record slot
// is (unit, row parity, lane).
//
// From a row's records: the row maximum is the largest g, the softmax
// denominator sum of s 2^((g - M) c); and the row's k best elements lie in its
// k best groups by (maximum desc, index of the maximum asc) -- were an element
// among the k best in a group outside them, the k groups ahead of its group
// would each hold an element that ranks before it.
#pragma once

#include "common.cuh"
#include "kernels.cuh"

namespace spec {

constexpr int kStreamThreads = 256;
constexpr int kStreamWarps = kStreamThreads / 32;
constexpr int kStreamPerSm = 2;                   // CTAs a SM (the ring and the registers allow two)
constexpr int kStreamStages = 3;                  // units in flight a lane
constexpr int kStreamVpt = 8;                     // 16-byte vectors a lane holds of a unit
constexpr int kUnitVecs = kStreamVpt * 32;        // vectors a unit
constexpr int kStreamCand = 32;                   // candidate elements a warp buffers (one a lane)

// 16-byte global -> shared copy; src_bytes 0 writes zeros and reads nothing.
__device__ __forceinline__ void stream_cp16(void* dst, const void* src, uint32_t src_bytes) {
  const uint32_t d = uint32_t(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void stream_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void stream_wait_group() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Element q (0 <= q < E, a runtime value) of a 16-byte vector, by selects.
template <typename T>
__device__ __forceinline__ float vec_elem(const uint4& x, int q) {
  if constexpr (sizeof(T) == 2) {
    const uint32_t w = q < 4 ? (q < 2 ? x.x : x.y) : (q < 6 ? x.z : x.w);
    return (q & 1) ? bf16_hi(w) : bf16_lo(w);
  } else {
    return __uint_as_float(q < 2 ? (q == 0 ? x.x : x.y) : (q == 2 ? x.z : x.w));
  }
}

// A warp's k best so far (lane j < k holds entry j, best first; the other
// lanes hold nothing) merged with the buffered candidates (lane l < ncand
// holds buffer entry l): k rounds of a warp argmax over each lane's two
// entries.  Element indices are unique within a row, so a winner is removed
// by its index.
__device__ __forceinline__ void stream_merge_candidates(const float* bv_s, const int* bi_s, int ncand, int k,
                                                        float& lv_r, int& li_r) {
  const int lane = threadIdx.x & 31;
  __syncwarp();  // the lanes' appends are visible
  float cv = lane < ncand ? bv_s[lane] : -INFINITY;
  int ci = lane < ncand ? bi_s[lane] : INT_MAX;
  float ev = lv_r;
  int ei = li_r;
  float nv = -INFINITY;
  int ni = INT_MAX;
  for (int j = 0; j < k; ++j) {
    const bool c_first = better(cv, ci, ev, ei);
    float bv = c_first ? cv : ev;
    int bi = c_first ? ci : ei;
    warp_argmax(bv, bi);
    if (ci == bi) {
      cv = -INFINITY;
      ci = INT_MAX;
    }
    if (ei == bi) {
      ev = -INFINITY;
      ei = INT_MAX;
    }
    if (lane == j) {
      nv = bv;
      ni = bi;
    }
  }
  lv_r = nv;
  li_r = ni;
  __syncwarp();  // every lane has read the buffer before it is refilled
}

// Two fp32 lanes in one 64-bit register: the packed FMA and add of sm_100
// and later (each lane rounded as the scalar instruction rounds it).
__device__ __forceinline__ unsigned long long f2_pack(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(unsigned long long r) {
  float2 v;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
  return v;
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b, unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// Per-vector maxima kept packed where the type allows it (bf16x2: both halves
// of a vector's maximum), combined into the batch maximum; value() gives the
// fp32 maximum.
template <typename T>
struct VecMax;
template <>
struct VecMax<uint16_t> {
  using type = __nv_bfloat162;
  __device__ static type of(const uint4& x) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&x);
    return __hmax2(__hmax2(h[0], h[1]), __hmax2(h[2], h[3]));
  }
  __device__ static type comb(type a, type b) { return __hmax2(a, b); }
  __device__ static float value(type a) { return fmaxf(__low2float(a), __high2float(a)); }
};
template <>
struct VecMax<float> {
  using type = float;
  __device__ static type of(const uint4& x) {
    return fmaxf(fmaxf(__uint_as_float(x.x), __uint_as_float(x.y)), fmaxf(__uint_as_float(x.z), __uint_as_float(x.w)));
  }
  __device__ static type comb(type a, type b) { return fmaxf(a, b); }
  __device__ static float value(type a) { return a; }
};

// Sum over the batch of 2^(x c - mc), two lanes at a time (packed FMA and
// add, one ex2 an element).
template <typename T>
__device__ __forceinline__ float batch_exp_sum(const uint4 (&x)[kStreamVpt], float c, float mc) {
  const unsigned long long c2 = f2_pack(c, c), nm2 = f2_pack(-mc, -mc);
  unsigned long long acc = f2_pack(0.f, 0.f);
#pragma unroll
  for (int u = 0; u < kStreamVpt; ++u) {
    const uint32_t wd[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
    if constexpr (sizeof(T) == 2) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 t = f2_unpack(f2_fma(f2_pack(bf16_lo(wd[j]), bf16_hi(wd[j])), c2, nm2));
        acc = f2_add(acc, f2_pack(fast_exp2(t.x), fast_exp2(t.y)));
      }
    } else {
#pragma unroll
      for (int j = 0; j < 4; j += 2) {
        const float2 t = f2_unpack(f2_fma(f2_pack(__uint_as_float(wd[j]), __uint_as_float(wd[j + 1])), c2, nm2));
        acc = f2_add(acc, f2_pack(fast_exp2(t.x), fast_exp2(t.y)));
      }
    }
  }
  const float2 s = f2_unpack(acc);
  return s.x + s.y;
}

// The record slot of (unit, row parity, lane).
__device__ __forceinline__ int stream_slot(int unit, int parity, int lane) { return (unit * 2 + parity) * 32 + lane; }

// The records of row `row` (of rows of rowU vectors): flat index f = (unit -
// first unit) * 32 + lane over the units the row touches.
struct RowRecords {
  int uf, F, par;
  long long rs, rend;  // the row's vectors
  __device__ __forceinline__ RowRecords(int row, long long rowU) {
    rs = (long long)row * rowU;
    rend = rs + rowU;
    uf = int(rs / kUnitVecs);
    F = (int((rend - 1) / kUnitVecs) - uf + 1) * 32;
    par = row & 1;
  }
  __device__ __forceinline__ int slot(int f) const { return stream_slot(uf + f / 32, par, f % 32); }
  // the first vector of group f (its vectors: + 32 u, those inside [rs, rend))
  __device__ __forceinline__ long long first_vec(int f) const { return (long long)(uf + f / 32) * kUnitVecs + f % 32; }
};

// Maximum / sum over a CTA of `nw` warps (scratch: a slot a warp); every
// thread gets the result.  Both end with a barrier, so the scratch may be
// reused.
__device__ __forceinline__ float block_max_f(float v, float* scratch, int nw) {
  v = warp_max(v);
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = scratch[0];
  for (int i = 1; i < nw; ++i) r = fmaxf(r, scratch[i]);
  __syncthreads();
  return r;
}
__device__ __forceinline__ float block_sum_f(float v, float* scratch, int nw) {
  v = warp_sum(v);
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = 0.f;
  for (int i = 0; i < nw; ++i) r += scratch[i];
  __syncthreads();
  return r;
}

}  // namespace spec
