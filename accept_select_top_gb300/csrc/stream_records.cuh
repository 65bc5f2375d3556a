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
// is (unit, row parity, lane).  On request the warp also writes a unit
// summary a row it touches: over the unit's groups of that row, the maximum gu
// and the sum of s 2^((g - gu) c) (a warp maximum and a warp sum); a caller
// that needs only those writes no records.
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

// The L2 policy of the streaming reads: every logit is read once, so its
// lines go first, and what later steps read again (records, summaries, the
// rows a request step or a terminal pass reloads) stays longer.
__device__ __forceinline__ unsigned long long stream_read_policy() {
  unsigned long long pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 16-byte global -> shared copy under L2 policy pol; src_bytes 0 writes zeros
// and reads nothing.
__device__ __forceinline__ void stream_cp16(void* dst, const void* src, uint32_t src_bytes, unsigned long long pol) {
  const uint32_t d = uint32_t(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(d), "l"(src), "r"(src_bytes),
               "l"(pol)
               : "memory");
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

// c = log2(e) / T as an unevaluated sum hi + lo, so that d * c for an exact
// difference d = x - g rounds about once: the exponents of a row's terms
// then carry no error proportional to the row maximum or to c's own
// rounding, which over a 128K vocabulary would reach 1e-6 of the softmax
// denominator.  Formed in fp32: log2(e) = E_HI + E_LO (two floats), hi =
// E_HI / T rounded toward zero, its remainder E_HI - hi T exact by one FMA,
// lo = (remainder + E_LO) / T.  hi <= c, so lo > 0: d = -inf then gives
// -inf, not -inf + inf.
struct ExpScale {
  float hi, lo;
  __device__ __forceinline__ ExpScale() : hi(0.f), lo(0.f) {}
  __device__ __forceinline__ explicit ExpScale(float T) {
    constexpr float kE_HI = 1.44269502162933349609375f;  // log2(e) rounded to fp32
    constexpr float kE_LO = 1.9259629911e-08f;           // log2(e) - kE_HI
    hi = __fdiv_rz(kE_HI, T);
    const float rem = fmaf(-hi, T, kE_HI);
    lo = __fdiv_rn(rem + kE_LO, T);
  }
  __device__ __forceinline__ float times(float d) const { return fmaf(d, hi, d * lo); }
};

__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// Sum over the batch of 2^((x - g) c), two lanes at a time: x - g (exact for
// bf16 values), times c as hi + lo, one ex2 an element, and the 64 (32) terms
// added as a tree (depth 6), so that no long chain of roundings builds up.
template <typename T>
__device__ __forceinline__ float batch_exp_sum(const uint4 (&x)[kStreamVpt], const ExpScale& sc, float g) {
  const unsigned long long hi2 = f2_pack(sc.hi, sc.hi), lo2 = f2_pack(sc.lo, sc.lo), ng2 = f2_pack(-g, -g);
  auto term = [&](float a, float b) {
    const unsigned long long d = f2_add(f2_pack(a, b), ng2);
    const float2 tt = f2_unpack(f2_fma(d, hi2, f2_mul(d, lo2)));
    return f2_pack(fast_exp2(tt.x), fast_exp2(tt.y));
  };
  unsigned long long vs[kStreamVpt];
#pragma unroll
  for (int u = 0; u < kStreamVpt; ++u) {
    if constexpr (sizeof(T) == 2) {
      const unsigned long long e0 = term(bf16_lo(x[u].x), bf16_hi(x[u].x)), e1 = term(bf16_lo(x[u].y), bf16_hi(x[u].y));
      const unsigned long long e2 = term(bf16_lo(x[u].z), bf16_hi(x[u].z)), e3 = term(bf16_lo(x[u].w), bf16_hi(x[u].w));
      vs[u] = f2_add(f2_add(e0, e1), f2_add(e2, e3));
    } else {
      vs[u] = f2_add(term(__uint_as_float(x[u].x), __uint_as_float(x[u].y)),
                     term(__uint_as_float(x[u].z), __uint_as_float(x[u].w)));
    }
  }
#pragma unroll
  for (int w = kStreamVpt / 2; w > 0; w >>= 1)
#pragma unroll
    for (int u = 0; u < w; ++u) vs[u] = f2_add(vs[u], vs[u + w]);
  const float2 s = f2_unpack(vs[0]);
  return s.x + s.y;
}

// The record slot of (unit, row parity, lane).
__device__ __forceinline__ int stream_slot(int unit, int parity, int lane) { return (unit * 2 + parity) * 32 + lane; }

// A thread's running maximum m of records (g, s) and its sum relative to it,
// sum of s 2^((g - m) c), compensated (Kahan) and rescaled when m grows.
struct RecSum {
  float m = -INFINITY, sum = 0.f, comp = 0.f;
  __device__ __forceinline__ void add_term(float v) {
    const float y = v - comp;
    const float t = sum + y;
    comp = (t - sum) - y;
    sum = t;
  }
  __device__ __forceinline__ void add(float g, float s, const ExpScale& sc) {
    if (g > m) {
      const float f = m > -INFINITY ? fast_exp2(sc.times(m - g)) : 0.f;
      sum *= f;
      comp *= f;
      m = g;
      add_term(s);
    } else {
      add_term(s * fast_exp2(sc.times(g - m)));
    }
  }
  // the sum relative to M (>= m)
  __device__ __forceinline__ float rel(float M, const ExpScale& sc) const {
    return sum > 0.f ? (sum - comp) * fast_exp2(sc.times(m - M)) : 0.f;
  }
};

}  // namespace spec
