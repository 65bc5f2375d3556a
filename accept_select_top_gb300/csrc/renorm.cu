// renorm.cu -- the relaxed penalties and the top-k / top-p renormalisation of
// the target distribution, before the accept.
//
// [SGL-XI eagle_sample 的骨架: acc_additive_penalties repeated over
// draft_token_num and added to the verify logits (the relaxed penalties)],
// [SGL-XI 路径三 and ACCEPT section 4: the target softmax by temperature, then
// top-k, then top-p, then renormalisation; that distribution is what the
// accept consumes].
//
// add_penalties: one pass over the logits (16-byte vectors), the request's
// penalty row read from L2 by its n verify rows.
// renorm: one CTA per verify row.  Pass 1 finds the row max (and the argmax).
// The top-k cut is the k-th largest order-preserving key, found by radix
// selection (8-bit digits from the top: a count histogram per level; bf16
// keys need two levels, fp32 four); the top-p cut is found the same way on
// fp64 histograms of exp((l - max)/T) over the tokens the top-k cut keeps.
// Ties at either cut are all kept.  The last pass writes p / Z (fp32).  The
// row is re-read from L2 by every pass after the first.
#include "common.cuh"
#include "kernels.cuh"

namespace spec {

namespace {

constexpr int kPenThreads = 256;

template <typename T>
__global__ void __launch_bounds__(kPenThreads) add_penalties_kernel(PenaltyParams a) {
  pdl_wait();
  pdl_trigger();
  constexpr int E = LogitTraits<T>::kVec;
  const long long rowv = a.V / E;  // 16-byte vectors a row (the host requires V % E == 0)
  const long long total = (long long)a.b * a.n * rowv;
  uint4* L = static_cast<uint4*>(a.logits);
  for (long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x; g < total;
       g += (long long)gridDim.x * blockDim.x) {
    const long long row = g / rowv, v = g % rowv;
    const int req = int(row / a.n);
    const float* pen = a.penalties + size_t(req) * a.V + size_t(v) * E;
    uint4 x = L[g];
    if constexpr (sizeof(T) == 4) {
      const float4 p = __ldg(reinterpret_cast<const float4*>(pen));
      x.x = __float_as_uint(__uint_as_float(x.x) + p.x);
      x.y = __float_as_uint(__uint_as_float(x.y) + p.y);
      x.z = __float_as_uint(__uint_as_float(x.z) + p.z);
      x.w = __float_as_uint(__uint_as_float(x.w) + p.w);
    } else {
      const float4 p0 = __ldg(reinterpret_cast<const float4*>(pen));
      const float4 p1 = __ldg(reinterpret_cast<const float4*>(pen) + 1);
      const float pp[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
      uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float lo = bf16_lo(w[q]) + pp[2 * q], hi = bf16_hi(w[q]) + pp[2 * q + 1];
        const uint32_t blo = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
        const uint32_t bhi = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
        w[q] = blo | (bhi << 16);
      }
      x = make_uint4(w[0], w[1], w[2], w[3]);
    }
    L[g] = x;
  }
}

constexpr int kRnThreads = 512;

// logit of element v of a row
template <typename T>
__device__ __forceinline__ float logit_of(const T* row, int v) {
  return LogitTraits<T>::load(row, size_t(v));
}

template <typename T>
__global__ void __launch_bounds__(kRnThreads) renorm_kernel(RenormParams a) {
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x;
  const int req = row / a.n;
  const int V = a.V, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  constexpr int nw = kRnThreads / 32;
  const T* L = static_cast<const T*>(a.logits) + size_t(row) * V;
  float* out = a.probs + size_t(row) * V;
  const float T0 = a.temperatures[req];
  const int k = a.top_k[req];
  const float tp = a.top_p[req];
  __shared__ float s_f[nw];
  __shared__ int s_i[nw];
  __shared__ unsigned s_cnt[256];
  __shared__ double s_mass[256];
  __shared__ double s_d[nw];
  __shared__ uint32_t s_prefix, s_need;
  __shared__ double s_t, s_gt;
  __shared__ int s_found;

  // pass 1: max and argmax (lowest index among equals)
  float bv = -INFINITY;
  int bi = INT_MAX;
  for (int v = tid; v < V; v += kRnThreads) {
    const float f = logit_of(L, v);
    if (better(f, v, bv, bi)) {
      bv = f;
      bi = v;
    }
  }
  warp_argmax(bv, bi);
  if (lane == 0) {
    s_f[w] = bv;
    s_i[w] = bi;
  }
  __syncthreads();
  if (w == 0) {
    float v = lane < nw ? s_f[lane] : -INFINITY;
    int i = lane < nw ? s_i[lane] : INT_MAX;
    warp_argmax(v, i);
    if (lane == 0) {
      s_f[0] = v;
      s_i[0] = i;
    }
  }
  __syncthreads();
  const float M = s_f[0];
  const int amax = s_i[0];
  if (!(T0 > 0.f)) {  // greedy row: one-hot at the argmax
    for (int v = tid; v < V; v += kRnThreads) out[v] = v == amax ? 1.f : 0.f;
    return;
  }
  // exp((l - max)/T): l - max is exact, the quotient correctly rounded
  auto weight = [&](float f) { return double(expf(__fdiv_rn(f - M, T0))); };
  const int levels = sizeof(T) == 2 ? 2 : 4;
  // a bf16 logit's key has low 16 bits all 0 (positive) or all 1 (negative)
  auto full_key = [&](uint32_t prefix) -> uint32_t {
    if (levels == 4) return prefix;
    const uint32_t hi = prefix << 16;
    return (hi & 0x80000000u) ? hi : (hi | 0xffffu);
  };

  // top-k: the k-th largest key (counts, digits from the top)
  uint32_t cut = 0;  // keep every token whose key is >= cut
  if (k > 0 && k < V) {
    if (tid == 0) {
      s_prefix = 0;
      s_need = uint32_t(k);
    }
    for (int lev = 0; lev < levels; ++lev) {
      const int shift = 24 - 8 * lev;
      for (int i = tid; i < 256; i += kRnThreads) s_cnt[i] = 0;
      __syncthreads();
      const uint32_t prefix = s_prefix;
      for (int v = tid; v < V; v += kRnThreads) {
        const uint32_t key = order_key(logit_of(L, v));
        const bool match = lev == 0 || (key >> (shift + 8)) == prefix;
        if (match) atomicAdd(&s_cnt[(key >> shift) & 0xffu], 1u);
      }
      __syncthreads();
      if (tid == 0) {
        uint32_t need = s_need;
        int d = 255;
        for (; d > 0 && s_cnt[d] < need; --d) need -= s_cnt[d];
        s_need = need;
        s_prefix = (prefix << 8) | uint32_t(d);
      }
      __syncthreads();
    }
    cut = full_key(s_prefix);
  }

  // top-p: the shortest descending prefix (of the tokens kept so far) whose
  // mass reaches top_p of their total, widened to its last key's ties
  double Z = 0.0;
  {
    double part = 0.0;
    for (int v = tid; v < V; v += kRnThreads) {
      const float f = logit_of(L, v);
      if (order_key(f) >= cut) part += weight(f);
    }
    part = warp_sum_d(part);
    if (lane == 0) s_d[w] = part;
    __syncthreads();
    if (tid == 0) {
      double z = 0.0;
      for (int i = 0; i < nw; ++i) z += s_d[i];
      s_t = z;
    }
    __syncthreads();
    Z = s_t;
    __syncthreads();  // every thread has read Z before s_t is reused below
  }
  if (tp < 1.f) {
    if (tid == 0) {
      s_prefix = 0;
      s_t = double(tp) * Z;  // mass still to reach below the current prefix
      s_gt = 0.0;            // mass of the tokens above the cut found so far
      s_found = 1;
    }
    for (int lev = 0; lev < levels; ++lev) {
      const int shift = 24 - 8 * lev;
      for (int i = tid; i < 256; i += kRnThreads) s_mass[i] = 0.0;
      __syncthreads();
      const uint32_t prefix = s_prefix;
      for (int v = tid; v < V; v += kRnThreads) {
        const float f = logit_of(L, v);
        const uint32_t key = order_key(f);
        const bool match = key >= cut && (lev == 0 || (key >> (shift + 8)) == prefix);
        if (match) atomicAdd(&s_mass[(key >> shift) & 0xffu], weight(f));
      }
      __syncthreads();
      if (tid == 0 && s_found) {
        double t = s_t, acc = 0.0;
        int d = 255;
        for (; d >= 0; --d) {
          if (acc + s_mass[d] >= t && s_mass[d] > 0.0) break;
          acc += s_mass[d];
        }
        if (d < 0) {  // rounding: the mass never reaches top_p of the total: keep the top-k set
          s_found = 0;
        } else {
          s_gt += acc;
          s_t = t - acc;
          s_prefix = (prefix << 8) | uint32_t(d);
          if (lev == levels - 1) s_d[0] = s_gt + s_mass[d];  // the kept mass
        }
      }
      __syncthreads();
    }
    if (s_found) {
      const uint32_t kp = full_key(s_prefix);
      if (kp > cut) cut = kp;
      Z = s_d[0];
    }
  }

  // write pass: p / Z on the kept tokens, 0 elsewhere
  const double invZ = 1.0 / Z;
  for (int v = tid; v < V; v += kRnThreads) {
    const float f = logit_of(L, v);
    out[v] = order_key(f) >= cut ? float(weight(f) * invZ) : 0.f;
  }
}

}  // namespace

int launch_add_penalties(const PenaltyParams& p, cudaStream_t stream) {
  const long long vecs = (long long)p.b * p.n * (p.V / (p.dtype == SPEC_F32 ? 4 : 8));
  long long ctas = (vecs + 4LL * kPenThreads - 1) / (4LL * kPenThreads);
  if (ctas > 8LL * 152) ctas = 8LL * 152;
  if (ctas < 1) ctas = 1;
  const cudaError_t e =
      p.dtype == SPEC_F32
          ? launch_pdl(add_penalties_kernel<float>, dim3(unsigned(ctas)), dim3(kPenThreads), 0, stream, p)
          : launch_pdl(add_penalties_kernel<uint16_t>, dim3(unsigned(ctas)), dim3(kPenThreads), 0, stream, p);
  if (e != cudaSuccess) return SPEC_ERR_LAUNCH;
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
}

int launch_renorm(const RenormParams& p, cudaStream_t stream) {
  const dim3 grid(p.b * p.n);
  const cudaError_t e = p.dtype == SPEC_F32
                            ? launch_pdl(renorm_kernel<float>, grid, dim3(kRnThreads), 0, stream, p)
                            : launch_pdl(renorm_kernel<uint16_t>, grid, dim3(kRnThreads), 0, stream, p);
  if (e != cudaSuccess) return SPEC_ERR_LAUNCH;
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
}

}  // namespace spec
