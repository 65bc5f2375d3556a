// attention_merge.cu -- combines the split-KV partials of the verify attention.
//
// Each split of a request's key list leaves, per (verify row, q head), an
// unnormalised output o_s, its running max m_s (log2 domain) and sum l_s.  The
// merge takes M = max m_s, L = sum l_s 2^(m_s - M), O = sum o_s 2^(m_s - M) / L,
// rounds O to bf16 (nearest even) and writes lse = (M + log2 L) ln 2.  One warp
// per (row, head), D/32 output dimensions per lane.
#include "common.cuh"
#include "kernels.cuh"

namespace spec {

namespace {

template <int D>
__global__ void __launch_bounds__(256) attention_merge_kernel(AttentionParams a) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int pairs = a.b * a.n * a.Hq;
  if (warp >= pairs) return;
  constexpr int DPL = D / 32;
  const float* po = reinterpret_cast<const float*>(a.partials);
  const float* pml = po + size_t(a.b) * a.n * a.Hq * a.splits * D;
  const size_t base = size_t(warp) * a.splits;
  float M = -INFINITY;
  for (int s = 0; s < a.splits; ++s) M = fmaxf(M, pml[(base + s) * 2]);
  float Lsum = 0.f, o[DPL];
#pragma unroll
  for (int d = 0; d < DPL; ++d) o[d] = 0.f;
  for (int s = 0; s < a.splits; ++s) {
    const float ms = pml[(base + s) * 2], ls = pml[(base + s) * 2 + 1];
    if (ls == 0.f) continue;
    const float f = exp2f(ms - M);
    Lsum += ls * f;
#pragma unroll
    for (int d = 0; d < DPL; ++d) o[d] += po[(base + s) * D + lane * DPL + d] * f;
  }
  const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
  uint16_t* out = static_cast<uint16_t*>(a.out);
#pragma unroll
  for (int d = 0; d < DPL; ++d) {
    const float y = o[d] * inv;
    // round to nearest even bf16
    uint32_t u = __float_as_uint(y);
    u += 0x7fffu + ((u >> 16) & 1u);
    out[size_t(warp) * D + lane * DPL + d] = uint16_t(u >> 16);
  }
  if (a.lse && lane == 0) a.lse[warp] = Lsum > 0.f ? (M + log2f(Lsum)) * 0.6931471805599453f : -INFINITY;
}

}  // namespace

size_t attention_partial_bytes(int b, int n, int Hq, int D, int splits) {
  return align256(size_t(b) * n * Hq * splits * (D + 2) * 4);
}

int launch_attention_merge(const AttentionParams& p, cudaStream_t stream) {
  const int pairs = p.b * p.n * p.Hq;
  const int mblocks = (pairs * 32 + 255) / 256;
  if (p.D == 128)
    attention_merge_kernel<128><<<mblocks, 256, 0, stream>>>(p);
  else
    attention_merge_kernel<64><<<mblocks, 256, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
}

}  // namespace spec
