// attention_simple.cu -- tree-masked verify attention on CUDA cores (split-KV).
//
// [EAGLE2 sections 4.2-4.3: the queries are the flattened tree nodes; the keys
// are the cached history (all visible) followed by the tree nodes, of which a
// query sees only its ancestors and itself], [SGL-XI QLEN_ONLY mask: the prefix
// columns are implicitly visible, only the n x n tree block is stored].
//
// Grid: (Hkv * row_groups, b, splits).  A CTA owns up to 64 query rows of one
// (request, kv head) -- rows are (node, q head in the group) pairs -- and one
// contiguous range of the request's key list (prefix positions then tree
// nodes).  Keys are staged 32 at a time in shared memory; each warp keeps an
// online softmax per row, one lane per key for the scores and D/32 output
// dimensions per lane.  Partials (unnormalised o, running max, sum) go to the
// workspace and attention_merge_kernel combines the splits.
#include "common.cuh"
#include "kernels.cuh"

namespace spec {

namespace {

constexpr int kAttThreads = 256;
constexpr int kRowsPerCta = 64;
constexpr int kKeyTile = 32;

template <int D>
__global__ void __launch_bounds__(kAttThreads) attention_simple_kernel(AttentionParams a) {
  constexpr int DW = D / 2;       // 32-bit words per key row
  constexpr int KS = DW + 1;      // padded smem stride (words): conflict-free lane-per-key reads
  constexpr int DPL = D / 32;     // output dims per lane
  __shared__ uint32_t q_s[kRowsPerCta][DW];
  __shared__ uint32_t k_s[kKeyTile][KS];
  __shared__ uint32_t v_s[kKeyTile][DW];
  __shared__ long long slot_s[kKeyTile];
  __shared__ int vis_bit_s[kKeyTile];  // -1: prefix key (visible), j: tree node j, -2: none

  const int G = a.Hq / a.Hkv;
  const int M = a.n * G;
  const int row_groups = (M + kRowsPerCta - 1) / kRowsPerCta;
  const int g = blockIdx.x / row_groups, rg = blockIdx.x % row_groups;
  const int req = blockIdx.y, split = blockIdx.z;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // request geometry (bounds-checked)
  int L = a.seq_lens[req];
  const int rq = a.req_pool_idx[req];
  bool ok = rq >= 0 && rq < a.req_rows;
  if (L < 0 || L > a.max_seq_len || L > a.row_w) {
    if (threadIdx.x == 0) raise_error(a.error, SPEC_DEV_LENGTH);
    L = max(0, min(L, min(a.max_seq_len, a.row_w)));
  }
  if (!ok && threadIdx.x == 0 && split == 0 && rg == 0 && g == 0) raise_error(a.error, SPEC_DEV_INDEX);
  const int total = ok ? L + a.n : 0;
  const int per = ((a.max_seq_len + a.n + a.splits - 1) / a.splits + kKeyTile - 1) / kKeyTile * kKeyTile;
  const int k0 = split * per, k1 = min(total, k0 + per);

  // stage q rows of this group: row r -> (node i = r / G, head h = g*G + r % G)
  const int r0 = rg * kRowsPerCta, rcount = min(kRowsPerCta, M - r0);
  for (int t = threadIdx.x; t < rcount * DW; t += blockDim.x) {
    const int r = t / DW, wd = t % DW;
    const int i = (r0 + r) / G, h = g * G + (r0 + r) % G;
    q_s[r][wd] = reinterpret_cast<const uint32_t*>(a.q)[((size_t(req) * a.n + i) * a.Hq + h) * DW + wd];
  }
  // per-warp row state
  constexpr int kRowsPerWarp = kRowsPerCta / (kAttThreads / 32);
  float m_r[kRowsPerWarp], l_r[kRowsPerWarp], o_r[kRowsPerWarp][DPL];
  uint64_t mask_r[kRowsPerWarp];
#pragma unroll
  for (int x = 0; x < kRowsPerWarp; ++x) {
    m_r[x] = -INFINITY;
    l_r[x] = 0.f;
#pragma unroll
    for (int d = 0; d < DPL; ++d) o_r[x][d] = 0.f;
    const int r = w + x * (kAttThreads / 32);
    mask_r[x] = r < rcount ? a.mask_bits[size_t(req) * a.n + (r0 + r) / G] : 0;
  }
  const float sl2 = a.scale * 1.4426950408889634f;
  const uint32_t* kp = reinterpret_cast<const uint32_t*>(a.k_pool);
  const uint32_t* vp = reinterpret_cast<const uint32_t*>(a.v_pool);

  for (int t0 = k0; t0 < k1; t0 += kKeyTile) {
    __syncthreads();
    if (threadIdx.x < kKeyTile) {
      const int t = t0 + threadIdx.x;
      long long slot = -1;
      int vb = -2;
      if (t < k1) {
        if (t < L) {
          slot = a.req_to_token[size_t(rq) * a.row_w + t];
          vb = -1;
        } else {
          slot = a.verify_loc[size_t(req) * a.n + (t - L)];
          vb = t - L;
        }
        if (slot < 0 || slot >= a.num_slots) {
          raise_error(a.error, SPEC_DEV_INDEX);
          slot = -1;
          vb = -2;
        }
      }
      slot_s[threadIdx.x] = slot;
      vis_bit_s[threadIdx.x] = vb;
    }
    __syncthreads();
    for (int t = threadIdx.x; t < kKeyTile * DW; t += blockDim.x) {
      const int j = t / DW, wd = t % DW;
      const long long s = slot_s[j];
      uint32_t kv = 0, vv = 0;
      if (s >= 0) {
        kv = kp[(size_t(s) * a.Hkv + g) * DW + wd];
        vv = vp[(size_t(s) * a.Hkv + g) * DW + wd];
      }
      k_s[j][wd] = kv;
      v_s[j][wd] = vv;
    }
    __syncthreads();
#pragma unroll
    for (int x = 0; x < kRowsPerWarp; ++x) {
      const int r = w + x * (kAttThreads / 32);
      if (r >= rcount) break;
      // score of key `lane` for row r
      float acc = 0.f;
#pragma unroll 8
      for (int wd = 0; wd < DW; ++wd) {
        const uint32_t qa = q_s[r][wd], ka = k_s[lane][wd];
        acc = fmaf(bf16_lo(qa), bf16_lo(ka), acc);
        acc = fmaf(bf16_hi(qa), bf16_hi(ka), acc);
      }
      const int vb = vis_bit_s[lane];
      const bool vis = vb == -1 || (vb >= 0 && ((mask_r[x] >> vb) & 1ull));
      const float s2 = vis ? acc * sl2 : -INFINITY;
      const float mt = warp_max(s2);
      const float mn = fmaxf(m_r[x], mt);
      if (mn == -INFINITY) continue;  // nothing visible yet
      const float corr = exp2f(m_r[x] - mn);
      const float pj = vis ? exp2f(s2 - mn) : 0.f;
      l_r[x] = l_r[x] * corr + warp_sum(pj);
      m_r[x] = mn;
#pragma unroll
      for (int d = 0; d < DPL; ++d) o_r[x][d] *= corr;
      for (int j = 0; j < kKeyTile; ++j) {
        const float pb = __shfl_sync(0xffffffffu, pj, j);
        if (pb == 0.f) continue;
#pragma unroll
        for (int d = 0; d < DPL; d += 2) {
          const uint32_t vv = v_s[j][(lane * DPL + d) / 2];
          o_r[x][d] = fmaf(pb, bf16_lo(vv), o_r[x][d]);
          o_r[x][d + 1] = fmaf(pb, bf16_hi(vv), o_r[x][d + 1]);
        }
      }
    }
  }
  // write partials: index ((row * Hq + h) * splits + split)
  float* po = reinterpret_cast<float*>(a.partials);
  float* pml = po + size_t(a.b) * a.n * a.Hq * a.splits * D;
#pragma unroll
  for (int x = 0; x < kRowsPerWarp; ++x) {
    const int r = w + x * (kAttThreads / 32);
    if (r >= rcount) break;
    const int i = (r0 + r) / G, h = g * G + (r0 + r) % G;
    const size_t idx = ((size_t(req) * a.n + i) * a.Hq + h) * a.splits + split;
#pragma unroll
    for (int d = 0; d < DPL; ++d) po[idx * D + lane * DPL + d] = o_r[x][d];
    if (lane == 0) {
      pml[idx * 2] = m_r[x];
      pml[idx * 2 + 1] = l_r[x];
    }
  }
}

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

int attention_splits(int b, int n, int Hq, int Hkv, int max_seq_len) {
  const int G = Hq / Hkv;
  const int rg = (n * G + kRowsPerCta - 1) / kRowsPerCta;
  const long units = long(b) * Hkv * rg;
  long s = (2L * kTargetCtas + units - 1) / units;
  const long by_len = (max_seq_len + n + 255) / 256;  // at least ~256 keys per split
  if (s > by_len) s = by_len;
  if (s < 1) s = 1;
  if (s > 256) s = 256;
  return int(s);
}

size_t attention_partial_bytes(int b, int n, int Hq, int D, int splits) {
  return align256(size_t(b) * n * Hq * splits * (D + 2) * 4);
}

int launch_attention_simple(const AttentionParams& p, cudaStream_t stream) {
  const int G = p.Hq / p.Hkv;
  const int rg = (p.n * G + kRowsPerCta - 1) / kRowsPerCta;
  dim3 grid(p.Hkv * rg, p.b, p.splits);
  const int pairs = p.b * p.n * p.Hq;
  const int mblocks = (pairs * 32 + 255) / 256;
  if (p.D == 128) {
    attention_simple_kernel<128><<<grid, kAttThreads, 0, stream>>>(p);
    attention_merge_kernel<128><<<mblocks, 256, 0, stream>>>(p);
  } else {
    attention_simple_kernel<64><<<grid, kAttThreads, 0, stream>>>(p);
    attention_merge_kernel<64><<<mblocks, 256, 0, stream>>>(p);
  }
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
}

}  // namespace spec
