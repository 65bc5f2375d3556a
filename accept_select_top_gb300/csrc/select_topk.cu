// select_topk.cu -- one step of select_top_k_tokens with the draft softmax and
// top-k fused in.
//
// [SGL-XI organize_draft_results: _select_top_k_tokens_first / _later, the
// parent offset topk_cs_index + topk^2 (i-1) + topk], [SGL-XI draft() 主循环].
//
// Grid: (chunks, rows), rows = b * (step ? k : 1).  Each CTA streams one chunk
// of one draft row once, keeping per thread an online softmax (running max and
// sum of exp) and a sorted top-K list (K = topk rounded up to a power of two);
// the CTA merges these into one partial (max, sum, K best logits).  The CTA
// arriving last for a request merges the partials of the request's rows (one
// warp per row: k-round tournament over the chunk lists), turns the k best
// logits into probabilities, and runs the path-score step for the request.
#include "common.cuh"
#include "kernels.cuh"

namespace spec {

namespace {

struct SelPart {
  float m;   // max logit of the chunk
  float s;   // sum of exp((x - m) / T) over the chunk
  float v[kMaxK];
  int i[kMaxK];
};

template <int K>
struct TopList {
  float v[K];
  int i[K];
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int j = 0; j < K; ++j) {
      v[j] = -INFINITY;
      i[j] = INT_MAX;
    }
  }
  // Insert (x, ix) if it ranks before the current K-th entry.
  __device__ __forceinline__ void push(float x, int ix) {
    if (!better(x, ix, v[K - 1], i[K - 1])) return;
    bool placed = false;
#pragma unroll
    for (int j = K - 1; j > 0; --j) {
      const bool up = !placed && better(x, ix, v[j - 1], i[j - 1]);
      const float nv = up ? v[j - 1] : (placed ? v[j] : x);
      const int ni = up ? i[j - 1] : (placed ? i[j] : ix);
      placed = placed || !up;
      v[j] = nv;
      i[j] = ni;
    }
    if (!placed) {
      v[0] = x;
      i[0] = ix;
    }
  }
  __device__ __forceinline__ void pop_front() {
#pragma unroll
    for (int j = 0; j < K - 1; ++j) {
      v[j] = v[j + 1];
      i[j] = i[j + 1];
    }
    v[K - 1] = -INFINITY;
    i[K - 1] = INT_MAX;
  }
};

template <typename T, int K>
__device__ __forceinline__ void scan_row(const T* row, int begin, int end, bool vec, float c,
                                         float& m, float& s, TopList<K>& top) {
  using Tr = LogitTraits<T>;
  constexpr int E = Tr::kVec;
  auto consume = [&](const float* f, int n_el, int first) {
    float vm = f[0];
    for (int e = 1; e < n_el; ++e) vm = fmaxf(vm, f[e]);
    if (vm >= top.v[K - 1]) {
      for (int e = 0; e < n_el; ++e) top.push(f[e], first + e);
    }
    if (vm > m) {
      s *= exp2f((m - vm) * c);
      m = vm;
    }
    for (int e = 0; e < n_el; ++e) s += exp2f((f[e] - m) * c);
  };
  if (vec) {
    const uint4* p = reinterpret_cast<const uint4*>(row);
    const int vb = begin / E, ve = end / E;
    constexpr int U = 4;
    for (int v0 = vb + threadIdx.x; v0 < ve; v0 += blockDim.x * U) {
      uint4 x[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        int idx = v0 + u * blockDim.x;
        if (idx < ve) x[u] = ld_stream(p + idx);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        int idx = v0 + u * blockDim.x;
        if (idx >= ve) break;
        float f[E];
        Tr::unpack(x[u], f);
        consume(f, E, idx * E);
      }
    }
  } else {
    for (int i = begin + threadIdx.x; i < end; i += blockDim.x) {
      float f = Tr::load(row, i);
      consume(&f, 1, i);
    }
  }
}

// Merge the lanes' sorted lists of a warp into the warp's best K (written by
// lane 0 to out_v / out_i).  Destroys the lanes' lists.
template <int K>
__device__ __forceinline__ void warp_merge(TopList<K>& top, float* out_v, int* out_i) {
  const int lane = threadIdx.x & 31;
  for (int r = 0; r < K; ++r) {
    float v = top.v[0];
    int i = top.i[0];
    warp_argmax(v, i);
    if (top.v[0] == v && top.i[0] == i && i != INT_MAX) top.pop_front();
    if (lane == 0) {
      out_v[r] = v;
      out_i[r] = i;
    }
  }
}

template <typename T, int K>
__global__ void __launch_bounds__(kThreads) select_kernel(SelectParams a) {
  const int row = blockIdx.y;
  const int chunk = blockIdx.x;
  const int rows_per_req = a.step ? a.k : 1;
  const int req = row / rows_per_req;
  const int begin = chunk * a.chunk_elems;
  const int end = min(a.V, begin + a.chunk_elems);
  const T* lrow = static_cast<const T*>(a.logits) + size_t(row) * a.V;
  const float c = 1.4426950408889634f / a.temperature;  // log2(e) / T

  float m = -3.0e38f, s = 0.f;
  TopList<K> top;
  top.init();
  scan_row<T, K>(lrow, begin, end, a.vec_ok, c, m, s, top);

  // ---- CTA merge: softmax stats and top-K ----
  __shared__ float wm[kThreads / 32], ws_[kThreads / 32];
  __shared__ float lv[kThreads / 32][K];
  __shared__ int li[kThreads / 32][K];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  {
    float M = warp_max(m);
    float sc = s * exp2f((m - M) * c);
    sc = warp_sum(sc);
    if (lane == 0) {
      wm[w] = M;
      ws_[w] = sc;
    }
  }
  warp_merge<K>(top, lv[w], li[w]);
  __syncthreads();
  SelPart* part = reinterpret_cast<SelPart*>(a.partials) + size_t(row) * a.chunks + chunk;
  if (w == 0) {
    float M = lane < nw ? wm[lane] : -3.0e38f;
    M = warp_max(M);
    float sc = lane < nw ? ws_[lane] * exp2f((wm[lane] - M) * c) : 0.f;
    sc = warp_sum(sc);
    // rank each of the nw*K candidates among all of them (lowest-index ties)
    for (int t = lane; t < nw * K; t += 32) {
      const float v = lv[t / K][t % K];
      const int ix = li[t / K][t % K];
      int rank = 0;
      for (int u = 0; u < nw * K; ++u) rank += better(lv[u / K][u % K], li[u / K][u % K], v, ix);
      if (rank < K) {
        part->v[rank] = v;
        part->i[rank] = ix;
      }
    }
    if (lane == 0) {
      part->m = M;
      part->s = sc;
    }
  }

  if (!arrive_last(a.counters + req, uint32_t(rows_per_req * a.chunks))) return;

  // ---- finalize request `req` ----
  const int k = a.k;
  __shared__ float heads_v[kThreads / 32][kMaxChunks * K];  // one warp per row
  __shared__ int heads_i[kThreads / 32][kMaxChunks * K];
  __shared__ float p_s[kMaxK][kMaxK];
  __shared__ int id_s[kMaxK][kMaxK];
  for (int r = w; r < rows_per_req; r += nw) {
    const int grow = req * rows_per_req + r;
    const SelPart* pr = reinterpret_cast<const SelPart*>(a.partials) + size_t(grow) * a.chunks;
    // softmax denominator of the whole row
    float M = -3.0e38f;
    for (int ch = lane; ch < a.chunks; ch += 32) M = fmaxf(M, __ldcg(&pr[ch].m));
    M = warp_max(M);
    float S = 0.f;
    for (int ch = lane; ch < a.chunks; ch += 32) S += __ldcg(&pr[ch].s) * exp2f((__ldcg(&pr[ch].m) - M) * c);
    S = warp_sum(S);
    // stage the chunk lists, then k rounds of a tournament over list heads
    for (int t = lane; t < a.chunks * K; t += 32) {
      heads_v[w][t] = __ldcg(&pr[t / K].v[t % K]);
      heads_i[w][t] = __ldcg(&pr[t / K].i[t % K]);
    }
    __syncwarp();
    int h0 = 0, h1 = 0;  // list heads of chunks lane and lane + 32
    for (int j = 0; j < k; ++j) {
      float v = -INFINITY;
      int ix = INT_MAX, src = -1;
      if (lane < a.chunks && h0 < K && better(heads_v[w][lane * K + h0], heads_i[w][lane * K + h0], v, ix)) {
        v = heads_v[w][lane * K + h0];
        ix = heads_i[w][lane * K + h0];
        src = 0;
      }
      if (lane + 32 < a.chunks && h1 < K &&
          better(heads_v[w][(lane + 32) * K + h1], heads_i[w][(lane + 32) * K + h1], v, ix)) {
        v = heads_v[w][(lane + 32) * K + h1];
        ix = heads_i[w][(lane + 32) * K + h1];
        src = 1;
      }
      float bv = v;
      int bi = ix;
      warp_argmax(bv, bi);
      if (src >= 0 && bv == v && bi == ix) {
        if (src == 0) ++h0;
        else ++h1;
      }
      if (lane == 0) {
        // p = exp((x - M) / T) / S with the exponential in fp64
        const double e = exp((double(bv) - double(M)) / double(a.temperature));
        p_s[r][j] = float(e / double(S));
        id_s[r][j] = bi;
      }
    }
    __syncwarp();
  }
  __syncthreads();
  if (a.topk_p_out) {
    for (int t = threadIdx.x; t < rows_per_req * k; t += blockDim.x)
      a.topk_p_out[size_t(req * rows_per_req + t / k) * k + t % k] = p_s[t / k][t % k];
  }
  const size_t sb = size_t(req) * a.score_ld;
  if (a.step == 0) {
    for (int j = threadIdx.x; j < k; j += blockDim.x) {
      a.score_blk[sb + j] = p_s[0][j];
      a.token_blk[sb + j] = id_s[0][j];
      a.scores_out[size_t(req) * k + j] = p_s[0][j];
      a.next_ids[size_t(req) * k + j] = id_s[0][j];
    }
    if (a.parent_blk)
      for (int j = threadIdx.x; j <= k; j += blockDim.x) a.parent_blk[size_t(req) * a.parent_ld + j] = j - 1;
  } else if (w == 0) {
    // expand[r*k + j] = scores_in[r] * p[r][j] (one fp32 multiply); top-k of k*k
    const int kk = k * k;
    __shared__ float ex[kMaxK * kMaxK];
    for (int f = lane; f < kk; f += 32) {
      ex[f] = __fmul_rn(a.scores_in[size_t(req) * k + f / k], p_s[f / k][f % k]);
      a.score_blk[sb + f] = ex[f];
      a.token_blk[sb + f] = id_s[f / k][f % k];
    }
    __syncwarp();
    for (int f = lane; f < kk; f += 32) {
      int rank = 0;
      for (int g = 0; g < kk; ++g) rank += better(ex[g], g, ex[f], f);
      if (rank < k) {
        if (a.parent_blk) a.parent_blk[size_t(req) * a.parent_ld + rank] = f + kk * (a.step - 1) + k;
        a.scores_out[size_t(req) * k + rank] = ex[f];
        a.next_ids[size_t(req) * k + rank] = id_s[f / k][f % k];
      }
    }
  }
  counter_reset(a.counters + req);
}

template <typename T>
int launch_t(const SelectParams& p, cudaStream_t stream) {
  dim3 grid(p.chunks, p.rows);
  const int K = p.k <= 1 ? 1 : p.k <= 2 ? 2 : p.k <= 4 ? 4 : p.k <= 8 ? 8 : 16;
  switch (K) {
    case 1: select_kernel<T, 1><<<grid, kThreads, 0, stream>>>(p); break;
    case 2: select_kernel<T, 2><<<grid, kThreads, 0, stream>>>(p); break;
    case 4: select_kernel<T, 4><<<grid, kThreads, 0, stream>>>(p); break;
    case 8: select_kernel<T, 8><<<grid, kThreads, 0, stream>>>(p); break;
    default: select_kernel<T, 16><<<grid, kThreads, 0, stream>>>(p); break;
  }
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
}

}  // namespace

size_t select_partial_bytes(int rows, int chunks) { return align256(size_t(rows) * chunks * sizeof(SelPart)); }

int launch_select_topk(const SelectParams& p, cudaStream_t stream) {
  return p.dtype == SPEC_F32 ? launch_t<float>(p, stream) : launch_t<uint16_t>(p, stream);
}

}  // namespace spec
