// verify_greedy.cu -- greedy accept: per-row argmax over the vocabulary, then
// the first-child / next-sibling walk from the root.
//
// [SGL-XI eagle_sample, 路径一:贪心验证], [ACCEPT section 3 (pseudocode of the
// walk, row/output shift)], [EAGLE2 section 5.3].
//
// Grid: (chunks, b*n).  Each CTA reduces one chunk of one verify row to its
// (max, lowest index) pair with 16-byte streaming loads; the CTA that finishes
// last for a request merges the request's partials into target_predict and
// runs the walk for that request (one thread: at most S levels of at most n
// siblings), then writes predict / accept_index / accept_lens.
#include "common.cuh"
#include "kernels.cuh"

namespace spec {

namespace {

struct ArgPart {
  float v;
  int i;
};

__device__ __forceinline__ void block_argmax(float& v, int& i) {
  __shared__ float sv[kThreads / 32];
  __shared__ int si[kThreads / 32];
  warp_argmax(v, i);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) {
    sv[w] = v;
    si[w] = i;
  }
  __syncthreads();
  if (w == 0) {
    v = l < int(blockDim.x >> 5) ? sv[l] : -INFINITY;
    i = l < int(blockDim.x >> 5) ? si[l] : INT_MAX;
    warp_argmax(v, i);
  }
}

// Argmax (max value, lowest index) of bf16 row[begin, end) by 16-byte
// vectors: per vector one packed max and one compare; the thread keeps its
// best vector (the first one with the best maximum) and resolves the element
// inside it at the end.  The thread's first vector is always taken, so a
// row of -inf still yields its lowest index.
__device__ __forceinline__ void scan_argmax_bf16(const uint16_t* row, int begin, int end, float& bv, int& bi) {
  constexpr int U = 8;  // 128 bytes per thread in flight: a chunk in about two round trips
  const uint4* p = reinterpret_cast<const uint4*>(row);
  const int nt = blockDim.x, ve = end / 8;
  int bvi = -1;
  uint4 bx = make_uint4(0u, 0u, 0u, 0u);
  for (int v0 = begin / 8 + int(threadIdx.x); v0 < ve; v0 += U * nt) {
    uint4 x[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + u * nt;
      x[u] = v < ve ? ld_stream(p + v) : VecOps<uint16_t>::neg_inf();
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + u * nt;
      const float mf = VecOps<uint16_t>::vmax(x[u]);
      if (v < ve && (mf > bv || (bvi < 0 && mf == mf))) {
        bv = mf;
        bvi = v;
        bx = x[u];
      }
    }
  }
  bi = INT_MAX;
  if (bvi >= 0) {
#pragma unroll
    for (int e = 7; e >= 0; --e)
      if (VecOps<uint16_t>::at(bx, e) == bv) bi = bvi * 8 + e;
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) greedy_kernel(GreedyParams a) {
  // The scan reads only the target logits and greedy's own partials and
  // counters.  When the caller has allowed overlap and the kernel before is
  // the verify attention on the same workspace, the scan runs before waiting
  // on it; only the finalize waits.  Otherwise everything waits.
  if (!a.early) {
    pdl_wait();
    pdl_trigger();
  }
  const int row = blockIdx.y;
  const int chunk = blockIdx.x;
  const int req = row / a.n;
  const int begin = chunk * a.chunk_elems;
  const int end = min(a.V, begin + a.chunk_elems);
  const T* lrow = static_cast<const T*>(a.logits) + size_t(row) * a.V;

  float bv = -INFINITY;
  int bi = INT_MAX;
  if constexpr (sizeof(T) == 2) {
    if (a.vec_ok) {
      scan_argmax_bf16(lrow, begin, end, bv, bi);
    } else {
      float unused_m = 0.f, unused_s = 0.f;
      scan_row_stats<T>(lrow, begin, end, false, false, 0.f, bv, bi, unused_m, unused_s);
    }
  } else {
    float unused_m = 0.f, unused_s = 0.f;
    scan_row_stats<T>(lrow, begin, end, a.vec_ok, false, 0.f, bv, bi, unused_m, unused_s);
  }
  block_argmax(bv, bi);
  ArgPart* part = reinterpret_cast<ArgPart*>(a.partials);
  if (threadIdx.x == 0) part[size_t(row) * a.chunks + chunk] = ArgPart{bv, bi};

  if (!arrive_last(a.counters + req, uint32_t(a.n * a.chunks))) return;
  if (a.early) {
    pdl_wait();
    pdl_trigger();
  }

  // ---- finalize request `req` (last CTA to arrive) ----
  const int n = a.n, base = req * n, W = a.S + 1;
  __shared__ int tp[kMaxN], tok[kMaxN], nt[kMaxN], ns[kMaxN], ri[kMaxN], pred[kMaxN], path[kMaxN + 1];
  __shared__ int2 stage[kMaxN * kMaxChunks];
  __shared__ int s_len;
  // the request's tree arrays (or chain tokens) and every (row, chunk)
  // partial in one round of loads; partials of other CTAs are read through L2
  // (__ldcg), not a stale L1 line
  const int tt = threadIdx.x;
  int tok0 = 0, x0 = -1, y0 = -1, r0 = base, pre = 0;
  if (a.chain) {
    tok0 = tt < a.S ? a.chain_drafts[size_t(req) * a.draft_ld + tt] : 0;
    if (tt == 0) pre = a.prefix_lens[req];
  } else {
    tok0 = tt < n ? a.draft_tokens[base + tt] : 0;
    x0 = tt < n ? a.next_token[base + tt] : -1;
    y0 = tt < n ? a.next_sibling[base + tt] : -1;
    r0 = tt < n ? a.retrieve_index[base + tt] : base;
  }
  for (int t = threadIdx.x; t < n * a.chunks; t += blockDim.x)
    stage[t] = __ldcg(reinterpret_cast<const int2*>(part + size_t(base) * a.chunks) + t);
  __syncthreads();
  if (a.chain) {
    // compute_dflash_correct_drafts_and_bonus [ACCEPT section 5]: the number
    // of leading chain positions whose draft token is the target's argmax
    // (the first mismatch ends it), the bonus at that position, the
    // fixed-width out tokens with the bonus scattered there, commit_lens =
    // correct_len + 1, new_seq_lens = prefix_lens + commit_lens
    for (int t = threadIdx.x; t < n; t += blockDim.x) {
      float v = -INFINITY;
      int i = INT_MAX;
      for (int c = 0; c < a.chunks; ++c) {
        const int2 q = stage[t * a.chunks + c];
        const float qv = __int_as_float(q.x);
        if (better(qv, q.y, v, i)) {
          v = qv;
          i = q.y;
        }
      }
      tp[t] = i;
      tok[t] = tok0;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int c = 0;
      while (c < a.S && tok[c] == tp[c]) ++c;
      s_len = c;
      a.correct_len[req] = c;
      a.bonus[req] = tp[c];
      a.commit_lens[req] = c + 1;
      a.new_seq_lens[req] = pre + c + 1;
    }
    __syncthreads();
    const int c = s_len;
    for (int j = threadIdx.x; j < n; j += blockDim.x) {
      a.out_tokens[size_t(req) * n + j] = j == c ? tp[c] : (j < a.S ? tok[j] : -1);
      if (a.accept_index) a.accept_index[size_t(req) * n + j] = j <= c ? base + j : -1;
    }
    counter_reset(a.counters + req);
    return;
  }
  for (int t = threadIdx.x; t < n; t += blockDim.x) {
    float v = -INFINITY;
    int i = INT_MAX;
    for (int c = 0; c < a.chunks; ++c) {
      const int2 q = stage[t * a.chunks + c];
      const float qv = __int_as_float(q.x);
      if (better(qv, q.y, v, i)) {
        v = qv;
        i = q.y;
      }
    }
    tp[t] = i;
    tok[t] = tok0;  // t == threadIdx.x: n <= kMaxN < blockDim.x
    int x = x0, y = y0, r = r0;
    if (x < -1 || x >= n || y < -1 || y >= n) {
      raise_error(a.error, SPEC_DEV_INDEX);
      x = x < -1 || x >= n ? -1 : x;
      y = y < -1 || y >= n ? -1 : y;
    }
    if (r < base || r >= base + n) {
      raise_error(a.error, SPEC_DEV_INDEX);
      r = base + t;
    }
    nt[t] = x;
    ns[t] = y;
    ri[t] = r;
    pred[t] = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int cur = 0, ncd = 0;
    path[0] = 0;
    // a valid tree is at most n-1 deep; the bound also stops a malformed (cyclic) one
    for (int d = 1; d <= a.S && ncd < n - 1; ++d) {
      int c = nt[cur], hit = -1, guard = 0;
      while (c != -1 && guard++ < n) {
        if (tok[c] == tp[cur]) {
          hit = c;
          break;
        }
        c = ns[c];
      }
      if (hit < 0) break;
      pred[cur] = tok[hit];
      path[++ncd] = hit;
      cur = hit;
    }
    pred[cur] = tp[cur];
    s_len = ncd + 1;
    a.accept_lens[req] = ncd + 1;
    if (a.next_root) a.next_root[req] = tp[cur];
  }
  __syncthreads();
  const int L = s_len;
  for (int t = threadIdx.x; t < n; t += blockDim.x) a.predict[ri[t]] = pred[t];
  for (int d = threadIdx.x; d < W; d += blockDim.x) {
    a.accept_index[size_t(req) * W + d] = d < L ? ri[path[d]] : -1;
    if (a.accepted_tokens) a.accepted_tokens[size_t(req) * W + d] = d < L ? pred[path[d]] : -1;
  }
  counter_reset(a.counters + req);
}

}  // namespace

int launch_verify_greedy(const GreedyParams& p, cudaStream_t stream) {
  dim3 grid(p.chunks, p.b * p.n);
  const cudaError_t e = p.dtype == SPEC_F32 ? launch_pdl(greedy_kernel<float>, grid, dim3(kThreads), 0, stream, p)
                                             : launch_pdl(greedy_kernel<uint16_t>, grid, dim3(kThreads), 0, stream, p);
  if (e != cudaSuccess) return SPEC_ERR_LAUNCH;
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
}

}  // namespace spec
