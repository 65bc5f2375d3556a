// select_topk.cu -- one step of select_top_k_tokens with the draft softmax and
// top-k fused in.
//
// [SGL-XI organize_draft_results: _select_top_k_tokens_first / _later, the
// parent offset topk_cs_index + topk^2 (i-1) + topk], [SGL-XI draft() 主循环].
//
// Grid: (chunks, rows), rows = b * (step ? k : 1).  Each CTA reads one chunk
// of one draft row once into registers (32 logits a thread).  Each warp takes
// its maximum Mw and its sum of exp((x - Mw) / T); the k-th largest warp
// maximum bounds the chunk's k best from below (k distinct elements in k
// different warps reach it), so only the few elements at or above it are
// ranked; the CTA writes one partial (max, sum, K best logits, K = topk
// rounded up to a power of two).  The CTA arriving last for a request merges
// the partials of the request's rows (one warp per row, each lane holding one
// chunk's list: a k-round tournament), turns the k best logits into
// probabilities, and runs the path-score step for the request.  With overlap
// allowed by the caller, the chunk pass may overlap the call before it (see
// the kernel).
#include "common.cuh"
#include "kernels.cuh"
#include "stream_records.cuh"

namespace spec {

namespace {

// 16-byte aligned, lists first, so that a lane reads a chunk's partial with
// 16-byte loads
struct alignas(16) SelPart {
  float v[kMaxK];
  int i[kMaxK];
  float m;   // max logit of the chunk
  float s;   // sum of exp((x - m) / T) over the chunk
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

// Elements one thread holds: its share of the chunk fits in registers.
constexpr int kPerThread = 32;

// Loads this thread's elements of row[begin, end) into f: vectors
// vb + tid + u*blockDim (16-byte loads) or single elements
// begin + tid + j*blockDim; -inf where there is none.  share_index() gives
// the vocabulary index of f[j].
template <typename T>
__device__ __forceinline__ void load_share(const T* row, int begin, int end, bool vec, float (&f)[kPerThread]) {
  using Tr = LogitTraits<T>;
  constexpr int E = Tr::kVec;
  constexpr int U = kPerThread / E;
  if (vec) {
    const uint4* p = reinterpret_cast<const uint4*>(row);
    const int vb = begin / E, ve = end / E;
    uint4 x[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = vb + threadIdx.x + u * blockDim.x;
      if (v < ve) x[u] = ld_stream(p + v);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = vb + threadIdx.x + u * blockDim.x;
      float g[E];
      if (v < ve) {
        Tr::unpack(x[u], g);
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) g[e] = -INFINITY;
      }
#pragma unroll
      for (int e = 0; e < E; ++e) f[u * E + e] = g[e];
    }
  } else {
#pragma unroll
    for (int j = 0; j < kPerThread; ++j) {
      const int i = begin + threadIdx.x + j * blockDim.x;
      f[j] = i < end ? Tr::load(row, i) : -INFINITY;
    }
  }
}

template <typename T>
__device__ __forceinline__ int share_index(int begin, bool vec, int j) {
  constexpr int E = LogitTraits<T>::kVec;
  return vec ? (begin / E + int(threadIdx.x) + (j / E) * int(blockDim.x)) * E + j % E
             : begin + int(threadIdx.x) + j * int(blockDim.x);
}

// The k-th largest of the lanes' values (-inf when fewer than k lanes hold one).
__device__ __forceinline__ float warp_kth_largest(float v, int k) {
  float kth = -INFINITY;
  for (int r = 0; r < k; ++r) {
    const float mx = warp_max(v);
    kth = mx;
    const unsigned holders = __ballot_sync(0xffffffffu, v == mx);
    if (holders == 0u) break;  // only NaN left
    if ((threadIdx.x & 31) == __ffs(holders) - 1) v = -INFINITY;
  }
  return kth;
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

// Warp 0 merges the warps' sorted lists lv/li[0, nw) (K entries each, best
// first) into the partial's k best, slots k..K-1 left empty: k rounds of a
// warp argmax over the lists' heads, lane l < nw reading list l.  Element
// indices are unique, so only the winner's lane advances.
template <int K>
__device__ __forceinline__ void merge_warp_lists(const float (*lv)[K], const int (*li)[K], int nw, int k,
                                                 SelPart* part) {
  const int lane = threadIdx.x & 31;
  const bool mine = lane < nw;
  int pos = 0;
  float ov = -INFINITY;
  int oi = INT_MAX;
  for (int j = 0; j < k; ++j) {
    float hv = mine && pos < K ? lv[lane][pos] : -INFINITY;
    int hi = mine && pos < K ? li[lane][pos] : INT_MAX;
    const int own = hi;
    warp_argmax(hv, hi);
    if (own == hi && hi != INT_MAX) ++pos;
    if (lane == j) {
      ov = hv;
      oi = hi;
    }
  }
  if (lane < K) {
    part->v[lane] = ov;
    part->i[lane] = oi;
  }
}

// Outputs of request req once p_s / id_s hold its rows' k probabilities and
// tokens (best first): topk_p_out, and for step 0 the first score block, else
// the path-score expansion scores_in[r] * p[r][j] (one fp32 multiply) and its
// top-k with parent offsets.  Called by every thread of the CTA after a
// __syncthreads (it may hold one more); sc_in is scores_in[req*k + lane/k]
// prefetched by warp 0 (read where k*k <= 32).
__device__ __forceinline__ void write_request(const SelectParams& a, int req, int rows_per_req,
                                              const float (*p_s)[kMaxK], const int (*id_s)[kMaxK], float sc_in) {
  const int k = a.k, kk = k * k, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
  } else if (kk <= 32) {
    if (w == 0) {
      // lane f: expansion f = (parent f / k, its j = f % k); rank among the
      // k*k by shuffles
      const bool on = lane < kk;
      const float ex = on ? __fmul_rn(sc_in, p_s[lane / k][lane % k]) : -INFINITY;
      const int id = on ? id_s[lane / k][lane % k] : 0;
      if (on) {
        a.score_blk[sb + lane] = ex;
        a.token_blk[sb + lane] = id;
      }
      int rank = 0;
#pragma unroll
      for (int g = 0; g < 32; ++g) {  // all lanes shuffle; lanes past k*k hold -inf
        const float o = __shfl_sync(0xffffffffu, ex, g);
        rank += (g < kk && better(o, g, ex, lane)) ? 1 : 0;
      }
      if (on && rank < k) {
        if (a.parent_blk) a.parent_blk[size_t(req) * a.parent_ld + rank] = lane + kk * (a.step - 1) + k;
        a.scores_out[size_t(req) * k + rank] = ex;
        a.next_ids[size_t(req) * k + rank] = id;
      }
    }
  } else {
    // more than 32 expansions: one a thread of the CTA (k*k <= 256); every
    // thread of the CTA takes this branch, so the barrier is the CTA's
    __shared__ float ex[kMaxK * kMaxK];
    for (int f = threadIdx.x; f < kk; f += blockDim.x) {
      ex[f] = __fmul_rn(a.scores_in[size_t(req) * k + f / k], p_s[f / k][f % k]);
      a.score_blk[sb + f] = ex[f];
      a.token_blk[sb + f] = id_s[f / k][f % k];
    }
    __syncthreads();
    for (int f = threadIdx.x; f < kk; f += blockDim.x) {
      int rank = 0;
      for (int g = 0; g < kk; ++g) rank += better(ex[g], g, ex[f], f);
      if (rank < k) {
        if (a.parent_blk) a.parent_blk[size_t(req) * a.parent_ld + rank] = f + kk * (a.step - 1) + k;
        a.scores_out[size_t(req) * k + rank] = ex[f];
        a.next_ids[size_t(req) * k + rank] = id_s[f / k][f % k];
      }
    }
  }
}

template <typename T, int K>
__global__ void __launch_bounds__(kThreads) select_kernel(SelectParams a) {
  // The chunk pass reads only the draft logits and this call's half of the
  // select's workspace area.  When the caller has allowed overlap and the
  // kernel before is the previous select (which uses the other half) or the
  // KV commit on the same workspace, the pass runs before waiting on it; only
  // the finalize, which reads the previous step's scores and writes this
  // step's outputs, waits.  Otherwise everything waits.
  if (!a.early) {
    pdl_wait();
    pdl_trigger();
  }
  const int row = blockIdx.y;
  const int chunk = blockIdx.x;
  const int rows_per_req = a.step ? a.k : 1;
  const int req = row / rows_per_req;
  const int begin = chunk * a.chunk_elems;
  const int end = min(a.V, begin + a.chunk_elems);
  const T* lrow = static_cast<const T*>(a.logits) + size_t(row) * a.V;
  const float c = 1.4426950408889634f / a.temperature;  // log2(e) / T

  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  constexpr int kCap = 512;
  __shared__ float cand_v[kCap];
  __shared__ int cand_i[kCap];
  __shared__ int cand_n;
  if (threadIdx.x == 0) cand_n = 0;  // first used after the barrier below

  // this thread's share of the chunk, in registers
  float f[kPerThread];
  load_share<T>(lrow, begin, end, a.vec_ok, f);
  float tm = -INFINITY;
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) tm = fmaxf(tm, f[j]);
  // The warp's max Mw, and the warp's sum of exp((x - Mw) / T): every exponent
  // is <= 0, and a warp with no element (past the row's end) sums to 0.
  const float Mw = warp_max(tm);
  const float mref = fmaxf(Mw, -3.0e38f);
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) s += fast_exp2((f[j] - mref) * c);
  s = warp_sum(s);
  __shared__ float wmax[kThreads / 32], wsum[kThreads / 32];
  __shared__ float tau_w[kThreads / 32];
  if (lane == 0) {
    wmax[w] = Mw;
    wsum[w] = s;
  }
  if (a.k > nw) {
    // more picks than warps: a warp's k-th largest thread maximum stands
    // for k distinct elements at or above it
    const float kth = warp_kth_largest(tm, a.k);
    if (lane == 0) tau_w[w] = kth;
  }
  __syncthreads();
  // Pruning bound tau: no element below it can be among the chunk's k best.
  // With k <= warps it is the k-th largest warp maximum (k distinct
  // elements, in k different warps, reach it): each warp ranks the nw warp
  // maxima by shuffles, with no dependent rounds.
  float tau = -INFINITY;
  if (a.k <= nw) {
    const float v = lane < nw ? wmax[lane] : -INFINITY;
    int rank = 0;
    for (int q = 0; q < nw; ++q) {
      const float o = __shfl_sync(0xffffffffu, v, q);
      rank += (o > v || (o == v && q < lane)) ? 1 : 0;
    }
    const unsigned at = __ballot_sync(0xffffffffu, lane < nw && rank == a.k - 1);
    tau = __shfl_sync(0xffffffffu, v, at ? __ffs(at) - 1 : 0);
    if (!at) tau = -INFINITY;
  } else {
    for (int q = 0; q < nw; ++q) tau = fmaxf(tau, tau_w[q]);
  }
  // Common case: few elements reach tau; they are appended to a shared
  // candidate list and ranked.  Heavy ties can overflow the list, and then
  // every thread keeps its own sorted top-K and the lists are merged (the
  // general path).
  if (tm >= tau) {
#pragma unroll
    for (int j = 0; j < kPerThread; ++j)
      if (f[j] >= tau) {
        const int pos = atomicAdd(&cand_n, 1);
        if (pos < kCap) {
          cand_v[pos] = f[j];
          cand_i[pos] = share_index<T>(begin, a.vec_ok, j);
        }
      }
  }
  __syncthreads();
  SelPart* part = reinterpret_cast<SelPart*>(a.partials) + size_t(row) * a.chunks + chunk;
  const int ncand = cand_n;
  if (w == nw - 1) {
    // the chunk's softmax statistics from the warps' (Mw, sum): one warp
    const float wm = lane < nw ? wmax[lane] : -INFINITY;
    const float M = fmaxf(warp_max(wm), -3.0e38f);
    const float t = lane < nw ? wsum[lane] * exp2f((fmaxf(wm, -3.0e38f) - M) * c) : 0.f;
    const float S = warp_sum(t);
    if (lane == 0) {
      part->m = M;
      part->s = S;
    }
  }
  if (ncand <= int(blockDim.x)) {
    // one candidate per thread: its rank among the candidates (a strict
    // order: no NaN passes the threshold, indices are distinct) is its slot
    if (int(threadIdx.x) < ncand) {
      const float v = cand_v[threadIdx.x];
      const int ix = cand_i[threadIdx.x];
      int rank = 0;
      for (int u = 0; u < ncand; ++u) rank += better(cand_v[u], cand_i[u], v, ix);
      if (rank < K) {
        part->v[rank] = v;
        part->i[rank] = ix;
      }
    } else if (int(threadIdx.x) < K) {  // fewer candidates than K: empty slots
      part->v[threadIdx.x] = -INFINITY;
      part->i[threadIdx.x] = INT_MAX;
    }
  } else if (ncand <= kCap) {
    if (w == 0) {
      for (int r = 0; r < K; ++r) {
        float v = -INFINITY;
        int ix = INT_MAX, slot = -1;
        for (int t = lane; t < ncand; t += 32)
          if (cand_i[t] != INT_MIN && better(cand_v[t], cand_i[t], v, ix)) {
            v = cand_v[t];
            ix = cand_i[t];
            slot = t;
          }
        float bv = v;
        int bi = ix;
        warp_argmax(bv, bi);
        if (slot >= 0 && bv == v && bi == ix) cand_i[slot] = INT_MIN;  // taken
        __syncwarp();
        if (lane == 0) {
          part->v[r] = bv;
          part->i[r] = bi;
        }
      }
    }
  } else {
    TopList<K> top;
    top.init();
    if (tm >= tau) {
#pragma unroll
      for (int j = 0; j < kPerThread; ++j)
        if (f[j] >= tau) top.push(f[j], share_index<T>(begin, a.vec_ok, j));
    }
    __shared__ float lv[kThreads / 32][K];
    __shared__ int li[kThreads / 32][K];
    warp_merge<K>(top, lv[w], li[w]);
    __syncthreads();
    if (w == 0) merge_warp_lists<K>(lv, li, nw, a.k, part);
  }

  if (!arrive_last(a.counters + req, uint32_t(rows_per_req * a.chunks))) return;
  if (a.early) {
    pdl_wait();
    pdl_trigger();
  }

  // ---- finalize request `req` ----
  // One warp per row: lane l holds chunk l's (m, s) and sorted top-K list in
  // registers (every load issued before any is used: one round trip through
  // L2, the partials were written by other CTAs); k rounds of a tournament
  // over the lanes' list heads give the row's k best, lane j keeping the
  // j-th.  Then the path step of the request.
  const int k = a.k, kk = k * k;
  // this lane's parent score for the path step (lane f < k*k: parent f / k)
  const float sc_in = (a.step > 0 && w == 0 && lane < kk) ? a.scores_in[size_t(req) * k + lane / k] : 0.f;
  __shared__ float p_s[kMaxK][kMaxK];
  __shared__ int id_s[kMaxK][kMaxK];
  for (int r = w; r < rows_per_req; r += nw) {
    const int grow = req * rows_per_req + r;
    const SelPart* pr = reinterpret_cast<const SelPart*>(a.partials) + size_t(grow) * a.chunks;
    const bool has = lane < a.chunks;
    float hv[K], pm = -3.0e38f, psum = 0.f;
    int hi[K];
    if constexpr (K % 4 == 0) {
#pragma unroll
      for (int q = 0; q < K; q += 4) {
        const float4 v4 = has ? __ldcg(reinterpret_cast<const float4*>(&pr[lane].v[q]))
                              : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        const int4 i4 = has ? __ldcg(reinterpret_cast<const int4*>(&pr[lane].i[q]))
                            : make_int4(INT_MAX, INT_MAX, INT_MAX, INT_MAX);
        hv[q] = v4.x, hv[q + 1] = v4.y, hv[q + 2] = v4.z, hv[q + 3] = v4.w;
        hi[q] = i4.x, hi[q + 1] = i4.y, hi[q + 2] = i4.z, hi[q + 3] = i4.w;
      }
    } else {
#pragma unroll
      for (int q = 0; q < K; ++q) {
        hv[q] = has ? __ldcg(&pr[lane].v[q]) : -INFINITY;
        hi[q] = has ? __ldcg(&pr[lane].i[q]) : INT_MAX;
      }
    }
    if (has) {
      const float2 ms = __ldcg(reinterpret_cast<const float2*>(&pr[lane].m));
      pm = ms.x;
      psum = ms.y;
    }
    // softmax denominator of the whole row
    const float M = warp_max(pm);
    const float S = warp_sum(psum * exp2f((pm - M) * c));
    float myv = -INFINITY;
    int myi = INT_MAX;
    for (int j = 0; j < k; ++j) {
      float bv = hv[0];
      int bi = hi[0];
      warp_argmax(bv, bi);
      if (hi[0] == bi && bi != INT_MAX) {  // this lane's head won: next entry up
#pragma unroll
        for (int q = 0; q + 1 < K; ++q) {
          hv[q] = hv[q + 1];
          hi[q] = hi[q + 1];
        }
        hv[K - 1] = -INFINITY;
        hi[K - 1] = INT_MAX;
      }
      if (lane == j) {
        myv = bv;
        myi = bi;
      }
    }
    // p = exp((x - M) / T) / S; x - M is exact for bf16 logits, so fp32 expf
    // (about 1 ulp) keeps p within 1e-6 relative of the fp64 value
    const float invS = 1.f / S;  // one more rounding than a division: within 1 ulp
    if (lane < k) {
      p_s[r][lane] = expf((myv - M) / a.temperature) * invS;
      id_s[r][lane] = myi;
    }
  }
  __syncthreads();
  write_request(a, req, rows_per_req, p_s, id_s, sc_in);
  counter_reset(a.counters + req);
}


// ---------------------------------------------------------------------------
// The streaming select: the logits streaming pass (stream_records.cu: one
// record, maximum and exp sum, a group of a lane's 8 vectors of a unit), then
// select_finalize_kernel, one CTA a row.  From the row's records: the row
// maximum M, the denominator S = sum of s 2^((g - M) c); theta = the k-th
// largest of the CTA's thread maxima, each the best of that thread's groups
// (k distinct groups reach it, so the k best elements all do); the groups
// that reach theta are reloaded, a vector a thread, and their elements that
// reach it ranked by warp 0 (the k best elements lie in the k best groups).
// The row's k probabilities and tokens are stored; the CTA whose row is the
// last of its request to arrive runs the path step of the request.

// The value of rank k - 1 among the nt (<= 32 NS) slots top[0, nt) by (value
// desc, slot asc), for every lane of the warp: lane l ranks slots l + 32 i by
// counting, in one pass over the slots.
template <int NS>
__device__ __forceinline__ float kth_slot(const float* top, int nt, int k) {
  const int lane = threadIdx.x & 31;
  float v[NS];
  int rank[NS];
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    v[i] = lane + 32 * i < nt ? top[lane + 32 * i] : -INFINITY;
    rank[i] = 0;
  }
#pragma unroll 8
  for (int o = 0; o < nt; ++o) {
    const float u = top[o];
#pragma unroll
    for (int i = 0; i < NS; ++i) rank[i] += (u > v[i] || (u == v[i] && o < lane + 32 * i)) ? 1 : 0;
  }
  float th = -INFINITY;
#pragma unroll
  for (int i = 0; i < NS; ++i)
    if (lane + 32 * i < nt && rank[i] == k - 1) th = v[i];
  return warp_max(th);  // (one slot has rank k - 1)
}

// The request step after the streaming kernel: one CTA a row.
constexpr int kFinalizeThreads = 256;
constexpr int kFinalizeWarps = kFinalizeThreads / 32;
constexpr int kElemCap = 32 * 32;    // gathered elements the request step ranks directly

template <typename T>
__global__ void __launch_bounds__(kFinalizeThreads, 1) select_finalize_kernel(SelectParams a) {
  constexpr int E = LogitTraits<T>::kVec;
  // the row's group maxima by flat record index f (an empty group as NaN,
  // which no comparison takes), then the gathered groups' indices
  extern __shared__ float gval[];
  __shared__ float p_s[kMaxK][kMaxK];
  __shared__ int id_s[kMaxK][kMaxK];
  __shared__ float el_v[kElemCap];               // the gathered elements (value, index in the row)
  __shared__ int el_i[kElemCap];
  __shared__ float cand_v[kStreamCand];
  __shared__ int cand_i[kStreamCand];
  __shared__ float s_m[kFinalizeWarps], s_s[kFinalizeWarps];
  __shared__ float s_top[kFinalizeWarps * kMaxK];  // each warp's k best lane maxima: [w * k + j]
  __shared__ int s_n, s_ne;
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x, tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int k = a.k, kk = k * k;
  const int rows_per_req = a.step ? k : 1;
  const int req = row / rows_per_req;
  const long long rowU = a.V / E;
  const float2* rec = reinterpret_cast<const float2*>(a.partials);
  const uint4* logits = static_cast<const uint4*>(a.logits);
  float2* best = reinterpret_cast<float2*>(a.partials + align256(size_t(a.stream_nb) * 2 * 32 * sizeof(float2)));
  const unsigned lanes_below = (1u << lane) - 1u;
  if (row == 0 && tid == 0) *a.queue = 0u;  // the streaming grid is done with the queue: ready for the next call
  const long long rs = (long long)row * rowU, rend = rs + rowU;  // the row's vectors
  const int uf = int(rs / kUnitVecs), ul = int((rend - 1) / kUnitVecs);
  const int F = (ul - uf + 1) * 32;  // the row's records: f = (unit - uf) * 32 + lane'
  const int par = row & 1;
  int* gsel = reinterpret_cast<int*>(gval + F);
  if (tid == 0) {
    s_n = 0;
    s_ne = 0;
  }
  // the path step's parent score (lane f < k*k of warp 0: parent f / k), loaded
  // now so that it is at hand at the end
  const float sc_in = (a.step > 0 && w == 0 && lane < kk) ? a.scores_in[size_t(req) * k + lane / k] : 0.f;

  // one pass over the records (thread tid: f = tid + 256 m, eight loads in
  // flight): the maxima to shared memory, this thread's maximum and its sum
  // relative to it; the CTA's sum in fp64
  const ExpScale sc(a.temperature);
  RecSum rsum;
  for (int f0 = 0; f0 < F; f0 += 8 * kFinalizeThreads) {
    float2 r[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int f = f0 + q * kFinalizeThreads + tid;
      r[q] = f < F ? __ldcg(&rec[stream_slot(uf + f / 32, par, f % 32)]) : make_float2(NAN, -1.f);
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int f = f0 + q * kFinalizeThreads + tid;
      if (f < F) gval[f] = r[q].y >= 0.f ? r[q].x : NAN;
      if (r[q].y > 0.f) rsum.add(r[q].x, r[q].y, sc);  // (s = 0: the group is all -inf)
    }
  }
  // one barrier for the row maximum M, the denominator S and theta: per warp
  // its maximum, its sum relative to it and its k best lane maxima
  {
    const float wm = warp_max(rsum.m);
    const float ws = warp_sum(rsum.rel(wm, sc));
    // the lanes' maxima sorted descending across the warp (a bitonic sort,
    // 15 exchange steps): lane j < k then holds the j-th largest
    float v = rsum.m;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, v, stride);
        const bool desc = (lane & size) == 0, lower = (lane & stride) == 0;
        v = desc == lower ? fmaxf(v, o) : fminf(v, o);
      }
    if (lane < k) s_top[w * k + lane] = v;
    if (lane == 0) {
      s_m[w] = wm;
      s_s[w] = ws;
    }
  }
  __syncthreads();
  float M = -INFINITY;
  for (int i = 0; i < kFinalizeWarps; ++i) M = fmaxf(M, s_m[i]);
  float S = 0.f;
  for (int i = 0; i < kFinalizeWarps; ++i)
    if (s_s[i] > 0.f) S += s_s[i] * fast_exp2(sc.times(s_m[i] - M));
  // theta = the k-th largest lane maximum of the CTA (the k best are among
  // the warps' k best; k distinct groups reach it, so the row's k best
  // elements all do): each warp ranks the nt = 8 k slots by counting, by
  // (value desc, slot asc) -- lane l holds slots l + 32 i, one pass over the
  // slots -- and takes the value of rank k - 1
  const int nt = kFinalizeWarps * k;
  const float theta = nt <= 32 ? kth_slot<1>(s_top, nt, k) : nt <= 64 ? kth_slot<2>(s_top, nt, k) : kth_slot<4>(s_top, nt, k);
  // the groups that reach theta, listed (gsel: one shared atomic a warp),
  // then reloaded a vector a thread (every load of the phase in flight at
  // once); their elements that reach theta
  {
    const int nm = (F + kFinalizeThreads - 1) / kFinalizeThreads;
    int cnt = 0;
    for (int m = 0; m < nm; ++m) {
      const int f = tid + m * kFinalizeThreads;
      cnt += (f < F && gval[f] >= theta) ? 1 : 0;
    }
    int inc = cnt;  // inclusive scan over the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    int base = 0;
    if (lane == 31) base = atomicAdd(&s_n, inc);
    int pos = __shfl_sync(0xffffffffu, base, 31) + inc - cnt;
    for (int m = 0; m < nm; ++m) {
      const int f = tid + m * kFinalizeThreads;
      if (f < F && gval[f] >= theta) gsel[pos++] = f;
    }
  }
  __syncthreads();
  const int ng = s_n;
  for (int i = tid; i < ng * kStreamVpt; i += kFinalizeThreads) {
    const int f = gsel[i / kStreamVpt], u = i % kStreamVpt;
    const long long gv = (long long)(uf + f / 32) * kUnitVecs + f % 32 + u * 32;
    if (gv >= rs && gv < rend) {
      const uint4 x = __ldcg(logits + gv);
#pragma unroll
      for (int q = 0; q < E; ++q) {
        const float v = VecOps<T>::at(x, q);
        if (v >= theta) {
          const int pos = atomicAdd(&s_ne, 1);
          if (pos < kElemCap) {
            el_v[pos] = v;
            el_i[pos] = int((gv - rs) * E) + q;
          }
        }
      }
    }
  }
  __syncthreads();
  if (w == 0) {
    const int ne = s_ne;
    float lv_r = -INFINITY;  // lane j < k: entry j of the row's k best
    int li_r = INT_MAX;
    if (ne <= 32) {
      // one element a lane, ranked by counting the elements ahead of it
      // (indices are unique); the entries of rank < k to their slots
      const float v = lane < ne ? el_v[lane] : -INFINITY;
      const int i = lane < ne ? el_i[lane] : INT_MAX;
      int rank = 0;
      for (int o = 0; o < ne; ++o) rank += better(el_v[o], el_i[o], v, i) ? 1 : 0;
      if (lane < ne && rank < k) {
        cand_v[rank] = v;
        cand_i[rank] = i;
      }
      __syncwarp();
      if (lane < k && lane < ne) {
        lv_r = cand_v[lane];
        li_r = cand_i[lane];
      }
    } else if (ne <= kElemCap) {
      // k rounds of a warp argmax over the gathered elements (lane l: entries l, l + 32, ...)
      uint32_t taken = 0;
      const int per = (ne - lane + 31) / 32;
      for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = INT_MAX, bm = -1;
        for (int m = 0; m < per; ++m) {
          const int e2 = lane + 32 * m;
          if (!(taken & (1u << m)) && better(el_v[e2], el_i[e2], bv, bi)) {
            bv = el_v[e2];
            bi = el_i[e2];
            bm = m;
          }
        }
        const int own = bi;
        warp_argmax(bv, bi);
        if (own == bi && bi != INT_MAX) taken |= 1u << bm;
        if (lane == j) {
          lv_r = bv;
          li_r = bi;
        }
      }
    } else {
      // more than kElemCap elements reach theta (values tied at the cut): the
      // listed groups again, through the candidate buffer, 32 at a time
      float cut = theta;
      int ncand = 0;
      for (int g0 = 0; g0 < ng; g0 += 32) {
        const int gi = g0 + lane;
        uint4 xv[kStreamVpt];
        uint32_t vin = 0;
        long long gv0 = 0;
        if (gi < ng) {
          const int f = gsel[gi];
          gv0 = (long long)(uf + f / 32) * kUnitVecs + f % 32;
#pragma unroll
          for (int u = 0; u < kStreamVpt; ++u) {
            const long long gv = gv0 + u * 32;
            if (gv >= rs && gv < rend) {
              vin |= 1u << u;
              xv[u] = __ldcg(logits + gv);
            }
          }
        }
#pragma unroll
        for (int u = 0; u < kStreamVpt; ++u) {
          uint32_t bits = 0;
          if (vin & (1u << u)) {
#pragma unroll
            for (int q = 0; q < E; ++q) bits |= (VecOps<T>::at(xv[u], q) >= cut ? 1u : 0u) << q;
          }
          for (;;) {  // one element a lane a round
            const unsigned mask = __ballot_sync(0xffffffffu, bits != 0u);
            if (!mask) break;
            const int nnew = __popc(mask);
            if (ncand + nnew > kStreamCand) {
              stream_merge_candidates(cand_v, cand_i, ncand, k, lv_r, li_r);
              ncand = 0;
              if (__shfl_sync(0xffffffffu, li_r, k - 1) != INT_MAX)  // the list holds k: a tighter bound
                cut = fmaxf(cut, __shfl_sync(0xffffffffu, lv_r, k - 1));
            }
            if (bits) {
              const int q = __ffs(bits) - 1;
              bits &= bits - 1u;
              const int pos = ncand + __popc(mask & lanes_below);
              cand_v[pos] = vec_elem<T>(xv[u], q);
              cand_i[pos] = int((gv0 + u * 32 - rs) * E) + q;
            }
            ncand += nnew;
          }
        }
      }
      if (ncand) stream_merge_candidates(cand_v, cand_i, ncand, k, lv_r, li_r);
    }
    const float invS = 1.f / S;
    if (lane < k) best[size_t(row) * kMaxK + lane] = make_float2(expf((lv_r - M) / a.temperature) * invS, __int_as_float(li_r));
  }
  // the last row of the request to arrive runs the path step
  if (!arrive_last(a.counters + req, uint32_t(rows_per_req))) return;
  for (int i = tid; i < rows_per_req * k; i += kFinalizeThreads) {
    const float2 v = __ldcg(&best[(size_t(req) * rows_per_req + i / k) * kMaxK + i % k]);
    p_s[i / k][i % k] = v.x;
    id_s[i / k][i % k] = __float_as_int(v.y);
  }
  __syncthreads();
  write_request(a, req, rows_per_req, p_s, id_s, sc_in);
  counter_reset(a.counters + req);
}

// Dynamic shared memory of the request step: a row's record maxima and indices.
inline size_t finalize_smem(int V, int vec) {
  const long long rowU = V / vec;
  return 2 * size_t(rowU / kUnitVecs + 2) * 32 * sizeof(float);
}

template <typename T>
cudaError_t launch_stream(const SelectParams& p, cudaStream_t stream) {
  StreamRecParams r{};
  r.logits = p.logits;
  r.rows = p.rows;
  r.V = p.V;
  r.temperature = p.temperature;
  r.temperatures = nullptr;
  r.rows_per_temp = 1;
  r.nu = p.stream_nb;
  r.rec = reinterpret_cast<float2*>(p.partials);
  r.queue = p.queue;
  r.early = p.early;
  if (launch_stream_records(r, p.stream_ctas, p.dtype, stream) != SPEC_OK) return cudaErrorLaunchFailure;
  const size_t fsmem = finalize_smem(p.V, LogitTraits<T>::kVec);
  cudaError_t e = cudaFuncSetAttribute(select_finalize_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(fsmem));
  if (e != cudaSuccess) return e;
  return launch_pdl(select_finalize_kernel<T>, dim3(p.rows), dim3(kFinalizeThreads), fsmem, stream, p);
}

template <typename T>
int launch_t(const SelectParams& p, cudaStream_t stream) {
  dim3 grid(p.chunks, p.rows);
  const int K = p.k <= 1 ? 1 : p.k <= 2 ? 2 : p.k <= 4 ? 4 : p.k <= 8 ? 8 : 16;
  cudaError_t e = cudaSuccess;
  if (p.stream_ctas > 0) {
    e = launch_stream<T>(p, stream);
    return e == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
  }
  switch (K) {
    case 1: e = launch_pdl(select_kernel<T, 1>, grid, dim3(kThreads), 0, stream, p); break;
    case 2: e = launch_pdl(select_kernel<T, 2>, grid, dim3(kThreads), 0, stream, p); break;
    case 4: e = launch_pdl(select_kernel<T, 4>, grid, dim3(kThreads), 0, stream, p); break;
    case 8: e = launch_pdl(select_kernel<T, 8>, grid, dim3(kThreads), 0, stream, p); break;
    default: e = launch_pdl(select_kernel<T, 16>, grid, dim3(kThreads), 0, stream, p); break;
  }
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
}

}  // namespace

size_t select_partial_bytes(int rows, int chunks) { return align256(size_t(rows) * chunks * sizeof(SelPart)); }

StreamGeometry select_stream_geometry(long rows, int V, int vec, int sms) {
  StreamGeometry g = stream_geometry(rows, V, vec, sms);
  if (g.ctas > 0) g.bytes += align256(size_t(rows) * kMaxK * sizeof(float2));  // the rows' k best
  return g;
}

int launch_select_topk(const SelectParams& p, cudaStream_t stream) {
  return p.dtype == SPEC_F32 ? launch_t<float>(p, stream) : launch_t<uint16_t>(p, stream);
}

}  // namespace spec
