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
  } else if (w == 0 && kk <= 32) {
    // lane f: expansion f = (parent f / k, its j = f % k); rank among the k*k
    // by shuffles
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
  } else {
    // more than 32 expansions: one a thread of the CTA (k*k <= 256)
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
// The streaming select: one persistent pass over the step's logits.  The
// flattened [rows, V] logits (16-byte vectors, rows contiguous) are cut into G
// equal contiguous ranges, one per CTA (three CTAs a SM).  Thread t of a CTA
// takes the range's vectors t, t + 256, t + 512, ... through a private ring of
// 16-byte cp.async copies, kStreamStages batches of kStreamVpt vectors deep,
// and waits for its own copies with cp.async.wait_group: no barrier and no
// polling while streaming.  Each thread keeps an online (max, sum of exp) of
// the row piece (the part of one row inside the CTA's range), rescaled once a
// batch.
//
// The k best are kept a warp at a time, behind a bound that only rises:
//   - every batch, the warp's lanes' running maxima give one: split the 32
//     lanes into k' groups (k' = k rounded up to a power of two); the smallest
//     group maximum is at most the k-th largest of k' distinct elements, so at
//     most the piece's k-th value (two shuffle trees);
//   - the warp's own k-th value once its list holds k;
//   - theta, the CTA's: the largest bound any warp has published (atomicMax
//     on an order key).
// An element below the bound cannot be among the piece's k best.  Elements
// that reach it are appended to the warp's candidate buffer (one ballot a
// batch finds the rare batch that has any; then one element a lane a round,
// positions by prefix counts of the ballot).  A full buffer is merged into the
// list (lane j < k holds entry j) by k rounds of a warp argmax.
//
// Only where a row piece ends does the CTA meet: warp 0 merges the warps'
// lists into the piece's partial (max, sum, k best), and the CTA whose piece
// is the last of a request to arrive merges the request's pieces and runs the
// path step, as the chunked kernel does.

constexpr int kStreamThreads = 256;
constexpr int kStreamWarps = kStreamThreads / 32;
constexpr int kStreamPerSm = 2;                   // CTAs a SM (the ring and the registers allow two)
constexpr int kStreamStages = 3;                  // batches in flight a thread
constexpr int kStreamVpt = 8;                     // 16-byte vectors a batch
constexpr int kStreamBatchVecs = kStreamVpt * kStreamThreads;  // vectors a CTA batch
constexpr int kStreamCand = 32;                   // candidate elements a warp buffers (one a lane)

// 16-byte global -> shared copy; src_bytes 0 writes zeros and reads nothing.
__device__ __forceinline__ void stream_cp16(void* dst, const void* src, uint32_t src_bytes) {
  const uint32_t d = uint32_t(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void stream_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void stream_wait_group() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// The owner CTA of vector u when U vectors are cut into G ranges
// [c*U/G, (c+1)*U/G).
__device__ __forceinline__ int stream_owner(long long u, long long U, int G) {
  return int(((u + 1) * G - 1) / U);
}

// Number of row pieces (ranges touching the row) of row r.
__device__ __forceinline__ int stream_pieces(int r, long long rowU, long long U, int G) {
  return stream_owner((r + 1) * rowU - 1, U, G) - stream_owner(r * rowU, U, G) + 1;
}

// Merge of one row's pieces by one warp (at most 32 pieces, one a lane: the
// host caps the grid so): lane q reads piece q's (m, s) and sorted list.  Lane
// j < k ends with the row's j-th best (value desc, index asc); every lane with
// the row's max M and sum S (of exp2((x - M) c)).
template <int K>
__device__ __forceinline__ void merge_row(const SelPart* pr, int count, int k, float c, float& myv, int& myi,
                                          float& M, float& S) {
  const int lane = threadIdx.x & 31;
  const bool has = lane < count;
  float hv[K], pm = -3.0e38f, psum = 0.f;
  int hi[K];
#pragma unroll
  for (int q = 0; q < K; ++q) {
    hv[q] = has ? __ldcg(&pr[lane].v[q]) : -INFINITY;
    hi[q] = has ? __ldcg(&pr[lane].i[q]) : INT_MAX;
  }
  if (has) {
    const float2 ms = __ldcg(reinterpret_cast<const float2*>(&pr[lane].m));
    pm = ms.x;
    psum = ms.y;
  }
  M = warp_max(pm);
  S = warp_sum(psum * exp2f((pm - M) * c));
  myv = -INFINITY;
  myi = INT_MAX;
  for (int j = 0; j < k; ++j) {
    float bv = hv[0];
    int bi = hi[0];
    warp_argmax(bv, bi);
    if (hi[0] == bi && bi != INT_MAX) {
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
}

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

template <typename T, int K>
__global__ void __launch_bounds__(kStreamThreads, kStreamPerSm) select_stream_kernel(SelectParams a) {
  constexpr int E = LogitTraits<T>::kVec;  // elements per 16-byte vector
  // ring: vector u of batch slot s of thread t at [(s * kStreamVpt + u) * 256 + t]
  extern __shared__ __align__(16) uint4 ring[];
  __shared__ float cand_v[kStreamWarps][kStreamCand];  // a warp's candidate elements
  __shared__ int cand_i[kStreamWarps][kStreamCand];    // their element indices in the row
  __shared__ uint32_t s_theta;  // order key of the CTA's lower bound on the piece's k-th value
  __shared__ float wmax[kStreamWarps], ws2[kStreamWarps];
  __shared__ float lv[kStreamWarps][K];
  __shared__ int li[kStreamWarps][K];
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, nw = kStreamWarps;
  const int G = gridDim.x;
  const long long rowU = a.V / E;
  const long long U = (long long)a.rows * rowU;
  const long long u_lo = (long long)blockIdx.x * U / G, u_hi = (long long)(blockIdx.x + 1) * U / G;
  const int n_vec = int(u_hi - u_lo);  // vectors of this CTA (a range is far below 2^31 vectors)
  const float c = 1.4426950408889634f / a.temperature;
  const uint4* src = static_cast<const uint4*>(a.logits) + u_lo;  // this CTA's first vector
  const unsigned lanes_below = (1u << lane) - 1u;
  // the lane-maxima bound uses K groups of 32 / K lanes (K, a power of two, is at least k)
  constexpr int kGroupLanes = 32 / K;

  bool waited = false;
  if (!a.early) {
    pdl_wait();
    pdl_trigger();
    waited = true;
  }
  if (tid == 0) s_theta = 0u;  // the smallest key: no bound yet
  __syncthreads();

  // batch bb of this thread: offsets (bb * Vpt + u) * 256 + t of the range
  auto issue = [&](int bb) {
    uint4* slot = ring + (unsigned(bb) % kStreamStages) * (kStreamVpt * kStreamThreads) + tid;
    const int o0 = bb * kStreamBatchVecs + tid;
    if (o0 + (kStreamVpt - 1) * kStreamThreads < n_vec) {  // the whole batch lies in the range
#pragma unroll
      for (int u = 0; u < kStreamVpt; ++u) stream_cp16(slot + u * kStreamThreads, src + o0 + u * kStreamThreads, 16u);
    } else {
#pragma unroll
      for (int u = 0; u < kStreamVpt; ++u) {
        const int o = o0 + u * kStreamThreads;
        const bool ok = o < n_vec;
        stream_cp16(slot + u * kStreamThreads, ok ? src + o : src, ok ? 16u : 0u);
      }
    }
    stream_commit();
  };
  const int nbatch = (n_vec + kStreamBatchVecs - 1) / kStreamBatchVecs;
#pragma unroll
  for (int q = 0; q < kStreamStages - 1; ++q) issue(q);

  float m = -3.0e38f, ssum = 0.f;  // this thread's online softmax of the current row piece
  float lv_r = -INFINITY;          // lane j < k: entry j of the warp's k best of the piece
  int li_r = INT_MAX;
  float thr_w = -INFINITY;         // the warp's bound (lane maxima, own list); warp-uniform
  float thr_pub = -INFINITY;       // the last bound this warp published
  int ncand = 0;                   // candidates in the warp's buffer (warp-uniform)
  int row = int(u_lo / rowU);
  int re = int((long long)(row + 1) * rowU - u_lo);  // end of the current row, as an offset of the range
  for (int bb = 0; bb < nbatch; ++bb) {
    issue(bb + kStreamStages - 1);  // (past the range: an empty group, so the count stays exact)
    stream_wait_group<kStreamStages - 1>();  // this thread's copies of batch bb have landed
    const uint4* slot = ring + (unsigned(bb) % kStreamStages) * (kStreamVpt * kStreamThreads);
    const int b0 = bb * kStreamBatchVecs;
    const int b1 = b0 + kStreamBatchVecs < n_vec ? b0 + kStreamBatchVecs : n_vec;
    int cur = b0;
    while (cur < b1) {  // the batch's vectors, one row piece at a time (uniform over the CTA)
      const int seg = b1 < re ? b1 : re;
      uint4 x[kStreamVpt];
      uint32_t vin;  // bit u: vector u lies in the segment (the others read as -inf)
      if (cur == b0 && seg == b0 + kStreamBatchVecs) {  // the common case: the whole batch
        vin = (1u << kStreamVpt) - 1u;
#pragma unroll
        for (int u = 0; u < kStreamVpt; ++u) x[u] = slot[u * kStreamThreads + tid];
      } else {
        vin = 0u;
#pragma unroll
        for (int u = 0; u < kStreamVpt; ++u) {
          const int o = b0 + u * kStreamThreads + tid;
          x[u] = VecOps<T>::neg_inf();
          if (o >= cur && o < seg) {
            vin |= 1u << u;
            x[u] = slot[u * kStreamThreads + tid];
          }
        }
      }
      typename VecMax<T>::type vm[kStreamVpt];  // each vector's maximum
#pragma unroll
      for (int u = 0; u < kStreamVpt; ++u) vm[u] = VecMax<T>::of(x[u]);
      typename VecMax<T>::type bmv = vm[0];
#pragma unroll
      for (int u = 1; u < kStreamVpt; ++u) bmv = VecMax<T>::comb(bmv, vm[u]);
      const float bm = VecMax<T>::value(bmv);
      if (bm > m) {
        ssum *= fast_exp2((m - bm) * c);
        m = bm;
      }
      // (m still the sentinel: every term is 0 anyway; -inf entries give 0)
      ssum += batch_exp_sum<T>(x, c, m > -1.0e30f ? m * c : 0.f);
      // the lane-maxima bound: max within groups of 32 / K lanes, min across the K groups
      float gb = m > -1.0e30f ? m : -INFINITY;
#pragma unroll
      for (int o = 1; o < kGroupLanes; o <<= 1) gb = fmaxf(gb, __shfl_xor_sync(0xffffffffu, gb, o));
#pragma unroll
      for (int o = kGroupLanes; o < 32; o <<= 1) gb = fminf(gb, __shfl_xor_sync(0xffffffffu, gb, o));
      thr_w = fmaxf(thr_w, gb);
      if (thr_w > thr_pub) {  // warp-uniform
        if (lane == 0) atomicMax(&s_theta, order_key(thr_w));
        thr_pub = thr_w;
      }
      // a stale (lower) theta only lets more through; key 0 reads as NaN, which fmaxf drops
      const float thr = fmaxf(key_value(*reinterpret_cast<volatile uint32_t*>(&s_theta)), thr_w);
      if (__ballot_sync(0xffffffffu, vin != 0u && bm >= thr)) {  // the rare batch with a candidate
        uint32_t vmask = 0;  // bit u: vector u holds an element that reaches the bound
        if (bm >= thr) {
#pragma unroll
          for (int u = 0; u < kStreamVpt; ++u)
            if ((vin & (1u << u)) && VecMax<T>::value(vm[u]) >= thr) vmask |= 1u << u;
        }
        const int rbase = int(u_lo - ((long long)row * rowU));  // vector o of the range is vector o + rbase of the row
        while (__any_sync(0xffffffffu, vmask != 0u)) {  // one candidate vector a lane a round
          uint32_t bits = 0;  // bit q: element q of vector u reaches the bound
          int u = 0;
          if (vmask) {
            u = __ffs(vmask) - 1;
            vmask &= vmask - 1u;
            const uint4 xv = slot[u * kStreamThreads + tid];  // (the batch is still in its slot)
#pragma unroll
            for (int q = 0; q < E; ++q) bits |= (VecOps<T>::at(xv, q) >= thr ? 1u : 0u) << q;
          }
          for (;;) {  // one element a lane a round
            const unsigned mask = __ballot_sync(0xffffffffu, bits != 0u);
            if (!mask) break;
            const int nnew = __popc(mask);
            if (ncand + nnew > kStreamCand) {
              stream_merge_candidates(cand_v[w], cand_i[w], ncand, a.k, lv_r, li_r);
              ncand = 0;
              if (__shfl_sync(0xffffffffu, li_r, a.k - 1) != INT_MAX) {  // the list holds k: its k-th
                thr_w = fmaxf(thr_w, __shfl_sync(0xffffffffu, lv_r, a.k - 1));
                if (thr_w > thr_pub) {
                  if (lane == 0) atomicMax(&s_theta, order_key(thr_w));
                  thr_pub = thr_w;
                }
              }
            }
            if (bits) {
              const int q = __ffs(bits) - 1;
              bits &= bits - 1u;
              const int pos = ncand + __popc(mask & lanes_below);
              cand_v[w][pos] = vec_elem<T>(slot[u * kStreamThreads + tid], q);
              cand_i[w][pos] = (b0 + u * kStreamThreads + tid + rbase) * E + q;
            }
            ncand += nnew;
          }
        }
      }
      cur = seg;
      if (seg == re || seg == n_vec) {
        // ---- end of a row piece: its partial ----
        if (ncand) stream_merge_candidates(cand_v[w], cand_i[w], ncand, a.k, lv_r, li_r);
        const float Mw = warp_max(m);
        const float Sw = warp_sum(ssum * exp2f((m - Mw) * c));
        if (lane == 0) {
          wmax[w] = Mw;
          ws2[w] = Sw;
        }
        if (lane < K) {  // lanes k..K-1 hold no entry
          lv[w][lane] = lv_r;
          li[w][lane] = li_r;
        }
        __syncthreads();
        if (w == 0) {
          if (!waited) {  // overlap: the partials are written only once the grid before is done
            pdl_wait();
            pdl_trigger();
            waited = true;
          }
          const int r0 = stream_owner((long long)row * rowU, U, G);
          SelPart* part = reinterpret_cast<SelPart*>(a.partials) + size_t(row) * a.stream_pmax + (blockIdx.x - r0);
          const float wm = lane < nw ? wmax[lane] : -3.0e38f;
          const float Mc = warp_max(wm);
          const float Sc = warp_sum(lane < nw ? ws2[lane] * exp2f((wm - Mc) * c) : 0.f);
          if (lane == 0) {
            part->m = Mc;
            part->s = Sc;
          }
          merge_warp_lists<K>(lv, li, nw, a.k, part);
        }
        m = -3.0e38f;
        ssum = 0.f;
        lv_r = -INFINITY;
        li_r = INT_MAX;
        thr_w = -INFINITY;
        thr_pub = -INFINITY;
        ncand = 0;
        if (tid == 0) s_theta = 0u;
        __syncthreads();  // lv / li are read and the bound is reset before the next piece
        re += int(rowU);
        ++row;
      }
    }
  }
  stream_wait_group<0>();  // no copy of this CTA is left in flight (the last groups are empty)
}

// The request step after the streaming select: one CTA a request, one warp a
// row of it merging the row's pieces (merge_row), then the path step
// (write_request).  Launched after the streaming kernel; it waits for that
// grid before it reads a partial.
constexpr int kFinalizeThreads = 32 * kMaxK;

template <int K>
__global__ void __launch_bounds__(kFinalizeThreads) select_finalize_kernel(SelectParams a) {
  __shared__ float p_s[kMaxK][kMaxK];
  __shared__ int id_s[kMaxK][kMaxK];
  pdl_wait();
  pdl_trigger();
  const int req = blockIdx.x, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int k = a.k, kk = k * k;
  const int rows_per_req = a.step ? k : 1;
  const int vec = a.dtype == SPEC_F32 ? 4 : 8;
  const long long rowU = a.V / vec;
  const long long U = (long long)a.rows * rowU;
  const int G = a.stream_ctas;
  const float c = 1.4426950408889634f / a.temperature;
  const float sc_in = (a.step > 0 && w == 0 && lane < kk) ? a.scores_in[size_t(req) * k + lane / k] : 0.f;
  if (w < rows_per_req) {
    const int grow = req * rows_per_req + w;
    const SelPart* pr = reinterpret_cast<const SelPart*>(a.partials) + size_t(grow) * a.stream_pmax;
    float myv, M, S;
    int myi;
    merge_row<K>(pr, stream_pieces(grow, rowU, U, G), k, c, myv, myi, M, S);
    const float invS = 1.f / S;
    if (lane < k) {
      p_s[w][lane] = expf((myv - M) / a.temperature) * invS;
      id_s[w][lane] = myi;
    }
  }
  __syncthreads();
  write_request(a, req, rows_per_req, p_s, id_s, sc_in);
}

// The split the streaming select uses: G CTAs (kStreamPerSm a SM, at least 64
// vectors each) and the pieces a row can have.
struct StreamSplit {
  int ctas, pmax;
};
inline StreamSplit stream_split(long rows, int V, int vec, int sms) {
  const long long rowU = V / vec;
  const long long U = rows * rowU;
  long long G = (long long)kStreamPerSm * sms;
  if (G > U / 64) G = U / 64;
  if (G < 1) G = 1;
  auto pmax_of = [&](long long g) {
    auto owner = [&](long long u) { return ((u + 1) * g - 1) / U; };
    long long pm = 1;
    for (long r = 0; r < rows; ++r) {
      const long long p = owner((r + 1) * rowU - 1) - owner(r * rowU) + 1;
      if (p > pm) pm = p;
    }
    return pm;
  };
  // at most 32 pieces a row, so that a warp merges a row one piece a lane
  long long pmax = pmax_of(G);
  while (pmax > 32 && G > 1) {
    G = G * 31 / 32;
    pmax = pmax_of(G);
  }
  return StreamSplit{int(G), int(pmax)};
}

template <typename T, int K>
cudaError_t launch_stream(const SelectParams& p, cudaStream_t stream) {
  constexpr size_t smem = size_t(kStreamStages) * kStreamVpt * kStreamThreads * 16;
  cudaError_t e =
      cudaFuncSetAttribute(select_stream_kernel<T, K>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  e = launch_pdl(select_stream_kernel<T, K>, dim3(p.stream_ctas), dim3(kStreamThreads), smem, stream, p);
  if (e != cudaSuccess) return e;
  const int requests = p.step ? p.rows / p.k : p.rows;
  return launch_pdl(select_finalize_kernel<K>, dim3(requests), dim3(kFinalizeThreads), 0, stream, p);
}

template <typename T>
int launch_t(const SelectParams& p, cudaStream_t stream) {
  dim3 grid(p.chunks, p.rows);
  const int K = p.k <= 1 ? 1 : p.k <= 2 ? 2 : p.k <= 4 ? 4 : p.k <= 8 ? 8 : 16;
  cudaError_t e = cudaSuccess;
  if (p.stream_ctas > 0) {
    switch (K) {
      case 1: e = launch_stream<T, 1>(p, stream); break;
      case 2: e = launch_stream<T, 2>(p, stream); break;
      case 4: e = launch_stream<T, 4>(p, stream); break;
      case 8: e = launch_stream<T, 8>(p, stream); break;
      default: e = launch_stream<T, 16>(p, stream); break;
    }
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
  const StreamSplit s = stream_split(rows, V, vec, sms);
  return StreamGeometry{s.ctas, s.pmax};
}

int launch_select_topk(const SelectParams& p, cudaStream_t stream) {
  return p.dtype == SPEC_F32 ? launch_t<float>(p, stream) : launch_t<uint16_t>(p, stream);
}

}  // namespace spec
