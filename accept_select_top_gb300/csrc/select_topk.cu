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
// The streaming select: two kernels.
//
// select_stream_kernel reads the step's logits once.  The flattened [rows, V]
// logits (16-byte vectors, rows contiguous) are cut into units of 256 vectors
// (4 KB).  Every warp of the persistent grid (two CTAs a SM) works on its own:
// it takes units in pairs, the first two pairs fixed by its index, the rest
// from a queue (an atomic counter, asked two pairs ahead so that its latency
// stays hidden), so that warps the memory serves faster take more.  Lane l
// holds vectors l, l + 32, ..., l + 224 of a unit in a private ring of 16-byte
// cp.async copies, three units deep, and waits for its own copies with
// cp.async.wait_group: no barrier and no wait on another warp anywhere.  A
// lane's vectors of one unit inside one row form a group; for each group it
// writes one record: the group's maximum g and s = sum over the group of
// 2^((x - g) c) (s = -1 where the lane has no vector in that row of the unit).
// A unit spans at most two rows, so the record slot is (unit, row parity,
// lane).
//
// select_finalize_kernel (one CTA a row) reads a row's records: the row
// maximum M is the largest g, the denominator S = sum of s 2^((g - M) c) (fp64
// accumulation).  The row's k best elements lie in its k best groups by
// (maximum desc, index of the maximum asc): were an element among the k best
// in a group outside them, the k groups ahead of its group would each hold an
// element that ranks before it.  So theta = the largest over warps of the
// warp's k-th largest group maximum (k distinct groups reach it); the groups
// whose maximum reaches theta are gathered, and their elements that reach it
// merged into the k best by warp 0 (k rounds of a warp argmax).  The row's k
// probabilities and tokens are stored; the CTA whose row is the last of its
// request to arrive runs the path step of the request.

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

template <typename T>
__global__ void __launch_bounds__(kStreamThreads, kStreamPerSm) select_stream_kernel(SelectParams a) {
  constexpr int E = LogitTraits<T>::kVec;  // elements per 16-byte vector
  // ring: vector u of stage s of lane l of warp w at [((w * stages + s) * Vpt + u) * 32 + l]
  extern __shared__ __align__(16) uint4 ring[];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const unsigned rowU = unsigned(a.V / E);
  const unsigned U = unsigned(a.rows) * rowU;  // (the host keeps it below 2^31)
  const int nu = a.stream_nb;                  // units in all
  const float c = 1.4426950408889634f / a.temperature;
  const uint4* src = static_cast<const uint4*>(a.logits);
  float2* rec = reinterpret_cast<float2*>(a.partials);
  uint4* wring = ring + w * (kStreamStages * kUnitVecs) + lane;

  // Without overlap: wait for the grid before, then let the request step
  // launch (it waits for this grid to finish before it reads a record).  With
  // overlap the reads start at once and a lane waits before its first record
  // write.
  bool waited = !a.early;
  if (waited) pdl_wait();
  pdl_trigger();

  // iteration j works on unit 2 * pair(j / 2) + (j & 1); pc = pair(j / 2), pn
  // = pair(j / 2 + 1); lane 0 holds the queue's answer for pair(j / 2 + 2)
  const int NW = gridDim.x * kStreamWarps, gw = blockIdx.x * kStreamWarps + w;
  int pc = gw, pn = gw + NW, pending = 0;
  if (lane == 0) pending = 2 * NW + int(atomicAdd(a.queue, 1u));
  auto issue = [&](int j, int unit) {  // stage j % 3 <- unit (an empty group past the last unit)
    if (unit < nu) {
      uint4* st = wring + (unsigned(j) % kStreamStages) * kUnitVecs;
      const unsigned o0 = unsigned(unit) * kUnitVecs + lane;
      if (o0 + (kStreamVpt - 1) * 32 < U) {  // the whole unit exists
#pragma unroll
        for (int u = 0; u < kStreamVpt; ++u) stream_cp16(st + u * 32, src + o0 + u * 32, 16u);
      } else {
#pragma unroll
        for (int u = 0; u < kStreamVpt; ++u) {
          const unsigned o = o0 + u * 32;
          const bool ok = o < U;
          stream_cp16(st + u * 32, ok ? src + o : src, ok ? 16u : 0u);
        }
      }
    }
    stream_commit();
  };
  issue(0, 2 * pc);
  issue(1, 2 * pc + 1);
  for (int j = 0;; ++j) {
    if (j >= 2 && !(j & 1)) {  // a new pair
      pc = pn;
      pn = __shfl_sync(0xffffffffu, pending, 0);
      if (lane == 0) pending = 2 * NW + int(atomicAdd(a.queue, 1u));
    }
    const int unit = 2 * pc + (j & 1);
    if (unit >= nu) break;  // (a warp's units only grow: every later one is past the end too)
    issue(j + 2, 2 * pn + (j & 1));
    stream_wait_group<kStreamStages - 1>();  // this lane's copies of unit j have landed
    const uint4* st = wring + (unsigned(j) % kStreamStages) * kUnitVecs;
    const unsigned b0 = unsigned(unit) * kUnitVecs;
    const unsigned b1 = b0 + kUnitVecs < U ? b0 + kUnitVecs : U;
    unsigned row = b0 / rowU;
    unsigned cur = b0;
    while (cur < b1) {  // the unit's vectors, one row at a time (at most two rows)
      const unsigned re = (row + 1) * rowU;
      const unsigned seg = b1 < re ? b1 : re;
      uint4 x[kStreamVpt];
      bool any = true;  // the group holds at least one vector
      if (cur == b0 && seg == b0 + kUnitVecs) {  // the common case: the whole unit
#pragma unroll
        for (int u = 0; u < kStreamVpt; ++u) x[u] = st[u * 32];
      } else {  // vectors outside the segment read as -inf
        any = false;
#pragma unroll
        for (int u = 0; u < kStreamVpt; ++u) {
          const unsigned o = b0 + u * 32 + lane;
          const bool in = o >= cur && o < seg;
          any = any || in;
          x[u] = in ? st[u * 32] : VecOps<T>::neg_inf();
        }
      }
      typename VecMax<T>::type gm = VecMax<T>::of(x[0]);
#pragma unroll
      for (int u = 1; u < kStreamVpt; ++u) gm = VecMax<T>::comb(gm, VecMax<T>::of(x[u]));
      const float g = VecMax<T>::value(gm);
      // (g = -inf: no element, or all -inf: every term is 0)
      const float s = batch_exp_sum<T>(x, c, g > -INFINITY ? g * c : 0.f);
      if (!waited) {
        pdl_wait();
        waited = true;
      }
      __stcg(&rec[stream_slot(unit, row & 1, lane)], make_float2(g, any ? s : -1.f));
      cur = seg;
      ++row;
    }
  }
  stream_wait_group<0>();  // no copy of this lane is left in flight (the last groups are empty)
}

// The request step after the streaming kernel: one CTA a row.
constexpr int kFinalizeThreads = 256;
constexpr int kFinalizeWarps = kFinalizeThreads / 32;
constexpr int kFinalizeMaxPer = 32;  // records a thread of the request step takes at most
constexpr int kElemCap = 32 * 32;    // gathered elements the request step ranks directly

// Maximum / sum over the CTA (scratch: a slot a warp); every thread gets the
// result.  Both end with a barrier, so the scratch may be reused.
__device__ __forceinline__ float block_max_f(float v, float* scratch) {
  v = warp_max(v);
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = scratch[0];
  for (int i = 1; i < kFinalizeWarps; ++i) r = fmaxf(r, scratch[i]);
  __syncthreads();
  return r;
}
__device__ __forceinline__ float block_sum_f(float v, float* scratch) {
  v = warp_sum(v);
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = 0.f;
  for (int i = 0; i < kFinalizeWarps; ++i) r += scratch[i];
  __syncthreads();
  return r;
}

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
  __shared__ float s_f[kFinalizeWarps];
  __shared__ int s_n, s_ne;
  __shared__ float s_vk;
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x, tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int k = a.k, kk = k * k;
  const int rows_per_req = a.step ? k : 1;
  const int req = row / rows_per_req;
  const long long rowU = a.V / E;
  const float c = 1.4426950408889634f / a.temperature;
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

  // one pass over the records (thread tid: f = tid + 256 m, eight loads in
  // flight): the maxima to shared memory, this thread's maximum and its sum
  // relative to it (fp32: a chain of at most 32 additions here, 8 across the CTA)
  float tm = -INFINITY, ts = 0.f;
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
      if (r[q].y > 0.f) {  // (s = 0: the group is all -inf)
        if (r[q].x > tm) {
          ts = ts * fast_exp2((tm - r[q].x) * c) + r[q].y;
          tm = r[q].x;
        } else {
          ts += r[q].y * fast_exp2((r[q].x - tm) * c);
        }
      }
    }
  }
  const float M = block_max_f(tm, s_f);
  const float S = block_sum_f(ts > 0.f ? ts * fast_exp2((tm - M) * c) : 0.f, s_f);
  // theta: the largest over warps of the k-th largest of the lanes' best group
  // maxima (k distinct groups reach it)
  {
    float bv = -INFINITY;
    for (int m = tid; m < F; m += kFinalizeThreads) bv = fmaxf(bv, gval[m]);
    float wk = -INFINITY;
    for (int j = 0; j < k; ++j) {
      float wv = bv;
      int wi = lane;
      warp_argmax(wv, wi);
      if (lane == wi) bv = -INFINITY;
      wk = wv;
    }
    if (lane == 0) s_f[w] = wk;
  }
  __syncthreads();
  float theta = -INFINITY;
  for (int i = 0; i < kFinalizeWarps; ++i) theta = fmaxf(theta, s_f[i]);
  // the groups that reach theta
  for (int m = 0; m < (F + kFinalizeThreads - 1) / kFinalizeThreads; ++m) {
    const int f = tid + m * kFinalizeThreads;
    const bool take = f < F && gval[f] >= theta;
    const unsigned mask = __ballot_sync(0xffffffffu, take);
    if (mask) {
      int base = 0;
      if (lane == 0) base = atomicAdd(&s_n, __popc(mask));
      base = __shfl_sync(0xffffffffu, base, 0);
      if (take) gsel[base + __popc(mask & lanes_below)] = f;
    }
  }
  __syncthreads();
  // v_k, the row's k-th largest group maximum, among the gathered (warp 0: k
  // rounds of a warp argmax; lane l takes gathered entries l, l + 32, ...)
  if (w == 0) {
    const int n0 = s_n;
    const int per = (n0 - lane + 31) / 32;
    uint64_t taken = 0;
    float vk = -INFINITY;
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int bi = INT_MAX, bm = -1;
      for (int m = 0; m < per && m < 64; ++m) {
        const int f = gsel[lane + 32 * m];
        if (!(taken & (1ull << m)) && better(gval[f], f, bv, bi)) {
          bv = gval[f];
          bi = f;
          bm = m;
        }
      }
      const int own = bi;
      warp_argmax(bv, bi);
      if (own == bi && bi != INT_MAX) taken |= 1ull << bm;
      vk = bv;
    }
    if (lane == 0) {
      // more than 2048 gathered (values tied at theta): theta itself stays the cut
      s_vk = n0 <= 32 * 64 ? vk : theta;
      s_n = 0;
    }
  }
  __syncthreads();
  const float vk = s_vk;  // k distinct groups reach it: the k best elements all do
  // the groups that reach v_k (every group with that maximum: a tie keeps them all)
  for (int m = 0; m < (F + kFinalizeThreads - 1) / kFinalizeThreads; ++m) {
    const int f = tid + m * kFinalizeThreads;
    const bool take = f < F && gval[f] >= vk;
    const unsigned mask = __ballot_sync(0xffffffffu, take);
    if (mask) {
      int base = 0;
      if (lane == 0) base = atomicAdd(&s_n, __popc(mask));
      base = __shfl_sync(0xffffffffu, base, 0);
      if (take) gsel[base + __popc(mask & lanes_below)] = f;
    }
  }
  __syncthreads();
  const int ng = s_n;
  // their elements that reach v_k: a vector a thread
  for (int i = tid; i < ng * kStreamVpt; i += kFinalizeThreads) {
    const int f = gsel[i / kStreamVpt], u = i % kStreamVpt;
    const long long gv = (long long)(uf + f / 32) * kUnitVecs + f % 32 + u * 32;
    if (gv >= rs && gv < rend) {
      const uint4 x = __ldcg(logits + gv);
#pragma unroll
      for (int q = 0; q < E; ++q) {
        const float v = VecOps<T>::at(x, q);
        if (v >= vk) {
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
    if (ne <= kElemCap) {
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
      // more than kElemCap elements reach v_k (values tied at the cut): the
      // groups again, through the candidate buffer, 32 at a time
      float theta = vk;
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
            for (int q = 0; q < E; ++q) bits |= (VecOps<T>::at(xv[u], q) >= theta ? 1u : 0u) << q;
          }
          for (;;) {  // one element a lane a round
            const unsigned mask = __ballot_sync(0xffffffffu, bits != 0u);
            if (!mask) break;
            const int nnew = __popc(mask);
            if (ncand + nnew > kStreamCand) {
              stream_merge_candidates(cand_v, cand_i, ncand, k, lv_r, li_r);
              ncand = 0;
              if (__shfl_sync(0xffffffffu, li_r, k - 1) != INT_MAX)  // the list holds k: a tighter bound
                theta = fmaxf(theta, __shfl_sync(0xffffffffu, lv_r, k - 1));
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
  const float sc_in = (a.step > 0 && w == 0 && lane < kk) ? a.scores_in[size_t(req) * k + lane / k] : 0.f;
  for (int i = tid; i < rows_per_req * k; i += kFinalizeThreads) {
    const float2 v = __ldcg(&best[(size_t(req) * rows_per_req + i / k) * kMaxK + i % k]);
    p_s[i / k][i % k] = v.x;
    id_s[i / k][i % k] = __float_as_int(v.y);
  }
  __syncthreads();
  write_request(a, req, rows_per_req, p_s, id_s, sc_in);
  counter_reset(a.counters + req);
}

// The streaming split: G CTAs (kStreamPerSm a SM) over the units.  None where
// a row is shorter than a unit (a unit then could span more than two rows),
// where the request step's threads would take more than kFinalizeMaxPer
// records, or where the vector count reaches 2^31.
StreamGeometry stream_geometry(long rows, int V, int vec, int sms) {
  const long long rowU = V / vec;
  if (rows < 1 || rowU < kUnitVecs) return StreamGeometry{0, 0, 0};
  if ((rowU / kUnitVecs + 2) * 32 > (long long)kFinalizeMaxPer * kFinalizeThreads) return StreamGeometry{0, 0, 0};
  const long long U = rows * rowU;
  if (U >= (1LL << 31) - kUnitVecs) return StreamGeometry{0, 0, 0};
  const long long nu = (U + kUnitVecs - 1) / kUnitVecs;
  long long G = (long long)kStreamPerSm * sms;
  const long long need = (nu + 2 * kStreamWarps - 1) / (2 * kStreamWarps);  // CTAs whose warps get a pair each
  if (G > need) G = need;
  if (G < 1) G = 1;
  const size_t bytes = align256(size_t(nu) * 2 * 32 * sizeof(float2)) + align256(size_t(rows) * kMaxK * sizeof(float2));
  return StreamGeometry{int(G), int(nu), bytes};
}

// Dynamic shared memory of the request step: a row's record maxima and indices.
inline size_t finalize_smem(int V, int vec) {
  const long long rowU = V / vec;
  return 2 * size_t(rowU / kUnitVecs + 2) * 32 * sizeof(float);
}

template <typename T>
cudaError_t launch_stream(const SelectParams& p, cudaStream_t stream) {
  constexpr size_t smem = size_t(kStreamWarps) * kStreamStages * kUnitVecs * 16;
  cudaError_t e = cudaFuncSetAttribute(select_stream_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  e = launch_pdl(select_stream_kernel<T>, dim3(p.stream_ctas), dim3(kStreamThreads), smem, stream, p);
  if (e != cudaSuccess) return e;
  const size_t fsmem = finalize_smem(p.V, LogitTraits<T>::kVec);
  e = cudaFuncSetAttribute(select_finalize_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(fsmem));
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

StreamGeometry select_stream_geometry(long rows, int V, int vec, int sms) { return stream_geometry(rows, V, vec, sms); }

int launch_select_topk(const SelectParams& p, cudaStream_t stream) {
  return p.dtype == SPEC_F32 ? launch_t<float>(p, stream) : launch_t<uint16_t>(p, stream);
}

}  // namespace spec
