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

// Outputs of request req once p_s / id_s hold its rows' k probabilities and
// tokens (best first): topk_p_out, and for step 0 the first score block, else
// the path-score expansion scores_in[r] * p[r][j] (one fp32 multiply) and its
// top-k with parent offsets.  Called by every thread of the CTA after a
// __syncthreads; sc_in is scores_in[req*k + lane/k] prefetched by warp 0.
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
  } else if (w == 0) {
    __shared__ float ex[kMaxK * kMaxK];
    for (int f = lane; f < kk; f += 32) {
      const float sin = f < 32 ? sc_in : a.scores_in[size_t(req) * k + f / k];
      ex[f] = __fmul_rn(sin, p_s[f / k][f % k]);
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
    if (w == 0) {
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
    }
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
// The streaming select: one persistent pass over the step's logits at HBM
// rate.  The flattened [rows, V] logits (16-byte vectors, rows contiguous) are
// cut into G equal contiguous ranges, one per CTA (G = a few CTAs per SM).  A
// CTA streams its range in 16 KB tiles through a ring of kStreamStages shared
// buffers filled by bulk asynchronous copies (cp.async.bulk, completion on an
// mbarrier), so several tiles are in flight while one is reduced.  Each
// thread keeps an online (max, sum of exp) of its elements; the CTA keeps the
// running k best of the row piece and its k-th value theta: only elements at
// or above theta are ranked (the first tile of a piece seeds theta from the
// k-th largest warp maximum).  A row piece (the part of one row inside one
// CTA's range) ends with one partial (max, sum, k best); the CTA whose piece
// is the last of a request to arrive merges the request's pieces and runs the
// path step, as the chunked kernel does.

constexpr int kStreamThreads = 256;
constexpr int kStreamStages = 4;
constexpr int kStreamTileBytes = 16384;
constexpr int kStreamTileVecs = kStreamTileBytes / 16;           // 1024 vectors a tile
constexpr int kStreamVpt = kStreamTileVecs / kStreamThreads;      // 4 vectors a thread a tile
constexpr int kStreamCap = kStreamThreads - kMaxK;                // ranked candidates + the running list <= 256
constexpr long long kStreamWaitCycles = 4000000000ll;              // ~2 s: bound of every mbarrier wait

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return uint32_t(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ bool stream_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(20000u)
      : "memory");
  return ok != 0;
}
// false once the bound passes (the copy never landed)
__device__ __forceinline__ bool stream_wait(uint32_t bar, uint32_t parity) {
  if (stream_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (clock64() - t0 < kStreamWaitCycles)
    if (stream_try_wait(bar, parity)) return true;
  return false;
}

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

template <typename T, int K>
__global__ void __launch_bounds__(kStreamThreads, K > 8 ? 2 : 3) select_stream_kernel(SelectParams a) {
  constexpr int E = LogitTraits<T>::kVec;  // elements per 16-byte vector
  extern __shared__ __align__(128) unsigned char ring[];  // kStreamStages tiles
  __shared__ __align__(8) uint64_t full[kStreamStages];
  __shared__ float cand_v[kStreamThreads];
  __shared__ int cand_i[kStreamThreads];
  __shared__ int cand_n[1];  // buffered candidates since the last merge
  __shared__ float best_v[K];
  __shared__ int best_i[K];
  __shared__ int best_n;
  __shared__ float s_theta;
  __shared__ float wmax[kStreamThreads / 32], tau_w[kStreamThreads / 32], ws2[kStreamThreads / 32];
  __shared__ float lv[kStreamThreads / 32][K];
  __shared__ int li[kStreamThreads / 32][K];
  __shared__ float p_s[kMaxK][kMaxK];
  __shared__ int id_s[kMaxK][kMaxK];
  __shared__ int s_abort;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, nw = kStreamThreads / 32;
  const int G = gridDim.x;
  const long long rowU = a.V / E;
  const long long U = (long long)a.rows * rowU;
  const long long u_lo = (long long)blockIdx.x * U / G, u_hi = (long long)(blockIdx.x + 1) * U / G;
  const int rows_per_req = a.step ? a.k : 1;
  const float c = 1.4426950408889634f / a.temperature;
  const unsigned char* src = static_cast<const unsigned char*>(a.logits);

  bool waited = false;
  if (!a.early) {
    pdl_wait();
    pdl_trigger();
    waited = true;
  }
  if (tid == 0) {
    for (int s = 0; s < kStreamStages; ++s)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&full[s])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    cand_n[0] = 0;
    best_n = 0;
    s_theta = -INFINITY;
    s_abort = 0;
  }
  __syncthreads();

  // Tiles of this CTA, in order: [u, min(u + tile, row end, u_hi)).  The
  // producer (thread 0) runs kStreamStages tiles ahead of the consumers; both
  // track the end of their current row instead of dividing.
  const long long first_row_end = (u_lo / rowU + 1) * rowU;
  auto tile_end = [&](long long u, long long re) {
    long long e = u + kStreamTileVecs;
    if (e > re) e = re;
    if (e > u_hi) e = u_hi;
    return e;
  };
  long long pu = u_lo, p_re = first_row_end;  // producer cursor and its row's end
  int issued = 0;
  auto issue = [&]() {  // thread 0: the next tile into stage issued % stages
    if (pu >= u_hi) return;
    const long long e = tile_end(pu, p_re);
    const uint32_t bytes = uint32_t((e - pu) * 16);
    const int s = issued % kStreamStages;
    const uint32_t bar = smem_addr(&full[s]);
    const uint32_t dst = smem_addr(ring + size_t(s) * kStreamTileBytes);
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src + pu * 16), "r"(bytes), "r"(bar)
                 : "memory");
    pu = e;
    if (pu == p_re) p_re += rowU;
    ++issued;
  };
  if (tid == 0)
    for (int s = 0; s < kStreamStages; ++s) issue();

  float m = -3.0e38f, ssum = 0.f;  // this thread's online softmax of the current row piece
  long long cu = u_lo, c_re = first_row_end;  // consumer cursor and its row's end
  int row = int(first_row_end / rowU) - 1;
  int j = 0;                                   // tile number
  while (cu < u_hi) {
    const long long e = tile_end(cu, c_re);
    const int nvec = int(e - cu);
    const bool piece_end = e == c_re || e >= u_hi;
    const int s = j % kStreamStages;
    const bool ok = stream_wait(smem_addr(&full[s]), uint32_t((j / kStreamStages) & 1));
    // this thread's vectors of the tile (a tile that never landed is read as is:
    // in bounds, and the CTA stops below)
    const uint4* tv = reinterpret_cast<const uint4*>(ring + size_t(s) * kStreamTileBytes);
    uint4 x[kStreamVpt];
    float vm[kStreamVpt];
#pragma unroll
    for (int i = 0; i < kStreamVpt; ++i) {
      const int v = tid + i * kStreamThreads;
      x[i] = v < nvec ? tv[v] : VecOps<T>::neg_inf();
      vm[i] = VecOps<T>::vmax(x[i]);
    }
    float tm = vm[0];
#pragma unroll
    for (int i = 1; i < kStreamVpt; ++i) tm = fmaxf(tm, vm[i]);
    if (tm > m) {
      ssum *= fast_exp2((m - tm) * c);
      m = tm;
    }
    // m * c of a thread that has seen only padding (m still the sentinel)
    // would overflow: its elements are -inf, any finite offset gives 0
    const float mc = m > -1.0e30f ? m * c : 0.f;
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < kStreamVpt; ++i)
#pragma unroll
      for (int q = 0; q < E; ++q) acc += fast_exp2(fmaf(VecOps<T>::at(x[i], q), c, -mc));
    ssum += acc;
    // Candidates gather across tiles against the theta of the last merge:
    // elements above it (an element equal to theta comes after theta's own
    // element in the row, so it cannot rank before it), or, while the piece
    // has fewer than k best (theta = -inf), at or above the tile's k-th
    // largest warp maximum.  Only the vectors whose maximum passes are
    // scanned.
    float thr = s_theta;
    const bool seed = thr == -INFINITY;
    if (seed) {
      const float Mw = warp_max(tm);
      if (lane == 0) wmax[w] = Mw;
      if (a.k > nw) {
        const float kth = warp_kth_largest(tm, a.k);
        if (lane == 0) tau_w[w] = kth;
      }
      __syncthreads();
      if (a.k <= nw) {
        const float v = lane < nw ? wmax[lane] : -INFINITY;
        int rank = 0;
        for (int q = 0; q < nw; ++q) {
          const float o = __shfl_sync(0xffffffffu, v, q);
          rank += (o > v || (o == v && q < lane)) ? 1 : 0;
        }
        const unsigned at = __ballot_sync(0xffffffffu, lane < nw && rank == a.k - 1);
        thr = at ? __shfl_sync(0xffffffffu, v, __ffs(at) - 1) : -INFINITY;
      } else {
        thr = -INFINITY;
        for (int q = 0; q < nw; ++q) thr = fmaxf(thr, tau_w[q]);
      }
    }
    const int ebase = int((cu - (c_re - rowU)) * E);  // element index (in its row) of the tile's first element
#pragma unroll
    for (int i = 0; i < kStreamVpt; ++i) {
      const int v = tid + i * kStreamThreads;
      if (v < nvec && (seed ? vm[i] >= thr : vm[i] > thr)) {
#pragma unroll
        for (int q = 0; q < E; ++q) {
          const float f = VecOps<T>::at(x[i], q);
          if (seed ? f >= thr : f > thr) {
            const int pos = atomicAdd(&cand_n[0], 1);
            if (pos < kStreamCap) {
              cand_v[pos] = f;
              cand_i[pos] = ebase + v * E + q;
            }
          }
        }
      }
    }
    if (__syncthreads_or(!ok)) {  // (A) a copy never landed: stop cleanly
      if (tid == 0) {
        raise_error(a.error, SPEC_DEV_TIMEOUT);
        for (int q = j; q < issued; ++q)  // wait (bounded) for this CTA's copies in flight
          stream_wait(smem_addr(&full[q % kStreamStages]), uint32_t((q / kStreamStages) & 1));
      }
      __syncthreads();
      return;
    }
    // Merge the gathered candidates into the running list after a seed tile
    // (to set theta), when the buffer is half full, and at the end of the
    // piece.  The count is cleared after the merge's first barrier (every
    // thread has read it by then) and the next pushes follow barrier (B).
    const int n = cand_n[0];
    if (n > 0 && (seed || piece_end || n > kStreamCap / 2)) {
      const int nb = best_n;
      if (n <= kStreamCap) {
        // rank the candidates with the running list: one entry a thread
        if (tid < nb) {
          cand_v[n + tid] = best_v[tid];
          cand_i[n + tid] = best_i[tid];
        }
        __syncthreads();
        if (tid == 0) cand_n[0] = 0;
        const int total = n + nb;
        if (tid < total) {
          const float v = cand_v[tid];
          const int ix = cand_i[tid];
          int rank = 0;
          for (int u = 0; u < total; ++u) rank += better(cand_v[u], cand_i[u], v, ix);
          if (rank < a.k) {
            best_v[rank] = v;
            best_i[rank] = ix;
            if (rank == a.k - 1) s_theta = v;
          }
        }
        if (tid == 0) {
          best_n = total < a.k ? total : a.k;
          if (total < a.k) s_theta = -INFINITY;
        }
      } else {
        // The buffer overflowed (heavy ties).  Rank together: the running
        // list, the buffered entries of earlier tiles (index below this
        // tile's), and the k best of this tile's elements that pass, kept by
        // every thread and merged by every warp.
        TopList<K> top;
        top.init();
#pragma unroll
        for (int i = 0; i < kStreamVpt; ++i) {
          const int v = tid + i * kStreamThreads;
#pragma unroll
          for (int q = 0; q < E; ++q) {
            const float f = VecOps<T>::at(x[i], q);
            if (v < nvec && (seed ? f >= thr : f > thr)) top.push(f, ebase + v * E + q);
          }
        }
        warp_merge<K>(top, lv[w], li[w]);
        __syncthreads();
        if (tid == 0) cand_n[0] = 0;
        auto entry = [&](int u, float& v, int& ix) -> bool {
          if (u < nb) {
            v = best_v[u];
            ix = best_i[u];
            return true;
          }
          u -= nb;
          if (u < kStreamCap) {
            v = cand_v[u];
            ix = cand_i[u];
            return ix < ebase;
          }
          u -= kStreamCap;
          v = lv[u / K][u % K];
          ix = li[u / K][u % K];
          return ix != INT_MAX;
        };
        const int total = nb + kStreamCap + nw * K;  // <= 16 + 240 + 128
        float rv[2];
        int ri[2], rr[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int t0 = tid + q * kStreamThreads;
          rr[q] = INT_MAX;
          float v;
          int ix;
          if (t0 < total && entry(t0, v, ix)) {
            int rank = 0;
            for (int u = 0; u < total; ++u) {
              float uv;
              int ui;
              if (entry(u, uv, ui)) rank += better(uv, ui, v, ix);
            }
            rv[q] = v;
            ri[q] = ix;
            rr[q] = rank;
          }
        }
        __syncthreads();  // every read of the list is done
        int real = 0;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          if (rr[q] != INT_MAX) ++real;
          if (rr[q] < a.k) {
            best_v[rr[q]] = rv[q];
            best_i[rr[q]] = ri[q];
          }
        }
        real = __syncthreads_count(real > 0 ? 1 : 0) + __syncthreads_count(real > 1 ? 1 : 0);
        if (tid == 0) {
          const int kept = real < a.k ? real : a.k;
          best_n = kept;
          s_theta = kept == a.k ? best_v[a.k - 1] : -INFINITY;
        }
      }
      __syncthreads();  // (B)
    }
    if (tid == 0) {  // the stage of tile j is free again: every thread has read it (barrier above)
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue();
    }
    cu = e;
    ++j;

    // ---- end of a row piece: its partial, and the request's finalize ----
    if (piece_end) {
      const float Mw = warp_max(m);
      const float Sw = warp_sum(ssum * exp2f((m - Mw) * c));
      if (lane == 0) {
        wmax[w] = Mw;
        ws2[w] = Sw;
      }
      __syncthreads();
      const int r0 = int(stream_owner((long long)row * rowU, U, G));
      SelPart* part = reinterpret_cast<SelPart*>(a.partials) + size_t(row) * a.stream_pmax + (blockIdx.x - r0);
      if (w == 0) {
        const float wm = lane < nw ? wmax[lane] : -3.0e38f;
        const float Mc = warp_max(wm);
        const float Sc = warp_sum(lane < nw ? ws2[lane] * exp2f((wm - Mc) * c) : 0.f);
        if (lane == 0) {
          part->m = Mc;
          part->s = Sc;
        }
        if (lane < K) {
          const bool has = lane < best_n;
          part->v[lane] = has ? best_v[lane] : -INFINITY;
          part->i[lane] = has ? best_i[lane] : INT_MAX;
        }
      }
      const int req = row / rows_per_req;
      uint32_t target = 0;
      for (int r = req * rows_per_req; r < (req + 1) * rows_per_req; ++r)
        target += uint32_t(stream_pieces(r, rowU, U, G));
      const bool last = arrive_last(a.counters + req, target);  // (syncs: the partial is written before)
      if (tid == 0) {
        best_n = 0;
        s_theta = -INFINITY;
      }
      m = -3.0e38f;
      ssum = 0.f;
      if (last) {
        if (!waited) {
          pdl_wait();
          pdl_trigger();
          waited = true;
        }
        const int k = a.k, kk = k * k;
        const float sc_in = (a.step > 0 && w == 0 && lane < kk) ? a.scores_in[size_t(req) * k + lane / k] : 0.f;
        for (int r = w; r < rows_per_req; r += nw) {
          const int grow = req * rows_per_req + r;
          const SelPart* pr = reinterpret_cast<const SelPart*>(a.partials) + size_t(grow) * a.stream_pmax;
          float myv, M, S;
          int myi;
          merge_row<K>(pr, stream_pieces(grow, rowU, U, G), k, c, myv, myi, M, S);
          const float invS = 1.f / S;
          if (lane < k) {
            p_s[r][lane] = expf((myv - M) / a.temperature) * invS;
            id_s[r][lane] = myi;
          }
        }
        __syncthreads();
        write_request(a, req, rows_per_req, p_s, id_s, sc_in);
        counter_reset(a.counters + req);
      }
      __syncthreads();  // the piece state is reset before the next tile
      if (cu == c_re) {
        c_re += rowU;
        ++row;
      }
    }
  }
}

// The split the streaming select uses: G CTAs (at most 3 a SM, at least 64
// vectors each) and the pieces a row can have.
struct StreamSplit {
  int ctas, pmax;
};
inline StreamSplit stream_split(long rows, int V, int vec, int sms) {
  const long long rowU = V / vec;
  const long long U = rows * rowU;
  long long G = 3LL * sms;
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
  constexpr size_t smem = size_t(kStreamStages) * kStreamTileBytes;
  const cudaError_t e =
      cudaFuncSetAttribute(select_stream_kernel<T, K>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(select_stream_kernel<T, K>, dim3(p.stream_ctas), dim3(kStreamThreads), smem, stream, p);
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
