// verify_sampling.cu -- rejection-sampling accept with residual resampling and
// the terminal bonus token.
//
// [ACCEPT section 4: accept x when u < min(1, p(x)/q(x)) tested without the
// division as u*q(x) < p(x); on rejection sample max(p - q, 0)/Z; after a fully
// accepted path sample the bonus from p], [INTERN 接受/拒绝], [EAGLE2 5.6: a
// rejected child passes to the next sibling, all rejected -> residual],
// [SGL-XI eagle_sample, 路径三:拒绝采样].
//
// The same two passes serve the target-only tree sampler [ACCEPT section 4,
// Target-only Tree Sampling]: only the walk and the terminal mass differ.
//
// Pass 1, grid (chunks, b*n): every verify row is reduced to (max, argmax,
// sum of exp((x - max)/T)) by chunk; the CTA arriving last for a request merges
// the request's rows and walks the tree with p(x) = exp((l_x - max)/T)/sum
// (fp32) read at the children's tokens only.  It writes everything but the
// terminal token, and leaves the request's state (terminal node, mode) in the
// workspace: mode 0 = done (greedy request, terminal = argmax), 1 = sample the
// terminal from p, 2 = sample it from the residual max(0, p - q), 3 = sample
// it from p without the terminal node's rejected children (target-only:
// relu(p - buffer), the buffer holding those children's p).
// Pass 2, grid (term_ctas, b), one wave: for requests of mode 1 to 3 each CTA
// sums, in fp64, the residual and p over chunks of the terminal row (chunk
// c by CTA c mod term_ctas); the last CTA of the request finds the chunk
// where u_final * Z falls and the token inside it by an in-order scan.
#include "common.cuh"
#include "kernels.cuh"
#include "stream_records.cuh"

namespace spec {

namespace {

struct StatPart {
  float m;
  int arg;
  float s;
  float pad;
};

struct ReqState {
  int cur;    // terminal node
  int mode;   // 0 done, 1 from p, 2 from residual, 3 from p without the rejected children
  int ncd;    // accepted drafts
  int row;    // verify row of the terminal node (logits / q row)
  float M;    // max logit of that row
  float S;    // sum of exp((x - M)/T) of that row
  float T;
  int out_row;  // retrieve_index row of the terminal node
};

struct MassPart {
  double res;   // sum of max(0, p - q) over the chunk
  double p;     // sum of p over the chunk
  int last_res; // last index with a positive residual, -1 if none
  int last_p;
  int pad[2];
};

// p of one token given the row statistics (T > 0).
__device__ __forceinline__ float p_of(float l, float M, float T, float S) { return expf((l - M) / T) / S; }

template <typename T, bool PROBS, int MAXCH = kMaxChunks>
__device__ __forceinline__ void sampling_walk(const SamplingParams& a, int req, float temp, bool soft, float c);

// PROBS: the probabilities mode (a.probs given), a separate instantiation so
// that the logit path carries none of its branches.
template <typename T, bool PROBS>
__global__ void __launch_bounds__(kThreads) sampling_stats_kernel(SamplingParams a) {
  pdl_wait();
  pdl_trigger();
  using Tr = LogitTraits<T>;
  const int row = blockIdx.y;
  const int chunk = blockIdx.x;
  const int req = row / a.n;
  const int begin = chunk * a.chunk_elems;
  const int end = min(a.V, begin + a.chunk_elems);
  const T* lrow = static_cast<const T*>(a.logits) + size_t(row) * a.V;
  const float temp = PROBS ? 1.f : a.temperatures[req];  // the probabilities mode has no temperature
  const bool soft = temp > 0.f;
  const float c = soft ? 1.4426950408889634f / temp : 0.f;

  float m = -3.0e38f, s = 0.f, bv = -INFINITY;
  int bi = INT_MAX;
  if (!PROBS) scan_row_stats<T>(lrow, begin, end, a.vec_ok, soft, c, bv, bi, m, s);
  // CTA reduction
  __shared__ float sm_[kThreads / 32], ss_[kThreads / 32], sv_[kThreads / 32];
  __shared__ int si_[kThreads / 32];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  {
    float M = warp_max(m);
    float sc = warp_sum(s * exp2f((m - M) * c));
    warp_argmax(bv, bi);
    if (lane == 0) {
      sm_[w] = M;
      ss_[w] = sc;
      sv_[w] = bv;
      si_[w] = bi;
    }
  }
  __syncthreads();
  StatPart* part = reinterpret_cast<StatPart*>(a.partials) + size_t(row) * a.chunks + chunk;
  if (w == 0) {
    float M = lane < nw ? sm_[lane] : -3.0e38f;
    M = warp_max(M);
    float sc = warp_sum(lane < nw ? ss_[lane] * exp2f((sm_[lane] - M) * c) : 0.f);
    float v = lane < nw ? sv_[lane] : -INFINITY;
    int i = lane < nw ? si_[lane] : INT_MAX;
    warp_argmax(v, i);
    if (lane == 0) *part = StatPart{soft ? M : v, i, sc, 0.f};
  }

  if (!arrive_last(a.counters + req, uint32_t(a.n * a.chunks))) return;
  sampling_walk<T, PROBS>(a, req, temp, soft, c);
}

// ---- the walk of request `req` (the CTA whose statistics arrived last) ----
// Merges the request's row statistics (a.chunks <= MAXCH partials a row),
// then walks the tree; every thread of the CTA calls it.
template <typename T, bool PROBS, int MAXCH>
__device__ __forceinline__ void sampling_walk(const SamplingParams& a, int req, float temp, bool soft, float c) {
  using Tr = LogitTraits<T>;
  const int n = a.n, base = req * n, W = a.S + 1;
  __shared__ float rM[kMaxN], rS[kMaxN];
  __shared__ int rA[kMaxN], tok[kMaxN], nt[kMaxN], ns[kMaxN], ri[kMaxN], pred[kMaxN], path[kMaxN + 1], par[kMaxN];
  __shared__ float lgs[kMaxN], qxs[kMaxN], us[kMaxN];
  __shared__ int s_len, s_mode;
  __shared__ float4 stage[kMaxN * MAXCH];  // (MAXCH: the most chunks a row of this caller has)
  // every (row, chunk) partial in one round of loads, through L2 (__ldcg)
  for (int t = threadIdx.x; t < n * a.chunks; t += blockDim.x)
    stage[t] = __ldcg(reinterpret_cast<const float4*>(
        reinterpret_cast<const StatPart*>(a.partials) + size_t(base) * a.chunks) + t);
  __syncthreads();
  for (int t = threadIdx.x; t < n; t += blockDim.x) {
    const float4* pr = stage + t * a.chunks;
    float M = -3.0e38f, v = -INFINITY;
    int arg = INT_MAX;
    for (int ch = 0; ch < a.chunks; ++ch) {
      const float4 q = pr[ch];
      M = fmaxf(M, q.x);
      // the argmax of a soft row is tracked through the chunk max
      if (better(q.x, __float_as_int(q.y), v, arg)) {
        v = q.x;
        arg = __float_as_int(q.y);
      }
    }
    float S = 0.f;
    for (int ch = 0; ch < a.chunks; ++ch) {
      const float4 q = pr[ch];
      S += q.z * exp2f((q.x - M) * c);
    }
    rM[t] = M;
    rS[t] = S;
    rA[t] = arg;
    tok[t] = a.draft_tokens[base + t];
    int x = a.next_token[base + t], y = a.next_sibling[base + t], r = a.retrieve_index[base + t];
    if (x < -1 || x >= n || y < -1 || y >= n || r < base || r >= base + n) {
      raise_error(a.error, SPEC_DEV_INDEX);
      x = x < -1 || x >= n ? -1 : x;
      y = y < -1 || y >= n ? -1 : y;
      r = r < base || r >= base + n ? base + t : r;
    }
    nt[t] = x;
    ns[t] = y;
    ri[t] = r;
    pred[t] = 0;
    par[t] = -1;
  }
  __syncthreads();
  // Every value the walk reads, loaded by all threads at once: node i's
  // logit (or probability) and q at its parent's row and its token, and its
  // coin.  The parent is taken from the children lists; the walk falls back to
  // a direct load wherever it reaches a node from another parent (a malformed
  // tree).
  const T* L = static_cast<const T*>(a.logits);
  for (int t = threadIdx.x; t < n; t += blockDim.x) {
    int ch = nt[t], guard = 0;
    while (ch != -1 && guard++ < n) {
      par[ch] = t;
      ch = ns[ch];
    }
  }
  __syncthreads();
  for (int t = threadIdx.x; t < n; t += blockDim.x) {
    const int pa = par[t], x = tok[t];
    us[t] = a.u[base + t];
    lgs[t] = 0.f;
    qxs[t] = 0.f;
    if (pa >= 0 && x >= 0 && x < a.V) {
      const size_t prow = size_t(base + pa);
      if (PROBS) lgs[t] = __ldg(a.probs + prow * a.V + x);
      else if (soft) lgs[t] = Tr::load(L, prow * a.V + x);
      if (!a.target_only) qxs[t] = __ldg(a.draft_probs + prow * a.V + x);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int cur = 0, ncd = 0, all_rejected = 0;
    path[0] = 0;
    // target-only: the coin of the node whose children are scanned (the
    // root's first, then each accepted child's own)
    float coin = a.target_only ? us[0] : 0.f;
    for (int d = 0; d < a.S && ncd < n - 1; ++d) {  // bounded by the tree depth
      const size_t vrow = size_t(base + cur);
      const float* q = a.target_only ? nullptr : a.draft_probs + vrow * a.V;
      int c2 = nt[cur], hit = -1, guard = 0;
      const int had_child = c2 != -1;
      float prob_acc = 0.f;  // target-only: the scanned siblings' mass, fp32
      while (c2 != -1 && guard++ < n) {
        const int x = tok[c2];
        if (x < 0 || x >= a.V) {
          raise_error(a.error, SPEC_DEV_INDEX);
          c2 = ns[c2];
          continue;
        }
        const bool pre = par[c2] == cur;  // the values loaded above are this node's at this row
        float px;
        if (PROBS) px = pre ? lgs[c2] : __ldg(a.probs + vrow * a.V + x);  // the given distribution
        else if (soft) px = p_of(pre ? lgs[c2] : Tr::load(L, vrow * a.V + x), rM[cur], temp, rS[cur]);
        else px = x == rA[cur] ? 1.f : 0.f;
        bool accept;
        if (a.target_only) {
          prob_acc = __fadd_rn(prob_acc, px);
          accept = px > 0.f && (coin < __fdiv_rn(prob_acc, a.thr_acc) || px >= a.thr_single);
        } else {
          accept = __fmul_rn(us[c2], pre ? qxs[c2] : __ldg(q + x)) < px;
        }
        if (accept) {
          hit = c2;
          break;
        }
        c2 = ns[c2];
      }
      if (hit < 0) {
        all_rejected = had_child;
        break;
      }
      pred[cur] = tok[hit];
      path[++ncd] = hit;
      cur = hit;
      if (a.target_only) coin = us[hit];
    }
    int mode = (soft || PROBS) ? (all_rejected ? (a.target_only ? 3 : 2) : 1) : 0;
    if (mode == 0) pred[cur] = rA[cur];
    ReqState* st = reinterpret_cast<ReqState*>(a.state) + req;
    if (PROBS) *st = ReqState{cur, mode, ncd, base + cur, 0.f, 1.f, 1.f, ri[cur]};
    else *st = ReqState{cur, mode, ncd, base + cur, rM[cur], rS[cur], temp, ri[cur]};
    a.accept_lens[req] = ncd + 1;
    if (mode == 0 && a.next_root) a.next_root[req] = pred[cur];
    s_len = ncd + 1;
    s_mode = mode;
  }
  __syncthreads();
  const int Lp = s_len;
  for (int t = threadIdx.x; t < n; t += blockDim.x) a.predict[ri[t]] = pred[t];
  for (int d = threadIdx.x; d < W; d += blockDim.x) {
    a.accept_index[size_t(req) * W + d] = d < Lp ? ri[path[d]] : -1;
    if (a.accepted_tokens) {
      const bool known = d < Lp - 1 || (d == Lp - 1 && s_mode == 0);
      a.accepted_tokens[size_t(req) * W + d] = known ? pred[path[d]] : -1;
    }
  }
  counter_reset(a.counters + req);
}

// Pass 1 on the streaming pass's unit summaries (stream_records.cu), one
// warp a verify row, the CTAs of a request holding only its rows (rpc =
// min(8, n) rows a CTA): the row maximum M (the largest unit maximum), the
// softmax denominator S = sum of su 2^((gu - M) c) (soft rows) and, for a
// greedy row, the argmax (the lowest index holding M: in the first unit whose
// maximum is M, reloaded) as one chunk's statistics; the CTA whose rows are
// the last of its request to arrive walks the request.
constexpr int kRowWarpsMax = 8;
constexpr int kSumPer = kRowRecordsMax / 32 / 32;  // unit summaries a lane reads (a row spans <= 256 units)

template <typename T>
__global__ void __launch_bounds__(32 * kRowWarpsMax, 1) sampling_rowstats_kernel(SamplingParams a) {
  constexpr int E = LogitTraits<T>::kVec;
  pdl_wait();
  pdl_trigger();
  const int rpc = int(blockDim.x) >> 5, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cpr = (a.n + rpc - 1) / rpc;  // CTAs a request
  const int req = blockIdx.x / cpr, rin = (blockIdx.x % cpr) * rpc + w;
  const float temp = a.temperatures[req];
  const bool soft = temp > 0.f;
  const float c = soft ? 1.4426950408889634f / temp : 0.f;
  if (blockIdx.x == 0 && threadIdx.x == 0) *a.queue = 0u;  // the streaming grid is done with the queue: ready for the next call
  if (rin < a.n) {
    const int row = req * a.n + rin;
    const long long rowU = a.V / E;
    const long long rs = (long long)row * rowU, rend = rs + rowU;  // the row's vectors
    const int uf = int(rs / kUnitVecs), nun = int((rend - 1) / kUnitVecs) - uf + 1;
    const int par = row & 1;
    // lane l: units l, l + 32, ... (all loads in flight)
    float2 us[kSumPer];
#pragma unroll
    for (int t = 0; t < kSumPer; ++t) {
      const int m = lane + 32 * t;
      us[t] = m < nun ? __ldcg(&a.usum[(uf + m) * 2 + par]) : make_float2(-INFINITY, 0.f);
    }
    const ExpScale sc = soft ? ExpScale(temp) : ExpScale();
    RecSum rsum;
    float lm = -INFINITY;
#pragma unroll
    for (int t = 0; t < kSumPer; ++t) {
      lm = fmaxf(lm, us[t].x);
      if (soft && us[t].y > 0.f) rsum.add(us[t].x, us[t].y, sc);  // (0: the unit's part of the row is all -inf)
    }
    const float M = warp_max(lm);
    const float S = soft ? warp_sum(rsum.rel(M, sc)) : 0.f;
    int arg = 0;  // (every element -inf: the first is the argmax)
    if (!soft && M > -INFINITY) {
      // the first unit whose maximum is M, then its first element equal to M
      int mf = INT_MAX;
#pragma unroll
      for (int t = kSumPer - 1; t >= 0; --t)
        if (lane + 32 * t < nun && us[t].x == M) mf = lane + 32 * t;
      mf = __reduce_min_sync(0xffffffffu, mf);
      const uint4* L = static_cast<const uint4*>(a.logits);
      uint4 x[kStreamVpt];
      bool in[kStreamVpt];
#pragma unroll
      for (int u = 0; u < kStreamVpt; ++u) {
        const long long gv = (long long)(uf + mf) * kUnitVecs + lane + u * 32;
        in[u] = gv >= rs && gv < rend;
        x[u] = in[u] ? __ldcg(L + gv) : make_uint4(0u, 0u, 0u, 0u);
      }
      int first = INT_MAX;
#pragma unroll
      for (int u = kStreamVpt - 1; u >= 0; --u) {  // (later vectors hold higher indices)
        if (!in[u]) continue;
        const long long gv = (long long)(uf + mf) * kUnitVecs + lane + u * 32;
#pragma unroll
        for (int q = E - 1; q >= 0; --q)
          if (VecOps<T>::at(x[u], q) == M) first = int((gv - rs) * E) + q;
      }
      arg = __reduce_min_sync(0xffffffffu, first);
      if (arg == INT_MAX) arg = 0;  // (not reached: the unit holds its maximum)
    }
    if (lane == 0) reinterpret_cast<StatPart*>(a.partials)[row] = StatPart{M, arg, S, 0.f};
  }
  if (!arrive_last(a.counters + req, uint32_t(cpr))) return;
  SamplingParams a1 = a;
  a1.chunks = 1;  // a row's statistics are one chunk's
  sampling_walk<T, false, 1>(a1, req, temp, soft, c);
}

// Compensated (Kahan) fp32 accumulation: the per-element work stays off the
// slow fp64 pipe; the few per-thread totals are combined in fp64.
struct Kahan {
  float sum = 0.f, comp = 0.f;
  __device__ __forceinline__ void add(float x) {
    const float y = x - comp;
    const float t = sum + y;
    comp = (t - sum) - y;
    sum = t;
  }
};

// p of a token of the terminal row from its logit: 2^((l - M) c) / S with
// c = log2(e) / T, by the hardware exp2 (relative error about 2^-22) and one
// multiply.  The chunk sums and the in-chunk search use the same p.
struct TermP {
  float M, c, invS;
  bool given;  // probabilities mode: the loaded value is p itself
  __device__ __forceinline__ TermP(const ReqState& st, bool probs)
      : M(st.M), c(1.4426950408889634f / st.T), invS(1.f / st.S), given(probs) {}
  __device__ __forceinline__ float p(float l) const { return given ? l : fast_exp2((l - M) * c) * invS; }
};

// The value the terminal pass loads for token v of a row: its logit, or its
// probability in the probabilities mode.
template <typename T, bool PROBS>
__device__ __forceinline__ float term_load(const SamplingParams& a, size_t row, int v) {
  if (PROBS) return __ldg(a.probs + row * a.V + v);
  return LogitTraits<T>::load(static_cast<const T*>(a.logits) + row * a.V, size_t(v));
}

// Target-only terminal draws leave out the terminal node's rejected children:
// their tokens, listed once per CTA, marked in a bitmap over one chunk of the
// row (a chunk holds at most 4096 tokens).
constexpr int kExclWords = 4096 / 32;

struct Excluded {
  int n;             // listed tokens
  const int* tok;    // [n] in shared memory
  uint32_t* bits;    // [kExclWords] in shared memory
  // Marks the listed tokens inside [lo, lo + 4096) (every thread of the CTA).
  __device__ __forceinline__ void mark(int lo) const {
    for (int i = threadIdx.x; i < kExclWords; i += blockDim.x) bits[i] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const int x = tok[i] - lo;
      if (x >= 0 && x < kExclWords * 32) atomicOr(&bits[x >> 5], 1u << (x & 31));
    }
    __syncthreads();
  }
  __device__ __forceinline__ bool has(int v, int lo) const {
    const int x = v - lo;
    return (bits[x >> 5] >> (x & 31)) & 1u;
  }
};

// Mass of a token of the terminal row given its logit l and q: the residual
// max(0, p - q) (mode 2), p unless the token is excluded (mode 3), or p.
__device__ __forceinline__ float term_mass(const TermP& tp, int mode, bool excluded, float l, float qv) {
  const float p = tp.p(l);
  if (mode == 3) return excluded ? 0.f : p;
  if (mode != 2) return p;
  return p > qv ? p - qv : 0.f;  // the fp32 difference of the two values
}

constexpr int kTermPer = 16;  // terminal tokens a thread holds at once

// Sums of the rule's mass (residual, or p without the excluded tokens) and of
// p over row[begin, end) of the terminal row, each thread loading kTermPer
// tokens (logit and q) before using any.
template <typename T, bool PROBS>
__device__ __forceinline__ void chunk_mass(const SamplingParams& a, const ReqState& st, const Excluded& ex,
                                           int begin, int end, double& res, double& ps, int& last_res,
                                           int& last_p) {
  const float* q = st.mode == 2 ? a.draft_probs + size_t(st.row) * a.V : nullptr;
  const TermP tp(st, PROBS);
  const int nt = blockDim.x;
  Kahan kr, kp;
  for (int b0 = begin + int(threadIdx.x); b0 < end; b0 += kTermPer * nt) {
    float lv[kTermPer], qv[kTermPer];
#pragma unroll
    for (int u = 0; u < kTermPer; ++u) {
      const int v = b0 + u * nt;
      lv[u] = v < end ? term_load<T, PROBS>(a, size_t(st.row), v) : (PROBS ? 0.f : -INFINITY);
      qv[u] = (q && v < end) ? __ldg(q + v) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kTermPer; ++u) {
      const int v = b0 + u * nt;
      const float p = v < end ? tp.p(lv[u]) : 0.f;
      float r = 0.f;
      if (st.mode == 2) r = p > qv[u] ? p - qv[u] : 0.f;
      else if (st.mode == 3 && v < end) r = ex.has(v, begin) ? 0.f : p;
      kr.add(r);
      kp.add(p);
      if (r > 0.f) last_res = v;
      if (p > 0.f) last_p = v;
    }
  }
  res = double(kr.sum) - double(kr.comp);
  ps = double(kp.sum) - double(kp.comp);
}

// As chunk_mass, for logit rows of whole 16-token vectors (a.vec_term):
// thread t takes the 16 consecutive tokens [begin + 16 t, + 16) with 16-byte
// loads (two or four of logits, four of q).  The chunk's tokens come in
// whole 16-token vectors (V % 16 == 0).
template <typename T>
__device__ __forceinline__ void chunk_mass_vec(const SamplingParams& a, const ReqState& st, const Excluded& ex,
                                               int begin, int end, double& res, double& ps, int& last_res,
                                               int& last_p) {
  constexpr int E = LogitTraits<T>::kVec;
  const int v0 = begin + kTermPer * int(threadIdx.x);
  const TermP tp(st, false);
  Kahan kr, kp;
  if (v0 < end) {
    const uint4* lrow = reinterpret_cast<const uint4*>(static_cast<const T*>(a.logits) + size_t(st.row) * a.V + v0);
    uint4 lx[kTermPer / E];
#pragma unroll
    for (int j = 0; j < kTermPer / E; ++j) lx[j] = __ldg(lrow + j);
    float4 qx[kTermPer / 4];
    if (st.mode == 2) {
      const float4* qrow = reinterpret_cast<const float4*>(a.draft_probs + size_t(st.row) * a.V + v0);
#pragma unroll
      for (int j = 0; j < kTermPer / 4; ++j) qx[j] = __ldg(qrow + j);
    } else {
#pragma unroll
      for (int j = 0; j < kTermPer / 4; ++j) qx[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kTermPer; ++u) {
      const int v = v0 + u;
      const float l = VecOps<T>::at(lx[u / E], u % E);
      const float4 q4 = qx[u / 4];
      const float qv = (u & 3) == 0 ? q4.x : (u & 3) == 1 ? q4.y : (u & 3) == 2 ? q4.z : q4.w;
      const float p = tp.p(l);
      float r = 0.f;
      if (st.mode == 2) r = p > qv ? p - qv : 0.f;
      else if (st.mode == 3) r = ex.has(v, begin) ? 0.f : p;
      kr.add(r);
      kp.add(p);
      if (r > 0.f) last_res = v;
      if (p > 0.f) last_p = v;
    }
  }
  res = double(kr.sum) - double(kr.comp);
  ps = double(kp.sum) - double(kp.comp);
}

// MINB: CTAs a SM the registers must allow -- 4 for the grid of a CTA a chunk
// (more CTAs resident, fewer waves), 2 for the looping grid (its one wave of
// two CTAs a SM; a tighter cap makes the loop spill).
template <typename T, bool PROBS, int MINB>
__global__ void __launch_bounds__(kThreads, MINB) sampling_bonus_kernel(SamplingParams a) {
  pdl_wait();
  pdl_trigger();
  using Tr = LogitTraits<T>;
  const int req = blockIdx.y;
  const ReqState st = reinterpret_cast<const ReqState*>(a.state)[req];
  if (st.mode == 0) return;  // every CTA of this request agrees: nothing to sample
  // The state comes from the workspace.  One the stats pass did not write (a
  // workspace used before its zero fill completed) must not steer an access:
  // every field that addresses memory is checked, and the request is skipped
  // with SPEC_DEV_INVARIANT (all CTAs of the request see the same state).
  {
    const int base = req * a.n;
    const bool ok = st.mode >= 1 && st.mode <= 3 && st.cur >= 0 && st.cur < a.n && st.row == base + st.cur &&
                    st.out_row >= base && st.out_row < base + a.n && st.ncd >= 0 && st.ncd <= a.S &&
                    st.S > 0.f && st.T > 0.f;
    if (!ok) {
      if (blockIdx.x == 0 && threadIdx.x == 0) raise_error(a.error, SPEC_DEV_INVARIANT);
      return;
    }
  }
  // mode 3: the tokens of the terminal node's children (all rejected), read
  // from the tree arrays in one round of loads and walked in shared memory
  __shared__ int s_tok[kMaxN], s_ns[kMaxN], s_excl[kMaxN];
  __shared__ int s_nexcl, s_first;
  __shared__ uint32_t s_bits[kExclWords];
  Excluded ex{0, s_excl, s_bits};
  if (st.mode == 3) {
    const int base = req * a.n, t = threadIdx.x;
    if (t < a.n) {
      s_tok[t] = a.draft_tokens[base + t];
      s_ns[t] = a.next_sibling[base + t];
    }
    if (t == kMaxN) s_first = a.next_token[base + st.cur];
    __syncthreads();
    if (t == 0) {
      int k = 0, c = s_first, guard = 0;
      while (c >= 0 && c < a.n && guard++ < a.n) {  // an index out of range ends the list
        const int x = s_tok[c];
        if (x >= 0 && x < a.V) s_excl[k++] = x;
        c = s_ns[c];
      }
      s_nexcl = k;
    }
    __syncthreads();
    ex.n = s_nexcl;
  }
  __shared__ double sres[kThreads / 32], sps[kThreads / 32];
  __shared__ int slr[kThreads / 32], slp[kThreads / 32];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  MassPart* parts = reinterpret_cast<MassPart*>(a.partials2) + size_t(req) * a.chunks2;
  // this CTA's chunks: blockIdx.x, + gridDim.x, ...
  for (int chunk = blockIdx.x; chunk < a.chunks2; chunk += gridDim.x) {
    const int begin = chunk * a.chunk2_elems;
    const int end = min(a.V, begin + a.chunk2_elems);
    if (st.mode == 3) ex.mark(begin);
    double res = 0.0, ps = 0.0;
    int last_res = -1, last_p = -1;
    if constexpr (!PROBS) {
      if (a.vec_term) chunk_mass_vec<T>(a, st, ex, begin, end, res, ps, last_res, last_p);
      else chunk_mass<T, PROBS>(a, st, ex, begin, end, res, ps, last_res, last_p);
    } else {
      chunk_mass<T, PROBS>(a, st, ex, begin, end, res, ps, last_res, last_p);
    }
    res = warp_sum_d(res);
    ps = warp_sum_d(ps);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      last_res = max(last_res, __shfl_xor_sync(0xffffffffu, last_res, o));
      last_p = max(last_p, __shfl_xor_sync(0xffffffffu, last_p, o));
    }
    if (lane == 0) {
      sres[w] = res;
      sps[w] = ps;
      slr[w] = last_res;
      slp[w] = last_p;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      MassPart mp{0.0, 0.0, -1, -1, {0, 0}};
      for (int i = 0; i < nw; ++i) {
        mp.res += sres[i];
        mp.p += sps[i];
        mp.last_res = max(mp.last_res, slr[i]);
        mp.last_p = max(mp.last_p, slp[i]);
      }
      parts[chunk] = mp;
    }
    __syncthreads();  // the chunk's sums and bitmap are read before the next chunk writes them
  }

  if (!arrive_last(a.counters + req, uint32_t(gridDim.x))) return;

  // ---- finalize: locate u_final * Z on the cumulative mass ----
  // every chunk's partial in one round of loads, then the prefix in shared memory
  __shared__ double s_res[kMaxChunks2], s_p[kMaxChunks2];
  __shared__ int s_lr[kMaxChunks2], s_lp[kMaxChunks2];
  for (int ch = threadIdx.x; ch < a.chunks2; ch += blockDim.x) {
    s_res[ch] = __ldcg(&parts[ch].res);
    s_p[ch] = __ldcg(&parts[ch].p);
    s_lr[ch] = __ldcg(&parts[ch].last_res);
    s_lp[ch] = __ldcg(&parts[ch].last_p);
  }
  __syncthreads();
  __shared__ int s_chunk, s_use_res, s_fallback;
  __shared__ double s_before, s_target;
  if (w == 0) {
    // warp 0: lane l holds chunks 2l and 2l + 1 (kMaxChunks2 = 64); inclusive
    // prefix sums of the lanes' pairs (fp64) give each chunk's running mass
    const int c0 = 2 * lane, c1 = c0 + 1;
    const double r0 = c0 < a.chunks2 ? s_res[c0] : 0.0, r1 = c1 < a.chunks2 ? s_res[c1] : 0.0;
    const double p0 = c0 < a.chunks2 ? s_p[c0] : 0.0, p1 = c1 < a.chunks2 ? s_p[c1] : 0.0;
    double sr = r0 + r1, sp = p0 + p1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double yr = __shfl_up_sync(0xffffffffu, sr, o), yp = __shfl_up_sync(0xffffffffu, sp, o);
      if (lane >= o) {
        sr += yr;
        sp += yp;
      }
    }
    const double zr = __shfl_sync(0xffffffffu, sr, 31), zp = __shfl_sync(0xffffffffu, sp, 31);
    int lr = max(c0 < a.chunks2 ? s_lr[c0] : -1, c1 < a.chunks2 ? s_lr[c1] : -1);
    int lp = max(c0 < a.chunks2 ? s_lp[c0] : -1, c1 < a.chunks2 ? s_lp[c1] : -1);
    lr = __reduce_max_sync(0xffffffffu, lr);
    lp = __reduce_max_sync(0xffffffffu, lp);
    const int use_res = (st.mode == 2 || st.mode == 3) && zr > 0.0;
    const double Z = use_res ? zr : zp;
    const double target = double(a.u_final[req]) * Z;
    // the first chunk whose running mass passes the target
    const double m0 = use_res ? r0 : p0, m1 = use_res ? r1 : p1;
    const double before = (use_res ? sr : sp) - m0 - m1;  // the mass of the chunks ahead of this lane's
    const int hit = c0 < a.chunks2 && target < before + m0 ? c0 : (c1 < a.chunks2 && target < before + m0 + m1 ? c1 : -1);
    const unsigned lanes = __ballot_sync(0xffffffffu, hit >= 0);
    if (lanes == 0u) {
      if (lane == 0) {
        s_chunk = -1;
        s_before = use_res ? zr : zp;
      }
    } else if (lane == __ffs(lanes) - 1) {
      s_chunk = hit;
      s_before = hit == c0 ? before : before + m0;
    }
    if (lane == 0) {
      s_use_res = use_res;
      s_target = target;
      s_fallback = use_res ? lr : lp;
    }
  }
  __syncthreads();
  __shared__ int s_bonus;
  if (threadIdx.x == 0) s_bonus = s_fallback;
  __syncthreads();
  if (s_chunk >= 0) {
    // In-order search of the chunk in one pass: thread t holds tokens
    // [cb + t*per, cb + (t+1)*per) (loaded at once), a block-wide exclusive
    // scan of the threads' totals gives each its running start, and the first
    // positive-mass token whose running sum passes the target is the draw.
    using Tr = LogitTraits<T>;
    const int cb = s_chunk * a.chunk2_elems;
    const int ce = min(a.V, cb + a.chunk2_elems);
    const bool use_res = s_use_res != 0;
    const int rule = use_res ? st.mode : 1;  // Z == 0 under the rule: draw from p
    if (rule == 3) ex.mark(cb);              // the bitmap of the searched chunk
    const TermP tp(st, PROBS);
    const float* qr = rule == 2 ? a.draft_probs + size_t(st.row) * a.V : nullptr;
    __shared__ float wtot[kThreads / 32];
    __shared__ int s_hit;
    if (threadIdx.x == 0) s_hit = INT_MAX;
    const int per = (ce - cb + int(blockDim.x) - 1) / int(blockDim.x);  // <= kTermPer
    const int t0 = cb + int(threadIdx.x) * per;
    float mv[kTermPer];
    float lv[kTermPer], qv[kTermPer];
#pragma unroll
    for (int u = 0; u < kTermPer; ++u) {
      const int v = t0 + u;
      const bool in = u < per && v < ce;
      lv[u] = in ? term_load<T, PROBS>(a, size_t(st.row), v) : (PROBS ? 0.f : -INFINITY);
      qv[u] = (in && qr) ? __ldg(qr + v) : 0.f;
    }
    float tot = 0.f;
#pragma unroll
    for (int u = 0; u < kTermPer; ++u) {
      const int v = t0 + u;
      const bool in = u < per && v < ce;
      mv[u] = in ? term_mass(tp, rule, rule == 3 && ex.has(v, cb), lv[u], qv[u]) : 0.f;
      tot += mv[u];
    }
    float incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) wtot[w] = incl;
    __syncthreads();
    float before = incl - tot;
    for (int i = 0; i < w; ++i) before += wtot[i];
    const float gap = float(s_target - s_before);
    float run = before;
#pragma unroll
    for (int u = 0; u < kTermPer; ++u) {
      if (mv[u] > 0.f && gap < run + mv[u]) {
        atomicMin(&s_hit, t0 + u);
        break;
      }
      run += mv[u];
    }
    __syncthreads();
    if (threadIdx.x == 0 && s_hit != INT_MAX) s_bonus = s_hit;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const int bonus = s_bonus;
    const int W = a.S + 1;
    a.predict[st.out_row] = bonus;
    if (a.accepted_tokens) a.accepted_tokens[size_t(req) * W + st.ncd] = bonus;
    if (a.next_root) a.next_root[req] = bonus;
  }
  counter_reset(a.counters + req);
}

}  // namespace

size_t sampling_partial_bytes(int rows, int chunks) { return align256(size_t(rows) * chunks * sizeof(StatPart)); }
size_t sampling_state_bytes(int b) { return align256(size_t(b) * sizeof(ReqState)); }
size_t sampling_partial2_bytes(int b, int chunks2) { return align256(size_t(b) * chunks2 * sizeof(MassPart)); }

template <typename T, bool PROBS>
cudaError_t launch_bonus(const SamplingParams& p, cudaStream_t stream) {
  const dim3 g2(p.term_ctas, p.b);
  return p.term_ctas == p.chunks2
             ? launch_pdl(sampling_bonus_kernel<T, PROBS, 4>, g2, dim3(kThreads), 0, stream, p)
             : launch_pdl(sampling_bonus_kernel<T, PROBS, 2>, g2, dim3(kThreads), 0, stream, p);
}

int launch_verify_sampling(const SamplingParams& p, cudaStream_t stream) {
  dim3 g1(p.chunks, p.b * p.n);
  cudaError_t e;
  if (!p.probs && p.stream_ctas > 0) {  // the streaming pass, then the row statistics and the walk
    StreamRecParams r{};
    r.logits = p.logits;
    r.rows = p.b * p.n;
    r.V = p.V;
    r.temperatures = p.temperatures;
    r.rows_per_temp = p.n;
    r.nu = p.stream_nu;
    r.rec = nullptr;  // the row statistics need only the unit summaries
    r.usum = p.usum;
    r.queue = p.queue;
    r.early = false;
    if (launch_stream_records(r, p.stream_ctas, p.dtype, stream) != SPEC_OK) return SPEC_ERR_LAUNCH;
    const int rpc = p.n < kRowWarpsMax ? p.n : kRowWarpsMax;  // rows a CTA
    const dim3 gr(p.b * ((p.n + rpc - 1) / rpc)), br(32 * rpc);
    if (p.dtype == SPEC_F32) {
      e = launch_pdl(sampling_rowstats_kernel<float>, gr, br, 0, stream, p);
      if (e == cudaSuccess) e = launch_bonus<float, false>(p, stream);
    } else {
      e = launch_pdl(sampling_rowstats_kernel<uint16_t>, gr, br, 0, stream, p);
      if (e == cudaSuccess) e = launch_bonus<uint16_t, false>(p, stream);
    }
    return e == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
  }
  if (p.probs) {  // fp32 probabilities
    e = launch_pdl(sampling_stats_kernel<float, true>, g1, dim3(kThreads), 0, stream, p);
    if (e == cudaSuccess) e = launch_bonus<float, true>(p, stream);
  } else if (p.dtype == SPEC_F32) {
    e = launch_pdl(sampling_stats_kernel<float, false>, g1, dim3(kThreads), 0, stream, p);
    if (e == cudaSuccess) e = launch_bonus<float, false>(p, stream);
  } else {
    e = launch_pdl(sampling_stats_kernel<uint16_t, false>, g1, dim3(kThreads), 0, stream, p);
    if (e == cudaSuccess) e = launch_bonus<uint16_t, false>(p, stream);
  }
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
}

}  // namespace spec
