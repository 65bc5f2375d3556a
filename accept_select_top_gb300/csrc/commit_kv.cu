// commit_kv.cu -- move the accepted rows' KV into the sequence and release the
// slots (or pages) the accepted path does not keep.
//
// [SGL-XI KV 回写: move_accept_tokens_to_target_kvcache -- target slots from
// req_to_token over [seq_len, seq_len + accept_len), source slots
// out_cache_loc[accept_index] (accept_index holds global rows, -1 unused),
// size by accept_index's width, not by num_draft_tokens], [ACCEPT section 3:
// the committed rows are the input rows R, A, C, not the output X],
// [EVOL 草稿、验证与槽位: only the accepted path's slots are kept].
//
// Grid: one CTA per request.  The CTA reads every source row of the request
// (all layers, K and V) into shared memory before writing any target row, in
// column slices small enough for shared memory; a target that is also a later
// source is therefore never clobbered.  Each CTA stages its request's free
// units in the workspace; the CTA arriving last concatenates them in request
// order into free_ids and writes n_free.
#include "common.cuh"
#include "kernels.cuh"

namespace spec {

namespace {

constexpr int kCommitThreads = 256;
constexpr int kSliceBytes = 32 * 1024;  // shared staging per slice (K and V of all L rows)

__global__ void __launch_bounds__(kCommitThreads) commit_kernel(CommitParams a) {
  const int req = blockIdx.x;
  const int n = a.n, W = a.W;
  __shared__ int src[kMaxN + 1], dst[kMaxN + 1];
  __shared__ int s_ok, s_L;
  __shared__ uint4 stage[kSliceBytes / 16];
  int* stage_free = reinterpret_cast<int*>(a.partials) + size_t(req) * n;
  int* counts = reinterpret_cast<int*>(a.partials) + size_t(a.b) * n;

  if (threadIdx.x == 0) {
    int ok = 1;
    const int L = a.accept_lens[req];
    const int s0 = a.seq_lens[req];
    const int rq = a.req_pool_idx[req];
    if (L < 1 || L > W || s0 < 0 || s0 + L > a.row_w) {
      raise_error(a.error, SPEC_DEV_LENGTH);
      ok = 0;
    }
    if (rq < 0 || rq >= a.req_rows) {
      raise_error(a.error, SPEC_DEV_INDEX);
      ok = 0;
    }
    s_L = ok ? L : 0;
    s_ok = ok;
  }
  __syncthreads();
  const int L = s_L;
  for (int kk = threadIdx.x; kk < L; kk += blockDim.x) {
    const int ai = a.accept_index[size_t(req) * W + kk];
    int s = -1, d = -1;
    if (ai >= 0 && ai < a.b * n) s = a.verify_loc[ai];
    d = a.req_to_token[size_t(a.req_pool_idx[req]) * a.row_w + a.seq_lens[req] + kk];
    if (s < 0 || s >= a.num_slots || d < 0 || d >= a.num_slots) {
      raise_error(a.error, SPEC_DEV_INDEX);
      atomicExch(&s_ok, 0);
    }
    src[kk] = s;
    dst[kk] = d;
  }
  __syncthreads();
  const bool ok = s_ok;

  if (ok) {
    const int units = a.Hkv * a.D * 2 / 16;         // 16-byte units per slot row
    const int slice = max(1, min(units, kSliceBytes / 16 / (2 * L)));
    for (int layer = 0; layer < a.num_layers; ++layer) {
      const uint4* kin = static_cast<const uint4*>(a.k_layers[layer]);
      const uint4* vin = static_cast<const uint4*>(a.v_layers[layer]);
      uint4* kout = static_cast<uint4*>(a.k_layers[layer]);
      uint4* vout = static_cast<uint4*>(a.v_layers[layer]);
      for (int c0 = 0; c0 < units; c0 += slice) {
        const int cw = min(slice, units - c0);
        const int tot = 2 * L * cw;
        for (int t = threadIdx.x; t < tot; t += blockDim.x) {
          const int which = t / (L * cw), rem = t % (L * cw), kk = rem / cw, col = rem % cw;
          const uint4* pool = which ? vin : kin;
          stage[t] = pool[size_t(src[kk]) * units + c0 + col];
        }
        __syncthreads();
        for (int t = threadIdx.x; t < tot; t += blockDim.x) {
          const int which = t / (L * cw), rem = t % (L * cw), kk = rem / cw, col = rem % cw;
          uint4* pool = which ? vout : kout;
          pool[size_t(dst[kk]) * units + c0 + col] = stage[t];
        }
        __syncthreads();
      }
    }
  }
  if (threadIdx.x == 0) a.new_seq_lens[req] = a.seq_lens[req] + (ok ? L : 0);

  // free units of this request, in ascending node order: node j's unit
  // (slot, or page = slot / page_size) is released when no target slot of the
  // request lies in it, at the first node that holds it.  One node per thread.
  __shared__ int unit_s[kMaxN];
  __shared__ int dst_unit_s[kMaxN + 1];
  __shared__ int s_count;
  const int ps = a.page_size;
  for (int kk = threadIdx.x; kk < L; kk += blockDim.x) dst_unit_s[kk] = int(dst[kk] / ps);
  bool free_j = false;
  int j = threadIdx.x;
  if (j < n) {
    const int slot = a.verify_loc[size_t(req) * n + j];
    unit_s[j] = (slot >= 0 && slot < a.num_slots) ? slot / ps : -1;
  }
  __syncthreads();
  if (j < n && ok) {
    const int u = unit_s[j];
    if (u < 0) {
      raise_error(a.error, SPEC_DEV_INDEX);
    } else {
      bool kept = false;
      for (int kk = 0; kk < L && !kept; ++kk) kept = dst_unit_s[kk] == u;
      bool listed = false;
      for (int jj = 0; jj < j && !listed; ++jj) listed = unit_s[jj] == u;
      free_j = !kept && !listed;
    }
  }
  // compaction in node order (n <= 64: the first two warps)
  __shared__ int warp_cnt[2];
  if (threadIdx.x < 64) {
    const unsigned bal = __ballot_sync(0xffffffffu, free_j);
    if ((threadIdx.x & 31) == 0) warp_cnt[threadIdx.x >> 5] = __popc(bal);
    __syncwarp();
  }
  __syncthreads();
  if (threadIdx.x < 64) {
    const unsigned bal = __ballot_sync(0xffffffffu, free_j);
    const int before = (threadIdx.x >= 32 ? warp_cnt[0] : 0) + __popc(bal & ((1u << (threadIdx.x & 31)) - 1u));
    if (free_j) stage_free[before] = unit_s[j];
    if (threadIdx.x == 0) {
      s_count = warp_cnt[0] + warp_cnt[1];
      counts[req] = s_count;
    }
  }

  if (!arrive_last(a.counters, uint32_t(a.b))) return;

  // ---- the last CTA concatenates the staged lists in request order:
  // a block-wide exclusive scan of the counts, then each thread copies its
  // request's entries ----
  __shared__ int warp_sum[kCommitThreads / 32];
  __shared__ int s_running;
  if (threadIdx.x == 0) s_running = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int r0 = 0; r0 < a.b; r0 += blockDim.x) {
    const int r = r0 + threadIdx.x;
    const int c = r < a.b ? __ldcg(counts + r) : 0;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sum[w] = incl;
    __syncthreads();
    int before = s_running;
    for (int i = 0; i < w; ++i) before += warp_sum[i];
    const int off = before + incl - c;
    if (r < a.b) {
      const int* from = reinterpret_cast<const int*>(a.partials) + size_t(r) * n;
      for (int e = 0; e < c; ++e) a.free_ids[off + e] = __ldcg(from + e);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int tot = 0;
      for (int i = 0; i < nw; ++i) tot += warp_sum[i];
      s_running += tot;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) *a.n_free = s_running;
  counter_reset(a.counters);
}

}  // namespace

size_t commit_partial_bytes(int b, int n) { return align256(size_t(b) * n * 4 + size_t(b) * 4); }

int launch_commit_kv(const CommitParams& p, cudaStream_t stream) {
  commit_kernel<<<p.b, kCommitThreads, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
}

}  // namespace spec
