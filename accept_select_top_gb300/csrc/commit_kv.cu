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
// Grid: (request, layer group).  CTA (req, g) moves layers g, g + G, ... of
// request req: per layer it reads every source row (K and V) of a column slice
// into shared memory before writing any target row of that slice, so a target
// that is also a source is never clobbered.  All loads that do not depend on
// one another are issued together (the kernel is a handful of short dependent
// round trips, not bandwidth).  CTA (req, 0) also writes new_seq_lens and
// stages the request's free units in the workspace; of those b CTAs the one
// arriving last concatenates the lists in request order into free_ids and
// writes n_free (the other layer groups take no part in it).
#include "common.cuh"
#include "kernels.cuh"

namespace spec {

namespace {

constexpr int kCommitThreads = 256;
constexpr int kSliceBytes = 32 * 1024;  // shared staging per slice (K and V of all L rows)

__global__ void __launch_bounds__(kCommitThreads) commit_kernel(CommitParams a) {
  pdl_wait();
  pdl_trigger();
  const int req = blockIdx.x, grp = blockIdx.y, G = gridDim.y;
  const int n = a.n, W = a.W, tid = threadIdx.x;
  __shared__ int src[kMaxN + 1], dst[kMaxN + 1], unit_s[kMaxN], dst_unit_s[kMaxN + 1];
  __shared__ int s_ok;
  __shared__ uint4 stage[kSliceBytes / 16];
  int* stage_free = reinterpret_cast<int*>(a.partials) + size_t(req) * n;
  int* counts = reinterpret_cast<int*>(a.partials) + size_t(a.b) * n;

  // round trip 1: the request's scalars, its accept_index row and (group 0)
  // its verify slots, all independent
  const int L0 = a.accept_lens[req];
  const int s0 = a.seq_lens[req];
  const int rq = a.req_pool_idx[req];
  const int ai = tid < W ? a.accept_index[size_t(req) * W + tid] : -1;
  const int vslot = (grp == 0 && tid < n) ? a.verify_loc[size_t(req) * n + tid] : -1;
  const bool len_ok = L0 >= 1 && L0 <= W && s0 >= 0 && s0 + L0 <= a.row_w;
  const bool rq_ok = rq >= 0 && rq < a.req_rows;
  if (tid == 0) {
    if (!len_ok) raise_error(a.error, SPEC_DEV_LENGTH);
    if (!rq_ok) raise_error(a.error, SPEC_DEV_INDEX);
    s_ok = len_ok && rq_ok;
  }
  const int L = (len_ok && rq_ok) ? L0 : 0;
  __syncthreads();
  // round trip 2: source slots (through accept_index) and target slots
  if (tid < L) {
    const int sl = (ai >= 0 && ai < a.b * n) ? a.verify_loc[ai] : -1;
    const int dl = a.req_to_token[size_t(rq) * a.row_w + s0 + tid];
    if (sl < 0 || sl >= a.num_slots || dl < 0 || dl >= a.num_slots) {
      raise_error(a.error, SPEC_DEV_INDEX);
      atomicExch(&s_ok, 0);
    }
    src[tid] = sl;
    dst[tid] = dl;
  }
  __syncthreads();
  const bool ok = s_ok;

  if (ok) {
    const int units = a.Hkv * a.D * 2 / 16;  // 16-byte units per slot row
    const int slice = max(1, min(units, kSliceBytes / 16 / (2 * L)));
    for (int layer = grp; layer < a.num_layers; layer += G) {
      const uint4* kin = static_cast<const uint4*>(a.k_layers[layer]);
      const uint4* vin = static_cast<const uint4*>(a.v_layers[layer]);
      uint4* kout = static_cast<uint4*>(a.k_layers[layer]);
      uint4* vout = static_cast<uint4*>(a.v_layers[layer]);
      for (int c0 = 0; c0 < units; c0 += slice) {
        const int cw = min(slice, units - c0);
        const int tot = 2 * L * cw;
        for (int t = tid; t < tot; t += blockDim.x) {
          const int which = t / (L * cw), rem = t % (L * cw), kk = rem / cw, col = rem % cw;
          const uint4* pool = which ? vin : kin;
          stage[t] = pool[size_t(src[kk]) * units + c0 + col];
        }
        __syncthreads();
        for (int t = tid; t < tot; t += blockDim.x) {
          const int which = t / (L * cw), rem = t % (L * cw), kk = rem / cw, col = rem % cw;
          uint4* pool = which ? vout : kout;
          pool[size_t(dst[kk]) * units + c0 + col] = stage[t];
        }
        __syncthreads();
      }
    }
  }

  if (grp == 0) {
    if (tid == 0) a.new_seq_lens[req] = s0 + (ok ? L : 0);
    // free units of this request, in ascending node order: node j's unit
    // (slot, or page = slot / page_size) is released when no target slot of
    // the request lies in it, at the first node that holds it.  One node per
    // thread.
    const int ps = a.page_size;
    if (tid < L) dst_unit_s[tid] = int(dst[tid] / ps);
    if (tid < n) unit_s[tid] = (vslot >= 0 && vslot < a.num_slots) ? vslot / ps : -1;
    __syncthreads();
    bool free_j = false;
    if (tid < n && ok) {
      const int u = unit_s[tid];
      if (u < 0) {
        raise_error(a.error, SPEC_DEV_INDEX);
      } else {
        bool kept = false;
        for (int kk = 0; kk < L && !kept; ++kk) kept = dst_unit_s[kk] == u;
        bool listed = false;
        for (int jj = 0; jj < tid && !listed; ++jj) listed = unit_s[jj] == u;
        free_j = !kept && !listed;
      }
    }
    // compaction in node order (n <= 64: the first two warps)
    __shared__ int warp_cnt[2];
    if (tid < 64) {
      const unsigned bal = __ballot_sync(0xffffffffu, free_j);
      if ((tid & 31) == 0) warp_cnt[tid >> 5] = __popc(bal);
    }
    __syncthreads();
    if (tid < 64) {
      const unsigned bal = __ballot_sync(0xffffffffu, free_j);
      const int before = (tid >= 32 ? warp_cnt[0] : 0) + __popc(bal & ((1u << (tid & 31)) - 1u));
      if (free_j) stage_free[before] = unit_s[tid];
      if (tid == 0) counts[req] = warp_cnt[0] + warp_cnt[1];
    }
  }

  // only the group-0 CTAs stage free lists; the others are done
  if (grp != 0 || !arrive_last(a.counters, uint32_t(a.b))) return;

  // ---- the last group-0 CTA concatenates the staged lists in request
  // order: per block of requests, the counts and every staged entry are
  // loaded together (one round trip), then an exclusive scan of the counts
  // places the entries ----
  __shared__ int warp_sum[kCommitThreads / 32];
  __shared__ int s_off[kCommitThreads], s_cnt[kCommitThreads];
  __shared__ int s_running;
  if (tid == 0) s_running = 0;
  __syncthreads();
  const int lane = tid & 31, w = tid >> 5, nw = blockDim.x >> 5;
  // requests per block: each thread holds at most kEnt staged entries
  constexpr int kEnt = 8;
  const int rblk = max(1, min(int(blockDim.x), kEnt * int(blockDim.x) / n));
  for (int r0 = 0; r0 < a.b; r0 += rblk) {
    const int nr = min(rblk, a.b - r0);
    const int r = r0 + tid;
    const int c = tid < nr ? __ldcg(counts + r) : 0;
    const int* from = reinterpret_cast<const int*>(a.partials) + size_t(r0) * n;
    int ent[kEnt];
#pragma unroll
    for (int j = 0; j < kEnt; ++j) {
      const int x = tid + j * int(blockDim.x);
      ent[j] = x < nr * n ? __ldcg(from + x) : 0;
    }
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sum[w] = incl;
    __syncthreads();
    int before = s_running;
    for (int q = 0; q < w; ++q) before += warp_sum[q];
    s_off[tid] = before + incl - c;
    s_cnt[tid] = c;
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kEnt; ++j) {
      const int x = tid + j * int(blockDim.x);
      if (x < nr * n) {
        const int ri = x / n, e = x - ri * n;
        if (e < s_cnt[ri]) a.free_ids[s_off[ri] + e] = ent[j];
      }
    }
    __syncthreads();
    if (tid == 0) {
      int tot = 0;
      for (int q = 0; q < nw; ++q) tot += warp_sum[q];
      s_running += tot;
    }
    __syncthreads();
  }
  if (tid == 0) *a.n_free = s_running;
  counter_reset(a.counters);
}

}  // namespace

size_t commit_partial_bytes(int b, int n) { return align256(size_t(b) * n * 4 + size_t(b) * 4); }

int launch_commit_kv(const CommitParams& p, cudaStream_t stream) {
  // layer groups: enough CTAs to spread deep models over the SMs
  int G = p.num_layers;
  const int cap = p.b > 0 ? (kTargetCtas + p.b - 1) / p.b : 1;
  if (G > cap) G = cap;
  if (G < 1) G = 1;
  if (launch_pdl(commit_kernel, dim3(p.b, G), dim3(kCommitThreads), 0, stream, p) != cudaSuccess)
    return SPEC_ERR_LAUNCH;
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
}

}  // namespace spec
