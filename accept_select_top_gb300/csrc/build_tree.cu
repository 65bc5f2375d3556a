// build_tree.cu -- organize_draft_results followed by build_tree, one CTA per
// request.
//
// [SGL-XI organize_draft_results (topk over the score list, sort of the
// indices, gather of the tokens, parent list)], [SGL-XI build_tree_kernel_efficient
// (bonus token at node 0, positions = prefix + depth, retrieve_* child/sibling
// arrays, bit-packed QLEN_ONLY mask)], [ACCEPT section 2], [EAGLE2 sections 4.3, 5.3].
//
// Steps inside the CTA (all in shared memory):
//   1. rank every score position among the C positions (value desc, index
//      asc); the n-1 with rank < n-1 are selected;
//   2. compact the selected positions in ascending order (warp ballots) ->
//      node j = 1 + its rank among the selected positions;
//   3. parent of node j: position parent_space[p / k] (-1 = root) mapped back
//      to its node through a position -> node table;
//   4. ancestors by walking parent pointers (<= n steps): mask row, depth;
//   5. first child / next sibling by scanning the parent array.
#include "common.cuh"
#include "kernels.cuh"

namespace spec {

namespace {

constexpr int kBuildThreads = 512;

__global__ void __launch_bounds__(kBuildThreads) build_tree_kernel(BuildParams a) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ unsigned char smem_raw[];
  const int req = blockIdx.x;
  const int C = a.k + (a.S - 1) * a.k * a.k;
  const int P = 1 + (a.S - 1) * a.k;
  const int n = a.n, need = n - 1;
  float* sc = reinterpret_cast<float*>(smem_raw);                      // [C]
  int* node_of = reinterpret_cast<int*>(sc + C);                       // [C]
  int* tok = node_of + C;                                              // [C]
  int* prow_s = tok + C;                                               // [P]
  unsigned char* sel = reinterpret_cast<unsigned char*>(prow_s + P);  // [C]
  __shared__ int sel_pos[kMaxN];
  __shared__ int par[kMaxN];
  __shared__ int warp_base[kBuildThreads / 32 + 1];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, nw = blockDim.x >> 5;

  // one round trip: the request's scores, tokens, parent list, prefix length
  // and bonus token (nothing below reads global memory again)
  const float* srow = a.score_space + size_t(req) * C;
  const int* trow = a.token_space + size_t(req) * C;
  const int* prow = a.parent_space + size_t(req) * P;
  __shared__ int s_len, s_bonus;
  for (int p = tid; p < C; p += blockDim.x) {
    const float v = srow[p];
    const int t = trow[p];
    sc[p] = v;
    tok[p] = t;
  }
  for (int t = tid; t < P; t += blockDim.x) prow_s[t] = prow[t];
  if (tid == 0) {
    s_len = a.seq_lens[req];
    s_bonus = a.bonus[req];
  }
  __syncthreads();

  // 1. selection by rank (counting stops once n-1 better ones are found)
  for (int p = tid; p < C; p += blockDim.x) {
    const float v = sc[p];
    int rank = 0;
    int q = 0;
    for (; q + 8 <= C && rank < need; q += 8) {  // eight independent reads per check
#pragma unroll
      for (int u = 0; u < 8; ++u) rank += better(sc[q + u], q + u, v, p);
    }
    for (; q < C && rank < need; ++q) rank += better(sc[q], q, v, p);
    sel[p] = rank < need;
    node_of[p] = -1;
  }
  __syncthreads();

  // 2. ascending compaction: each warp counts its contiguous slice, then assigns
  const int per_warp = (C + nw - 1) / nw;
  const int lo = w * per_warp, hi = min(C, lo + per_warp);
  int cnt = 0;
  for (int p0 = lo; p0 < hi; p0 += 32) {
    const int p = p0 + lane;
    cnt += __popc(__ballot_sync(0xffffffffu, p < hi && sel[p]));
  }
  if (lane == 0) warp_base[w + 1] = cnt;
  __syncthreads();
  if (tid == 0) {
    warp_base[0] = 0;
    for (int i = 1; i <= nw; ++i) warp_base[i] += warp_base[i - 1];
  }
  __syncthreads();
  int base = warp_base[w];
  for (int p0 = lo; p0 < hi; p0 += 32) {
    const int p = p0 + lane;
    const bool s = p < hi && sel[p];
    const unsigned bal = __ballot_sync(0xffffffffu, s);
    if (s) {
      const int j = base + __popc(bal & ((1u << lane) - 1));
      if (j < need) {
        sel_pos[j] = p;
        node_of[p] = j + 1;
      }
    }
    base += __popc(bal);
  }
  __syncthreads();

  // 3. parents
  for (int j = tid; j < n; j += blockDim.x) {
    if (j == 0) {
      par[0] = -1;
      continue;
    }
    const int p = sel_pos[j - 1];
    const int t = p / a.k;
    int parent = 0;
    const int ppos = t < P ? prow_s[t] : -2;
    if (ppos >= 0 && ppos < C && node_of[ppos] > 0 && node_of[ppos] < j) {
      parent = node_of[ppos];
    } else if (ppos != -1) {
      raise_error(a.error, SPEC_DEV_INVARIANT);
    }
    par[j] = parent;
  }
  __syncthreads();

  // 4.-5. per node outputs
  const size_t rb = size_t(req) * n;
  for (int i = tid; i < n; i += blockDim.x) {
    uint64_t m = 0;
    int depth = -1, x = i;
    for (int g = 0; x >= 0 && g <= n; ++g) {
      m |= uint64_t(1) << x;
      ++depth;
      x = par[x];
    }
    int first = -1;
    for (int c = i + 1; c < n && first < 0; ++c)
      if (par[c] == i) first = c;
    int sib = -1;
    if (i > 0)
      for (int c = i + 1; c < n && sib < 0; ++c)
        if (par[c] == par[i]) sib = c;
    a.mask_bits[rb + i] = m;
    a.positions[rb + i] = s_len + depth;
    a.retrieve_index[rb + i] = int(rb + i);
    a.next_token[rb + i] = first;
    a.next_sibling[rb + i] = sib;
    a.draft_tokens[rb + i] = i == 0 ? s_bonus : tok[sel_pos[i - 1]];
  }
}

// build_chain_tree [SGL-XI 平台分派与 chain 特化]: with topk = 1 and
// num_draft_tokens = num_steps + 1 the tree is a chain whose structure is
// constant (node i hangs below node i - 1, the mask is lower triangular); one
// thread per node writes it, reading only its own token and the request's
// prefix length.
__global__ void __launch_bounds__(256) build_chain_kernel(ChainParams a) {
  pdl_wait();
  pdl_trigger();
  const int n = a.S + 1;
  const int g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= a.b * n) return;
  const int req = g / n, i = g - req * n;
  const int tok = i == 0 ? a.bonus[req] : a.draft_tokens[size_t(req) * a.draft_ld + i - 1];
  a.tree_tokens[g] = tok;
  a.positions[g] = a.seq_lens[req] + i;
  a.retrieve_index[g] = g;
  a.next_token[g] = i + 1 < n ? i + 1 : -1;
  a.next_sibling[g] = -1;
  a.mask_bits[g] = i == 63 ? ~uint64_t(0) : (uint64_t(1) << (i + 1)) - 1;  // nodes 0..i
}

}  // namespace

int launch_build_chain_tree(const ChainParams& p, cudaStream_t stream) {
  const int total = p.b * (p.S + 1);
  if (launch_pdl(build_chain_kernel, dim3((total + 255) / 256), dim3(256), 0, stream, p) != cudaSuccess)
    return SPEC_ERR_LAUNCH;
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
}

size_t build_tree_smem_bytes(int k, int S) {
  const size_t C = size_t(k) + size_t(S - 1) * k * k;
  const size_t P = 1 + size_t(S - 1) * k;
  return C * (sizeof(float) + 2 * sizeof(int) + 1) + P * sizeof(int);
}

int launch_build_tree(const BuildParams& p, cudaStream_t stream) {
  const size_t smem = build_tree_smem_bytes(p.k, p.S);
  if (smem > 200 * 1024) return SPEC_ERR_ARG;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(build_tree_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
    return SPEC_ERR_LAUNCH;
  if (launch_pdl(build_tree_kernel, dim3(p.b), dim3(kBuildThreads), smem, stream, p) != cudaSuccess)
    return SPEC_ERR_LAUNCH;
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
}

}  // namespace spec
