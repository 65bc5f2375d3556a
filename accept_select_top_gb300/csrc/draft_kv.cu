// draft_kv.cu -- the draft side of the KV: where the draft steps write, the
// prefix-tail copy of paged branches, and the materialised verify mask.
//
// [SGL-XI draft 前向的输入准备:prepare_for_draft -- assign_draft_cache_locs
// (contiguous slots per draft row for page_size 1 or topk 1, the first draft
// row's position in the same call), duplicate_prefix_tail_to_draft_branches
// (each branch's page-aligned region starts with holes over the prefix's last
// partial page, filled with the real prefix-tail KV so whole-page reads stay
// coherent)], [EVOL 草稿、验证与槽位 (the last partial page is duplicated)],
// [SGL-XI 三种 mask 形态 (FULL_MASK; fill_prefix_mask skips the prefix columns)].
//
// All three are small: slot lookups, a few KV rows per branch, and a byte mask
// written once (HBM-bound for long prefixes: 16-byte stores).
#include "common.cuh"
#include "kernels.cuh"

namespace spec {

namespace {

// Region geometry of paged branches: holes, page-aligned base, region span.
struct BranchRegion {
  int last_page, prefix_base, R;
  __device__ __forceinline__ BranchRegion(int L, int S, int page) {
    last_page = L % page;
    prefix_base = L - last_page;
    R = (last_page + S + page - 1) / page * page;
  }
};

__global__ void __launch_bounds__(256) assign_draft_locs_kernel(DraftLocParams a) {
  pdl_wait();
  pdl_trigger();
  const int g = blockIdx.x * blockDim.x + threadIdx.x;
  const int per_req = a.topk * a.S;
  if (g >= a.b * per_req) return;
  const int req = g / per_req, t = (g % per_req) / a.S, s = g % a.S;
  const int L = a.seq_lens[req];
  const int rq = a.req_pool_idx[req];
  long pos;
  if (a.page_size == 1 || a.topk == 1) {
    pos = long(L) + long(t) * a.S + s;  // each branch's steps are contiguous after the prefix
  } else {
    const BranchRegion br(L, a.S, a.page_size);
    pos = long(br.prefix_base) + long(t) * br.R + br.last_page + s;
  }
  int slot = -1;
  if (L < 0 || rq < 0 || rq >= a.req_rows || pos >= a.row_w) {
    raise_error(a.error, SPEC_DEV_INDEX);
  } else {
    slot = a.req_to_token[size_t(rq) * a.row_w + pos];
    if (slot < 0 || slot >= a.num_slots) {
      raise_error(a.error, SPEC_DEV_INDEX);
      slot = -1;
    }
  }
  a.out_cache_loc[g] = slot;
  if (a.positions && a.topk == 1 && s == 0) a.positions[req] = L;
}

// CTA (request, branch t >= 1): the last_page prefix-tail rows of every layer,
// K and V, into the branch's hole slots, 16 bytes per thread per step.
__global__ void __launch_bounds__(256) duplicate_prefix_tail_kernel(DupTailParams a) {
  pdl_wait();
  pdl_trigger();
  const int req = blockIdx.y, t = blockIdx.x + 1;
  __shared__ int src[64], dst[64];  // last_page < page_size <= 64
  __shared__ int s_n;
  const int L = a.seq_lens[req];
  const int rq = a.req_pool_idx[req];
  if (L < 0 || rq < 0 || rq >= a.req_rows) {
    if (threadIdx.x == 0) raise_error(a.error, SPEC_DEV_INDEX);
    return;
  }
  const BranchRegion br(L, a.S, a.page_size);
  if (threadIdx.x == 0) s_n = br.last_page;
  if (int(threadIdx.x) < br.last_page) {  // last_page < page_size <= 64 (checked on the host)
    const long sp = long(br.prefix_base) + threadIdx.x;
    const long dp = long(br.prefix_base) + long(t) * br.R + threadIdx.x;
    int sl = -1, dl = -1;
    if (sp < a.row_w && dp < a.row_w) {
      sl = a.req_to_token[size_t(rq) * a.row_w + sp];
      dl = a.req_to_token[size_t(rq) * a.row_w + dp];
    }
    if (sl < 0 || sl >= a.num_slots || dl < 0 || dl >= a.num_slots) {
      raise_error(a.error, SPEC_DEV_INDEX);
      sl = dl = -1;
    }
    src[threadIdx.x] = sl;
    dst[threadIdx.x] = dl;
  }
  __syncthreads();
  const int units = a.Hkv * a.D * 2 / 16;  // 16-byte units of one slot row
  const int per_layer = 2 * s_n * units;  // K and V rows of the tail
  for (int e = threadIdx.x; e < a.num_layers * per_layer; e += blockDim.x) {
    const int layer = e / per_layer, r = e % per_layer;
    const int which = r / (s_n * units), j = (r / units) % s_n, u = r % units;
    if (src[j] < 0) continue;
    uint4* pool = static_cast<uint4*>(which ? a.v_layers[layer] : a.k_layers[layer]);
    pool[size_t(dst[j]) * units + u] = pool[size_t(src[j]) * units + u];
  }
}

// The byte of the FULL_MASK at flat index e, given its request's block
// (offset off, prefix L, n tree nodes): 1 in the prefix columns, else the
// tree bit.
__device__ __forceinline__ uint8_t mask_byte(long e, long off, int L, int n, const uint64_t* bits, int req) {
  const long x = e - off;
  const int w = L + n;
  const int i = int(x / w), j = int(x % w);
  if (j < L) return 1;
  return uint8_t((bits[size_t(req) * n + i] >> (j - L)) & 1u);
}

// fill_prefix: every byte of the flat mask, in 16-byte groups (grid-stride);
// a group inside one row's prefix is a constant store.  Request offsets are
// a prefix sum of n * (L + n) over the requests, built once per CTA in
// shared memory (dynamic: 8 bytes per request).
__global__ void __launch_bounds__(256) full_mask_kernel(FullMaskParams a) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ long long offs[];  // [b + 1]
  __shared__ long long s_carry;
  const int n = a.n;
  if (threadIdx.x == 0) s_carry = 0;
  __syncthreads();
  int bad = 0;
  for (int r0 = 0; r0 < a.b; r0 += blockDim.x) {
    const int r = r0 + threadIdx.x;
    const int L = r < a.b ? a.seq_lens[r] : 0;
    bad |= L < 0;
    long long v = r < a.b ? (long long)n * ((L < 0 ? 0 : L) + n) : 0;
    // inclusive block scan of v
    __shared__ long long wsum[256 / 32];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    if (lane == 31) wsum[w] = v;
    __syncthreads();
    long long before = s_carry;
    for (int q = 0; q < w; ++q) before += wsum[q];
    if (r < a.b) offs[r + 1] = before + v;
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) s_carry = before + v;
    __syncthreads();
  }
  if (threadIdx.x == 0) offs[0] = 0;
  // a negative length has no block: nothing is written
  if (__syncthreads_or(bad)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) raise_error(a.error, SPEC_DEV_LENGTH);
    return;
  }
  const long long total = offs[a.b];
  if (total > (long long)a.mask_bytes) {
    if (blockIdx.x == 0 && threadIdx.x == 0) raise_error(a.error, SPEC_DEV_LENGTH);
    return;
  }
  uint8_t* m = a.mask;
  // 16-byte groups of the flat buffer: [head, aligned body, tail]
  const long long head = (16 - (reinterpret_cast<uintptr_t>(m) & 15)) & 15;
  const long long first = head < total ? head : total;
  const long long groups = (total - first) / 16;
  const long long tail0 = first + groups * 16;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  auto req_of = [&](long long e) {  // the request whose block holds byte e
    int lo = 0, hi = a.b - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (offs[mid] <= e) lo = mid;
      else hi = mid - 1;
    }
    return lo;
  };
  for (long long e = tid; e < first; e += stride) {
    const int r = req_of(e);
    m[e] = mask_byte(e, offs[r], a.seq_lens[r], n, a.mask_bits, r);
  }
  for (long long e = tail0 + tid; e < total; e += stride) {
    const int r = req_of(e);
    m[e] = mask_byte(e, offs[r], a.seq_lens[r], n, a.mask_bits, r);
  }
  for (long long g = tid; g < groups; g += stride) {
    const long long e0 = first + g * 16;
    int r = req_of(e0);
    const int L = a.seq_lens[r];
    const long long x = e0 - offs[r];
    const long long w = L + n;
    const long long col = x % w;
    uint32_t wd[4] = {0x01010101u, 0x01010101u, 0x01010101u, 0x01010101u};  // inside one row's prefix
    if (!(col + 16 <= L)) {
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const long long e = e0 + u;
        while (r + 1 < a.b && offs[r + 1] <= e) ++r;  // a group may cross into the next request
        const uint32_t byte = mask_byte(e, offs[r], a.seq_lens[r], n, a.mask_bits, r);
        wd[u >> 2] = (wd[u >> 2] & ~(0xffu << (8 * (u & 3)))) | (byte << (8 * (u & 3)));
      }
    }
    *reinterpret_cast<uint4*>(m + e0) = make_uint4(wd[0], wd[1], wd[2], wd[3]);  // 16-byte aligned
  }
}

// fill_prefix off: only the n tree columns of every row are written (one
// thread per tree byte); the prefix columns keep what the buffer holds.
__global__ void __launch_bounds__(256) full_mask_tree_kernel(FullMaskParams a) {
  pdl_wait();
  pdl_trigger();
  const int n = a.n;
  const long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= (long long)a.b * n * n) return;
  const int r = int(g / (n * n)), i = int(g / n % n), j = int(g % n);
  long long off = 0;
  bool bad = false;
  for (int q = 0; q < r; ++q) {
    const int Lq = a.seq_lens[q];
    bad |= Lq < 0;
    off += (long long)n * (Lq + n);
  }
  const int L = a.seq_lens[r];
  const long long e = off + (long long)i * (L + n) + L + j;
  if (bad || L < 0 || e < 0 || e >= (long long)a.mask_bytes) {
    raise_error(a.error, SPEC_DEV_LENGTH);
    return;
  }
  a.mask[e] = uint8_t((a.mask_bits[size_t(r) * n + i] >> j) & 1u);
}

}  // namespace

int launch_assign_draft_locs(const DraftLocParams& p, cudaStream_t stream) {
  const int total = p.b * p.topk * p.S;
  if (launch_pdl(assign_draft_locs_kernel, dim3((total + 255) / 256), dim3(256), 0, stream, p) != cudaSuccess)
    return SPEC_ERR_LAUNCH;
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
}

int launch_duplicate_prefix_tail(const DupTailParams& p, cudaStream_t stream) {
  if (p.topk < 2 || p.page_size < 2) return SPEC_OK;  // nothing to copy
  if (launch_pdl(duplicate_prefix_tail_kernel, dim3(p.topk - 1, p.b), dim3(256), 0, stream, p) != cudaSuccess)
    return SPEC_ERR_LAUNCH;
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
}

int launch_full_mask(const FullMaskParams& p, cudaStream_t stream) {
  cudaError_t e;
  if (p.fill_prefix) {
    const size_t smem = sizeof(long long) * (size_t(p.b) + 1);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(full_mask_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
            cudaSuccess)
      return SPEC_ERR_LAUNCH;
    // about four 16-byte groups per thread, at most 8 CTAs per SM
    const long long groups = (long long)(p.mask_bytes / 16) + 1;
    long long ctas = (groups + 4 * 256 - 1) / (4 * 256);
    if (ctas > 8LL * 152) ctas = 8LL * 152;
    if (ctas < 1) ctas = 1;
    e = launch_pdl(full_mask_kernel, dim3(unsigned(ctas)), dim3(256), smem, stream, p);
  } else {
    const long long total = (long long)p.b * p.n * p.n;
    e = launch_pdl(full_mask_tree_kernel, dim3(unsigned((total + 255) / 256)), dim3(256), 0, stream, p);
  }
  if (e != cudaSuccess) return SPEC_ERR_LAUNCH;
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
}

}  // namespace spec
