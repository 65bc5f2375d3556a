// attention_tc.cu -- tree-masked verify attention on the tcgen05 tensor cores.
//
// [EAGLE2 sections 4.2-4.3: the verify queries are the flattened tree nodes,
// the keys are the cached history (all visible) plus the tree nodes, of which a
// query sees only its ancestors and itself; history KV is read once and shared
// by all candidates], [SGL-XI QLEN_ONLY mask: prefix columns implicitly visible].
//
// One CTA = 128 query rows of one (request, kv head) -- row r is (node r / G,
// q head g*G + r % G), G = Hq / Hkv -- and one split of that request's key list
// (prefix positions, then the n tree nodes), 128 keys per pipeline stage:
//   warp 0      TMA producer: per tile, looks the 128 keys' slots up
//               (req_to_token / verify_loc) and gathers their K and V rows
//               (cp.async.bulk.tensor tile::gather4, 128B swizzle) into one of
//               two shared-memory stages;
//   warp 1      MMA issuer (one thread): S = Q K^T (M=128, N=128, K=D) into one
//               of two TMEM S buffers; O += P V (M=128, N=64 per half, K=128)
//               with P read from TMEM;
//   warps 2..5  one query row per thread: masked online softmax of the S row
//               (tcgen05.ld), P written back over S as bf16 (tcgen05.st), lazy
//               rescaling of O in TMEM, and the epilogue.
// Partials (unnormalised O, running max, sum) go to the workspace and
// attention_merge_kernel combines the splits.
//
// TMEM columns: O [0, D), S0 [128, 256), S1 [256, 384); P(b) aliases the first
// 64 columns of S(b).  Every mbarrier wait is bounded: on timeout the CTA sets
// SPEC_DEV_TIMEOUT, stops, drains what it issued and frees its TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace spec {

namespace {

constexpr int kRows = 128;
constexpr int kKeys = 64;
constexpr int kStages = 2;
constexpr int kTcThreads = 192;
constexpr uint32_t kTmemCols = 256;  // two CTAs share an SM's 512 columns
constexpr uint32_t kColO = 0;
// S buffer b lives at TMEM columns [128 + 64 b, 192 + 64 b)
__host__ __device__ constexpr uint32_t col_s(int b) { return 128u + 64u * uint32_t(b); }
constexpr float kRescaleLog2 = 8.f;       // O is rescaled only when the row max grows by more than 2^8
constexpr long long kWaitCycles = 4000000000ll;  // ~2 s at 2 GHz: bound of every mbarrier wait

template <int D>
struct Smem {
  static constexpr int kHalves = D / 64;
  static constexpr int kQBlock = kRows * 128;      // [128 rows x 64 bf16], 128B-swizzled: 16 KB
  static constexpr int kQTile = kHalves * kQBlock;
  static constexpr int kKBlock = kKeys * 128;      // [64 keys x 64 bf16]: 8 KB
  static constexpr int kKTile = kHalves * kKBlock; // a K or V tile
  static constexpr int kQ = 0;
  static constexpr int kStage = kQTile;            // stage s: K at kStage + 2*s*kKTile, V at + kKTile
  static constexpr int kFlags = kStage + kStages * 2 * kKTile;  // per stage: 4 words of key flags
  static constexpr int kBars = kFlags + 64;
  static constexpr int kBytes = kBars + 256;
  static constexpr int kTx = 2 * kKTile;           // bytes one stage receives
};

// barriers (uint64 each), by index
enum { kFull0 = 0, kFull1, kEmpty0, kEmpty1, kQFull, kSFull0, kSFull1, kPReady0, kPReady1, kODone, kDrain, kNumBars };

// ------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase of the given parity: false once kWaitCycles SM
// cycles have passed (try_wait itself may suspend the thread for a while).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long start = clock64();
  while (clock64() - start < kWaitCycles)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* tm, int x, int y0, int y1, int y2, int y3,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: 128B swizzle, descriptor version 1.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return uint64_t((saddr >> 4) & 0x3FFFu) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
         (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// Instruction descriptor of kind::f16: bf16 A and B, f32 accumulator.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) | (uint32_t(N >> 3) << 17) |
         (uint32_t(M >> 4) << 24);
}

__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(
          d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// 32 consecutive TMEM columns of this thread's lane, waited for.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
      " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive TMEM columns of this thread's lane, then wait for the store.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14,"
      " %15, %16};\n"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st32f(uint32_t taddr, const float (&v)[32]) {
  uint32_t a[16], b[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    a[i] = __float_as_uint(v[i]);
    b[i] = __float_as_uint(v[16 + i]);
  }
  tmem_st16(taddr, a);
  tmem_st16(taddr + 16, b);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  // round to nearest even, lower key in the low half
  uint32_t a = __float_as_uint(lo), b = __float_as_uint(hi);
  a += 0x7fffu + ((a >> 16) & 1u);
  b += 0x7fffu + ((b >> 16) & 1u);
  return (a >> 16) | (b & 0xffff0000u);
}

struct TcArgs {
  AttentionParams p;
  int m_tiles;
  int split_tiles;
};

// Per-stage key flags (4 words in shared memory):
//   [0] bit j: key 2j of the tile has a valid slot      [1] same for key 2j+1
//   [2] 1 when every key of the tile is a valid prefix key (no masking needed)
__device__ __forceinline__ bool key_valid(const uint32_t* f, int c) { return (f[c & 1] >> (c >> 1)) & 1u; }

template <int D>
__global__ void __launch_bounds__(kTcThreads, 2)
    attention_tc_kernel(const __grid_constant__ TcArgs args, const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  using L = Smem<D>;
  const AttentionParams& a = args.p;
  const int G = a.Hq / a.Hkv, M = a.n * G;
  const int mt = blockIdx.x % args.m_tiles, g = blockIdx.x / args.m_tiles;
  const int req = blockIdx.y, split = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned FULL = 0xffffffffu;

  // ---- request geometry (bounds-checked) ----
  int Lp = a.seq_lens[req];
  const int rq = a.req_pool_idx[req];
  const bool req_ok = rq >= 0 && rq < a.req_rows;
  if (Lp < 0 || Lp > a.max_seq_len || Lp > a.row_w) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && split == 0) raise_error(a.error, SPEC_DEV_LENGTH);
    Lp = max(0, min(Lp, min(a.max_seq_len, a.row_w)));
  }
  if (!req_ok && threadIdx.x == 0 && blockIdx.x == 0 && split == 0) raise_error(a.error, SPEC_DEV_INDEX);
  const int total = req_ok ? Lp + a.n : 0;
  const int k0 = split * args.split_tiles * kKeys;
  const int k1 = min(total, k0 + args.split_tiles * kKeys);
  const int T = k0 < k1 ? (k1 - k0 + kKeys - 1) / kKeys : 0;
  const bool direct = a.splits == 1;  // one split: write the normalised output here

  float* po = reinterpret_cast<float*>(a.partials);
  float* pml = po + size_t(a.b) * a.n * a.Hq * a.splits * D;
  if (T == 0) {  // nothing in this split: an empty partial for every valid row
    if (!direct && threadIdx.x < kRows) {
      const int rg = mt * kRows + threadIdx.x;
      if (rg < M) {
        const size_t idx = ((size_t(req) * a.n + rg / G) * a.Hq + g * G + rg % G) * a.splits + split;
        pml[idx * 2] = -INFINITY;
        pml[idx * 2 + 1] = 0.f;
      }
    }
    return;
  }

  // ---- shared memory (1024-aligned for the 128B swizzle atoms) ----
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  unsigned char* sp = smem_raw + (sbase - raw);
  uint32_t* flags = reinterpret_cast<uint32_t*>(sp + L::kFlags);  // [stage][4]
  const uint32_t bars = sbase + L::kBars;
  auto bar = [&](int i) { return bars + 8u * uint32_t(i); };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sp + L::kBars + 8 * kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sp + L::kBars + 8 * kNumBars + 8);

  if (threadIdx.x == 0) {
    mbar_init(bar(kFull0), 1);
    mbar_init(bar(kFull1), 1);
    mbar_init(bar(kEmpty0), 1);
    mbar_init(bar(kEmpty1), 1);
    mbar_init(bar(kQFull), 1);
    mbar_init(bar(kSFull0), 1);
    mbar_init(bar(kSFull1), 1);
    mbar_init(bar(kPReady0), kRows);
    mbar_init(bar(kPReady1), kRows);
    mbar_init(bar(kODone), 1);
    mbar_init(bar(kDrain), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  auto fail = [&]() {
    raise_error(a.error, SPEC_DEV_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp == 0) {
    // =========================== TMA producer ===========================
    // Q rows 4*lane .. 4*lane+3 of this CTA
    {
      int y[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int rg = mt * kRows + 4 * lane + e;
        y[e] = rg < M ? (req * a.n + rg / G) * a.Hq + g * G + rg % G : -1;  // -1: zero-filled
      }
      if (lane == 0) mbar_expect_tx(bar(kQFull), L::kQTile);
      __syncwarp();
#pragma unroll
      for (int h = 0; h < L::kHalves; ++h)
        tma_gather4(sbase + L::kQ + h * L::kQBlock + 512u * lane, &tm_q, 64 * h, y[0], y[1], y[2], y[3],
                    bar(kQFull));
    }
    // Keys 2*lane and 2*lane+1 of tile t: the slot loads are issued one tile
    // ahead (issue) and their values consumed only after this tile's gathers
    // are out (finish), so the lookup latency hides behind the pipeline.
    auto issue = [&](int t, int (&slot)[2], int (&kind)[2]) {  // kind: 0 none, 1 prefix, 2 tree node
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int kg = k0 + t * kKeys + 2 * lane + e;
        slot[e] = -1;
        kind[e] = 0;
        if (kg < k1) {
          if (kg < Lp) {
            slot[e] = a.req_to_token[size_t(rq) * a.row_w + kg];
            kind[e] = 1;
          } else {
            slot[e] = a.verify_loc[size_t(req) * a.n + (kg - Lp)];
            kind[e] = 2;
          }
        }
      }
    };
    auto finish = [&](const int (&slot)[2], const int (&kind)[2], int (&row)[2], bool (&pre)[2]) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const bool ok_slot = slot[e] >= 0 && slot[e] < a.num_slots;
        if (kind[e] != 0 && !ok_slot) raise_error(a.error, SPEC_DEV_INDEX);
        const bool v = kind[e] != 0 && ok_slot;
        row[e] = v ? int(slot[e] * a.Hkv + g) : -1;  // -1: zero-filled, masked out
        pre[e] = v && kind[e] == 1;
      }
    };
    int row[2], slot_n[2], kind_n[2];
    bool pre[2];
    issue(0, slot_n, kind_n);
    finish(slot_n, kind_n, row, pre);
    int issued = 0;
    for (int t = 0; t < T; ++t) {
      const int s = t & 1;
      if (t + 1 < T) issue(t + 1, slot_n, kind_n);  // in flight while this warp waits
      const bool e_ok = (t < 2 || mbar_wait(bar(kEmpty0 + s), ((t >> 1) - 1) & 1)) && !*abort_flag;
      if (!__all_sync(FULL, e_ok)) {  // the warp leaves the loop together
        if (!*abort_flag) fail();
        break;
      }
      const unsigned v0 = __ballot_sync(FULL, row[0] >= 0), v1 = __ballot_sync(FULL, row[1] >= 0);
      const bool all_pre = __all_sync(FULL, pre[0] && pre[1]);
      if (lane == 0) {
        flags[4 * s + 0] = v0;
        flags[4 * s + 1] = v1;
        flags[4 * s + 2] = all_pre ? 1u : 0u;
        mbar_expect_tx(bar(kFull0 + s), L::kTx);
      }
      // lane l gathers keys 4(l%16) .. 4(l%16)+3 of K (l < 16) or V (l >= 16)
      const int grp = lane & 15;
      const int y0 = __shfl_sync(FULL, row[0], 2 * grp), y1 = __shfl_sync(FULL, row[1], 2 * grp);
      const int y2 = __shfl_sync(FULL, row[0], 2 * grp + 1), y3 = __shfl_sync(FULL, row[1], 2 * grp + 1);
      __syncwarp();
      const bool is_v = lane >= 16;
      const uint32_t dst = sbase + L::kStage + 2u * s * L::kKTile + (is_v ? L::kKTile : 0) + 512u * grp;
#pragma unroll
      for (int h = 0; h < L::kHalves; ++h)
        tma_gather4(dst + h * L::kKBlock, is_v ? &tm_v : &tm_k, 64 * h, y0, y1, y2, y3, bar(kFull0 + s));
      issued = t + 1;
      if (t + 1 < T) finish(slot_n, kind_n, row, pre);
    }
    // drain: every stage this warp filled has landed before the CTA can exit
    for (int t = max(0, issued - 2); t < issued; ++t) mbar_wait(bar(kFull0 + (t & 1)), (t >> 1) & 1);
  } else if (warp == 1) {
    // ============================ MMA issuer ============================
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(kRows, kKeys, false);
      constexpr uint32_t idesc_pv = idesc_bf16(kRows, 64, true);
      auto issue_pv = [&](int u) -> bool {
        const int b = u & 1;
        if (!mbar_wait(bar(kPReady0 + b), (u >> 1) & 1)) return false;
        if (*abort_flag) return false;
        tc_fence_after();
        const uint32_t vbase = sbase + L::kStage + 2u * b * L::kKTile + L::kKTile;
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk) {
#pragma unroll
          for (int h = 0; h < L::kHalves; ++h) {
            // V half h, keys 16kk..16kk+15: MN-major, 8-key groups 1024 B apart
            const uint64_t bd = sdesc(vbase + h * L::kKBlock + kk * 16 * 128, 1024, 1024);
            mma_ts(tmem + kColO + 64 * h, tmem + col_s(b) + 8 * kk, bd, idesc_pv, (u > 0 || kk > 0) ? 1u : 0u);
          }
        }
        mma_commit(bar(kODone));
        mma_commit(bar(kEmpty0 + b));
        return true;
      };
      bool ok = mbar_wait(bar(kQFull), 0);
      if (!ok) fail();
      for (int t = 0; ok && t < T; ++t) {
        const int s = t & 1;
        if (!mbar_wait(bar(kFull0 + s), (t >> 1) & 1) || *abort_flag) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t kbase = sbase + L::kStage + 2u * s * L::kKTile;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ko = (kk >> 2) * L::kKBlock + (kk & 3) * 32;
          const uint32_t qo = (kk >> 2) * L::kQBlock + (kk & 3) * 32;
          const uint64_t ad = sdesc(sbase + L::kQ + qo, 16, 1024);
          const uint64_t bd = sdesc(kbase + ko, 16, 1024);
          mma_ss(tmem + col_s(s), ad, bd, idesc_qk, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(kSFull0 + s));
        if (t >= 1 && !issue_pv(t - 1)) {
          ok = false;
          break;
        }
      }
      if (ok) ok = issue_pv(T - 1);
      if (!ok && !*abort_flag) fail();
      // drain: every MMA issued has completed before TMEM is released
      mma_commit(bar(kDrain));
      mbar_wait(bar(kDrain), 0);
    }
    __syncwarp();
  } else {
    // ============================ softmax rows ============================
    // tcgen05.ld / tcgen05.st are .sync.aligned: every lane of the warp issues
    // them together, so every branch around them and every loop exit below is
    // warp-uniform (padding rows compute and store zeros instead of skipping).
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    const int r = 32 * quarter + lane;
    const int rg = mt * kRows + r;
    const bool valid = rg < M;
    const int node = valid ? rg / G : 0;
    const uint64_t mask = valid ? a.mask_bits[size_t(req) * a.n + node] : 0ull;
    const uint32_t tl = tmem + (uint32_t(32 * quarter) << 16);
    const float sl2 = a.scale * 1.4426950408889634f;
    float m_ref = -INFINITY, lsum = 0.f;
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      const int s = t & 1;
      const bool w_ok = mbar_wait(bar(kSFull0 + s), (t >> 1) & 1) && mbar_wait(bar(kFull0 + s), (t >> 1) & 1) &&
                        !*abort_flag;
      if (!__all_sync(FULL, w_ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float x[kKeys];
#pragma unroll
      for (int q = 0; q < kKeys / 32; ++q) {
        float v[32];
        tmem_ld32(tl + col_s(s) + 32 * q, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) x[32 * q + i] = v[i];
      }
      const uint32_t* f = flags + 4 * s;
      const bool all_pre = f[2] != 0;
      const int kbase = k0 + t * kKeys;
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < kKeys; ++c) {
        float v = x[c] * sl2;
        if (!all_pre) {
          const int kg = kbase + c;
          const bool vis = key_valid(f, c) && (kg < Lp || ((mask >> (kg - Lp)) & 1ull));
          v = vis ? v : -INFINITY;
        }
        x[c] = v;
        mx = fmaxf(mx, v);
      }
      // lazy rescaling: move the reference max only when it grows by > 2^8
      const bool need = valid && mx > m_ref + kRescaleLog2;
      const float factor = need ? exp2f(m_ref - mx) : 1.f;  // 0 when nothing was seen yet
      if (t > 0 && __any_sync(FULL, need)) {
        const bool o_ok = mbar_wait(bar(kODone), (t - 1) & 1);  // O holds P V of tile t-1
        if (!__all_sync(FULL, o_ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
          float v[32];
          tmem_ld32(tl + kColO + 32 * q, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= factor;
          tmem_st32f(tl + kColO + 32 * q, v);
        }
      }
      if (need) {
        lsum *= factor;
        m_ref = mx;
      }
      const bool live = valid && m_ref != -INFINITY;
      float part = 0.f;
#pragma unroll
      for (int q = 0; q < kKeys / 32; ++q) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = live ? exp2f(x[32 * q + 2 * i] - m_ref) : 0.f;
          const float p1 = live ? exp2f(x[32 * q + 2 * i + 1] - m_ref) : 0.f;
          part += p0 + p1;
          pk[i] = pack_bf16(p0, p1);
        }
        tmem_st16(tl + col_s(s) + 16 * q, pk);
      }
      lsum += part;
      tc_fence_before();
      mbar_arrive(bar(kPReady0 + s));
    }
    if (!ok && !*abort_flag) fail();
    // epilogue: wait for the last P V, then write this row's output or partial
    const bool e_ok = ok && mbar_wait(bar(kODone), (T - 1) & 1);
    if (__all_sync(FULL, e_ok)) {
      tc_fence_after();
      const int head = g * G + rg % G;
      const size_t orow = (size_t(req) * a.n + node) * a.Hq + head;
      const size_t idx = orow * a.splits + split;
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
#pragma unroll
      for (int q = 0; q < D / 32; ++q) {
        float v[32];
        tmem_ld32(tl + kColO + 32 * q, v);
        if (valid) {
          if (direct) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + orow * D) + 4 * q;
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(pack_bf16(v[8 * i] * inv, v[8 * i + 1] * inv),
                                  pack_bf16(v[8 * i + 2] * inv, v[8 * i + 3] * inv),
                                  pack_bf16(v[8 * i + 4] * inv, v[8 * i + 5] * inv),
                                  pack_bf16(v[8 * i + 6] * inv, v[8 * i + 7] * inv));
          } else {
            float4* dst = reinterpret_cast<float4*>(po + idx * D);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[8 * q + i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          }
        }
      }
      if (valid) {
        if (direct) {
          if (a.lse) a.lse[orow] = lsum > 0.f ? (m_ref + log2f(lsum)) * 0.6931471805599453f : -INFINITY;
        } else {
          pml[idx * 2] = m_ref;
          pml[idx * 2 + 1] = lsum;
        }
      }
    } else if (!*abort_flag) {
      fail();
    }
  }

  // ---- teardown: every role is done with TMEM ----
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// ------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2D bf16 view [rows, D] (row pitch D*2 bytes), boxes of 64 columns x 1 row,
// 128B swizzle: the tile::gather4 operand.
bool encode_rows(CUtensorMap* m, const void* base, long long rows, int D) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cuuint64_t(D), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(D) * 2};
  cuuint32_t box[2] = {64, 1};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
int launch_t(const AttentionParams& p, const TcGeometry& geo, cudaStream_t stream) {
  alignas(64) CUtensorMap tq, tk, tv;
  if (!encode_rows(&tq, p.q, (long long)p.b * p.n * p.Hq, D) ||
      !encode_rows(&tk, p.k_pool, p.num_slots * p.Hkv, D) || !encode_rows(&tv, p.v_pool, p.num_slots * p.Hkv, D))
    return SPEC_ERR_LAUNCH;
  const int smem = Smem<D>::kBytes + 1024;
  static bool attr_set = false;  // per template instance
  if (!attr_set) {
    if (cudaFuncSetAttribute(attention_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return SPEC_ERR_LAUNCH;
    attr_set = true;
  }
  TcArgs args{p, geo.m_tiles, geo.split_tiles};
  dim3 grid(p.Hkv * geo.m_tiles, p.b, p.splits);
  attention_tc_kernel<D><<<grid, kTcThreads, smem, stream>>>(args, tq, tk, tv);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_LAUNCH;
  return p.splits == 1 ? SPEC_OK : launch_attention_merge(p, stream);
}

}  // namespace

TcGeometry attention_tc_geometry(int b, int n, int Hq, int Hkv, int max_seq_len) {
  TcGeometry geo{};
  const int G = Hq / Hkv;
  geo.m_tiles = (n * G + kRows - 1) / kRows;
  const long units = long(b) * Hkv * geo.m_tiles;
  const long tiles = (long(max_seq_len) + n + kKeys - 1) / kKeys;
  // aim at two waves of two CTAs per SM, splits of at least 8 tiles, and at
  // most 16 splits (each split adds a partial per row to write and merge)
  long splits = (2L * 2 * 152 + units - 1) / units;
  if (splits > tiles / 8) splits = tiles / 8;
  if (splits > 16) splits = 16;
  if (splits < 1) splits = 1;
  geo.split_tiles = int((tiles + splits - 1) / splits);
  geo.splits = int((tiles + geo.split_tiles - 1) / geo.split_tiles);
  return geo;
}

int launch_attention_tc(const AttentionParams& p, const TcGeometry& geo, cudaStream_t stream) {
  if (p.D == 128) return launch_t<128>(p, geo, stream);
  if (p.D == 64) return launch_t<64>(p, geo, stream);
  return SPEC_ERR_UNSUPPORTED;
}

}  // namespace spec
