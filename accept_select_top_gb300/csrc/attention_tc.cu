// attention_tc.cu -- tree-masked verify attention on the tcgen05 tensor cores.
//
// [EAGLE2 sections 4.2-4.3: the verify queries are the flattened tree nodes,
// the keys are the cached history (all visible) plus the tree nodes, of which a
// query sees only its ancestors and itself; history KV is read once and shared
// by all candidates], [SGL-XI QLEN_ONLY mask: prefix columns implicitly visible].
//
// Persistent kernel, one CTA per SM.  A work item is 128 query rows of one
// (request, kv head) -- row r is (node r / G, q head g*G + r % G), G = Hq/Hkv --
// and one split of that request's key list (prefix positions, then the n tree
// nodes).  Items are taken from a global counter; every role walks the same
// flat stream of 64-key tiles:
//   warp 0      producer: takes items, publishes them in a two-slot ring,
//               gathers each item's Q rows (cp.async.bulk.tensor tile::gather4)
//               and, per tile, looks the keys' slots up (req_to_token /
//               verify_loc, one tile ahead) and copies their K and V rows into
//               a four-stage ring with 16-byte cp.async, 128B-swizzled by hand
//               (the same layout a swizzled TMA box would give; per-lane copies
//               keep far more scattered rows in flight than gather4 does);
//   warp 1      MMA issuer (one thread): S = Q K^T (M=128, N=64, K=D) into one
//               of two TMEM S buffers; O += P V (M=128, N=D, K=64) with both
//               operands in shared memory, into the item's O buffer (two);
//   warps 2..5  one query row per thread: masked online softmax of the S row
//               (tcgen05.ld), P as bf16 into one of two shared-memory P
//               buffers (128B-swizzled, K-major), lazy rescaling of O in TMEM,
//               and the item's epilogue (bf16 output directly when the key
//               list is not split, else partials that attention_merge_kernel
//               combines).
// P goes through shared memory rather than TMEM because an MMA that reads its
// A operand from TMEM measured about three times slower on this part than the
// same MMA reading shared memory.
// TMEM columns: O0 [0,128), O1 [128,256), S0 [256,320), S1 [320,384).  Every
// mbarrier wait is bounded: on timeout the CTA sets SPEC_DEV_TIMEOUT, stops,
// drains and frees its TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace spec {

namespace {

constexpr int kRows = 128;
constexpr int kKeys = 64;
constexpr int kStages = 4;
constexpr int kTcThreads = 320;  // warps: 0 lead copy, 1 MMA, 2-5 softmax, 6 7 9 copy, 8 idle
constexpr uint32_t kTmemCols = 512;
// O buffer i at TMEM columns [128 i, 128 i + 128); S buffer b at [256 + 64 b, 320 + 64 b)
__host__ __device__ constexpr uint32_t col_o(int i) { return 128u * uint32_t(i); }
__host__ __device__ constexpr uint32_t col_s(int b) { return 256u + 64u * uint32_t(b); }
constexpr float kRescaleLog2 = 8.f;             // O is rescaled only when the row max grows by more than 2^8
constexpr long long kWaitCycles = 4000000000ll;  // ~2 s at 2 GHz: bound of every mbarrier wait

template <int D>
struct Smem {
  static constexpr int kHalves = D / 64;
  static constexpr int kQBlock = kRows * 128;      // [128 rows x 64 bf16], 128B-swizzled: 16 KB
  static constexpr int kQTile = kHalves * kQBlock;
  static constexpr int kKBlock = kKeys * 128;      // [64 keys x 64 bf16]: 8 KB
  static constexpr int kKTile = kHalves * kKBlock; // a K or V tile
  static constexpr int kQ = 0;                     // two Q buffers
  static constexpr int kStage = 2 * kQTile;        // stage s: K at kStage + 2*s*kKTile, V at + kKTile
  static constexpr int kPBuf = kRows * kKeys * 2;  // P: [128 rows x 64 keys] bf16, 128B-swizzled: 16 KB
  static constexpr int kP = kStage + kStages * 2 * kKTile;      // two P buffers
  static constexpr int kFlags = kP + 2 * kPBuf;                 // per stage: 4 words of key flags
  static constexpr int kItems = kFlags + kStages * 32;          // two published item ids
  static constexpr int kBars = kItems + 64;
  static constexpr int kBytes = kBars + 512;
};

static_assert(Smem<128>::kBytes + 1024 <= 227 * 1024, "shared memory of one CTA");

// barriers (uint64 each), by index
enum {
  kFull0 = 0,                  // + stage: K/V landed (the producer's 32 cp.async arrivals + its flags arrival)
  kEmpty0 = kFull0 + kStages,  // + stage: PV of the tile done (stage free)
  kItemFull0 = kEmpty0 + kStages,
  kItemEmpty0 = kItemFull0 + 2,
  kQFull0 = kItemEmpty0 + 2,
  kQEmpty0 = kQFull0 + 2,
  kSFull0 = kQEmpty0 + 2,
  kPReady0 = kSFull0 + 2,
  kOFree0 = kPReady0 + 2,
  kODone0 = kOFree0 + 2,  // + (PV index & 1): two barriers, so no wait is ever two phases behind
  kDrain = kODone0 + 2,
  kNumBars
};

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
// One try_wait: the thread may sleep in hardware until the phase completes or
// kSuspendNs pass, so waiting warps take no issue slots from their neighbours.
constexpr uint32_t kSuspendNs = 20000;
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase of the given parity: false once kWaitCycles SM
// cycles have passed.
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

// 16-byte global -> shared copy; src_bytes 0 writes zeros and reads nothing.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
// One arrival on `bar` once every earlier cp.async of this thread has landed.
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
// Orders generic-proxy shared-memory writes (cp.async) that this thread has
// observed before its later async-proxy reads (tcgen05.mma operands).
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

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


// two floats to bf16 (round to nearest even), lower key in the low half
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}


struct TcArgs {
  AttentionParams p;
  int m_tiles;
  int split_tiles;
  int num_items;
  uint32_t* work_counter;  // next item to take (zero between launches)
  uint32_t* exit_counter;  // CTAs done (zero between launches)
};

// Geometry of a work item, computed alike by every role from the item id.
// id = ((split * b + req) * Hkv + g) * m_tiles + mt: the row tiles of one
// (request, kv head, split) are consecutive, so they run together and share
// their K/V reads through L2.
struct Item {
  int req, g, mt, split, Lp, rq, k0, k1, T;
};

__device__ __forceinline__ Item item_of(const TcArgs& args, int id, bool report) {
  const AttentionParams& a = args.p;
  Item it;
  it.mt = id % args.m_tiles;
  int rest = id / args.m_tiles;
  it.g = rest % a.Hkv;
  rest /= a.Hkv;
  it.req = rest % a.b;
  it.split = rest / a.b;
  const bool first = report && it.g == 0 && it.mt == 0 && it.split == 0;
  int Lp = a.seq_lens[it.req];
  it.rq = a.req_pool_idx[it.req];
  const bool req_ok = it.rq >= 0 && it.rq < a.req_rows;
  if (Lp < 0 || Lp > a.max_seq_len || Lp > a.row_w) {
    if (first) raise_error(a.error, SPEC_DEV_LENGTH);
    Lp = max(0, min(Lp, min(a.max_seq_len, a.row_w)));
  }
  if (!req_ok && first) raise_error(a.error, SPEC_DEV_INDEX);
  it.Lp = Lp;
  const int total = req_ok ? Lp + a.n : 0;
  it.k0 = it.split * args.split_tiles * kKeys;
  it.k1 = min(total, it.k0 + args.split_tiles * kKeys);
  it.T = it.k0 < it.k1 ? (it.k1 - it.k0 + kKeys - 1) / kKeys : 0;
  return it;
}

// Per-stage key flags (8 words in shared memory), written by copy warp p:
//   [p]     bit j: key 16p+j of the tile has a valid slot
//   [4+p]   1 when each of keys 16p..16p+15 is a valid prefix key

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    attention_tc_kernel(const __grid_constant__ TcArgs args, const __grid_constant__ CUtensorMap tm_q) {
  using L = Smem<D>;
  const AttentionParams& a = args.p;
  const int G = a.Hq / a.Hkv, M = a.n * G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned FULL = 0xffffffffu;
  const bool direct = a.splits == 1;  // one split: the normalised output is written here
  float* po = reinterpret_cast<float*>(a.partials);
  float* pml = po + size_t(a.b) * a.n * a.Hq * a.splits * D;
  const unsigned char* kbytes = static_cast<const unsigned char*>(a.k_pool);
  const unsigned char* vbytes = static_cast<const unsigned char*>(a.v_pool);

  // ---- shared memory (1024-aligned for the 128B swizzle atoms) ----
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  unsigned char* sp = smem_raw + (sbase - raw);
  uint32_t* flags = reinterpret_cast<uint32_t*>(sp + L::kFlags);  // [stage][4]
  volatile int* items = reinterpret_cast<volatile int*>(sp + L::kItems);
  const uint32_t bars = sbase + L::kBars;
  auto bar = [&](int i) { return bars + 8u * uint32_t(i); };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sp + L::kBars + 8 * kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sp + L::kBars + 8 * kNumBars + 8);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(kFull0 + i), 4 * 32 + 4);  // four copy warps: cp.async arrivals + flag arrivals
      mbar_init(bar(kEmpty0 + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kItemFull0 + i), 1);
      mbar_init(bar(kItemEmpty0 + i), 1 + kRows + 3);  // the MMA thread, the softmax rows, three copy warps
      mbar_init(bar(kQFull0 + i), 1);
      mbar_init(bar(kQEmpty0 + i), 1);
      mbar_init(bar(kSFull0 + i), 1);
      mbar_init(bar(kPReady0 + i), kRows);
      mbar_init(bar(kOFree0 + i), kRows);
      mbar_init(bar(kODone0 + i), 1);
    }
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

  if (warp == 0 || warp == 6 || warp == 7 || warp == 9) {
    // ============================ producers ============================
    // Four copy warps, one per SM sub-partition (warp & 3), so the copy
    // instructions do not all land next to one softmax warp.  Copy warp
    // `part` looks up and copies keys 16*part .. 16*part+15 of every tile;
    // warp 0 (the lead) also takes the items from the work counter,
    // publishes them and gathers each item's Q rows.
    const int part = warp & 3;
    const bool lead = warp == 0;
    // Key 16*part + lane (lanes 0..15) of tile t: slot load issued one tile
    // ahead (issue), value consumed after that tile's copies (finish).
    auto issue = [&](const Item& it, int t, int& slot, int& kind) {  // kind: 0 none, 1 prefix, 2 tree
      const int kg = it.k0 + t * kKeys + 16 * part + lane;
      slot = -1;
      kind = 0;
      if (lane < 16 && kg < it.k1) {
        if (kg < it.Lp) {
          slot = a.req_to_token[size_t(it.rq) * a.row_w + kg];
          kind = 1;
        } else {
          slot = a.verify_loc[size_t(it.req) * a.n + (kg - it.Lp)];
          kind = 2;
        }
      }
    };
    auto finish = [&](const Item& it, int slot, int kind, int& row, bool& pre) {
      const bool ok_slot = slot >= 0 && slot < a.num_slots;
      if (kind != 0 && !ok_slot) raise_error(a.error, SPEC_DEV_INDEX);
      const bool v = kind != 0 && ok_slot;
      row = v ? int(slot * a.Hkv + it.g) : -1;  // -1: zero-filled, masked out
      pre = lane >= 16 || (v && kind == 1);
    };
    int ct = 0, ci = 0;
    bool ok = true;
    while (ok) {
      Item it{};
      if (lead) {
        int id = 0;
        if (lane == 0) id = int(atomicAdd(args.work_counter, 1u));
        id = __shfl_sync(FULL, id, 0);
        const bool last = id >= args.num_items;
        if (!last) {
          it = item_of(args, id, lane == 0);
          if (it.T == 0) {  // nothing in this split (or a rejected request): not published
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int rg = it.mt * kRows + 4 * lane + e;
              if (rg < M) {
                const size_t orow = (size_t(it.req) * a.n + rg / G) * a.Hq + it.g * G + rg % G;
                if (direct) {  // zero output, empty lse
                  uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + orow * D);
                  for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
                  if (a.lse) a.lse[orow] = -INFINITY;
                } else {  // an empty partial, skipped by the merge
                  const size_t idx = orow * a.splits + it.split;
                  pml[idx * 2] = -INFINITY;
                  pml[idx * 2 + 1] = 0.f;
                }
              }
            }
            continue;
          }
        }
        // publish the item (or the end marker) in slot ci % 2
        const bool slot_ok =
            (ci < 2 || mbar_wait(bar(kItemEmpty0 + (ci & 1)), ((ci >> 1) - 1) & 1)) && !*abort_flag;
        if (!__all_sync(FULL, slot_ok)) {
          if (!*abort_flag) fail();
          break;
        }
        if (lane == 0) {
          items[ci & 1] = last ? -1 : id;
          mbar_arrive(bar(kItemFull0 + (ci & 1)));
        }
        __syncwarp();
        if (last) break;
        // the item's Q rows into Q buffer ci % 2, rows 4*lane .. 4*lane+3
        const bool q_ok = (ci < 2 || mbar_wait(bar(kQEmpty0 + (ci & 1)), ((ci >> 1) - 1) & 1)) && !*abort_flag;
        if (!__all_sync(FULL, q_ok)) {
          if (!*abort_flag) fail();
          break;
        }
        int y[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int rg = it.mt * kRows + 4 * lane + e;
          y[e] = rg < M ? (it.req * a.n + rg / G) * a.Hq + it.g * G + rg % G : -1;  // -1: zero-filled
        }
        if (lane == 0) mbar_expect_tx(bar(kQFull0 + (ci & 1)), L::kQTile);
        __syncwarp();
#pragma unroll
        for (int h = 0; h < L::kHalves; ++h)
          tma_gather4(sbase + L::kQ + (ci & 1) * L::kQTile + h * L::kQBlock + 512u * lane, &tm_q, 64 * h, y[0], y[1],
                      y[2], y[3], bar(kQFull0 + (ci & 1)));
      } else {
        const bool i_ok = mbar_wait(bar(kItemFull0 + (ci & 1)), (ci >> 1) & 1) && !*abort_flag;
        if (!__all_sync(FULL, i_ok)) {
          if (!*abort_flag) fail();
          break;
        }
        const int id = items[ci & 1];
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kItemEmpty0 + (ci & 1)));
        if (id < 0) break;
        it = item_of(args, id, false);
      }
      int row = -1, slot_n = -1, kind_n = 0;
      bool pre = true;
      issue(it, 0, slot_n, kind_n);
      finish(it, slot_n, kind_n, row, pre);
      for (int t = 0; t < it.T; ++t, ++ct) {
        const int s = ct % kStages;
        if (t + 1 < it.T) issue(it, t + 1, slot_n, kind_n);  // in flight while this warp waits
        const bool e_ok = (ct < kStages || mbar_wait(bar(kEmpty0 + s), ((ct / kStages) - 1) & 1)) && !*abort_flag;
        if (!__all_sync(FULL, e_ok)) {
          if (!*abort_flag) fail();
          ok = false;
          break;
        }
        const unsigned vbits = __ballot_sync(FULL, row >= 0);  // lanes 16..31 hold no key
        const bool all_pre = __all_sync(FULL, pre);
        if (lane == 0) {
          flags[8 * s + part] = vbits;
          flags[8 * s + 4 + part] = all_pre ? 1u : 0u;
          mbar_arrive(bar(kFull0 + s));
        }
        // lane: 16-byte chunk c of key row r; one instruction covers kRowsPerOp
        // whole rows (coalesced).  Shared address: half c/8 of the row,
        // 128-byte line r, chunk (c%8) ^ (r%8) (128B swizzle).
        constexpr int kChunks = D / 8;
        constexpr int kRowsPerOp = 32 / kChunks;
        const int c = lane % kChunks, rsub = lane / kChunks;
        const uint32_t kdst = sbase + L::kStage + 2u * s * L::kKTile + uint32_t(c >> 3) * L::kKBlock;
#pragma unroll
        for (int i = 0; i < 16 / kRowsPerOp; ++i) {
          const int rl = kRowsPerOp * i + rsub, r = 16 * part + rl;
          const int y = __shfl_sync(FULL, row, rl);  // key r's pool row, held by lane rl
          const uint32_t dst = kdst + uint32_t(r) * 128u + (uint32_t((c & 7) ^ (r & 7)) << 4);
          const size_t off = size_t(y < 0 ? 0 : y) * (D * 2) + size_t(c) * 16;
          const uint32_t nb = y < 0 ? 0u : 16u;
          cp_async16(dst, kbytes + off, nb);
          cp_async16(dst + L::kKTile, vbytes + off, nb);
        }
        cp_async_arrive(bar(kFull0 + s));
        if (t + 1 < it.T) finish(it, slot_n, kind_n, row, pre);
      }
      ++ci;
    }
    // drain: every copy this warp issued has landed before the CTA can exit
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == 1) {
    // ============================ MMA issuer ============================
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(kRows, kKeys, false);
      constexpr uint32_t idesc_pv = idesc_bf16(kRows, D, true);
      // O += P V for global tile u, local tile lt of the item with ordinal ic
      auto issue_pv = [&](int u, int ic, int lt) -> bool {
        const int b = u & 1, s = u % kStages;
        if (lt == 0 && ic >= 2 && !mbar_wait(bar(kOFree0 + (ic & 1)), ((ic >> 1) - 1) & 1)) return false;
        if (!mbar_wait(bar(kPReady0 + b), (u >> 1) & 1) || *abort_flag) return false;
        tc_fence_after();
        const uint32_t vbase = sbase + L::kStage + 2u * s * L::kKTile + L::kKTile;
        const uint32_t pbase = sbase + L::kP + uint32_t(b) * L::kPBuf;
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk) {
          // A: P keys 16kk..16kk+15 (K-major, 32 bytes into each 128-byte row);
          // B: V rows 16kk.. (MN-major: 64-column halves kKBlock apart, 8-key groups 1024 B apart)
          mma_ss(tmem + col_o(ic & 1), sdesc(pbase + kk * 32, 16, 1024),
                 sdesc(vbase + kk * 16 * 128, L::kKBlock, 1024), idesc_pv, (lt > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar(kODone0 + (u & 1)));
        mma_commit(bar(kEmpty0 + s));
        return true;
      };
      int ct = 0, ci = 0, pend_ic = 0, pend_lt = 0;
      bool ok = true;
      while (ok) {
        if (!mbar_wait(bar(kItemFull0 + (ci & 1)), (ci >> 1) & 1) || *abort_flag) {
          ok = false;
          break;
        }
        const int id = items[ci & 1];
        mbar_arrive(bar(kItemEmpty0 + (ci & 1)));
        if (id < 0) break;
        const Item it = item_of(args, id, false);
        if (!mbar_wait(bar(kQFull0 + (ci & 1)), (ci >> 1) & 1)) {
          ok = false;
          break;
        }
        const uint32_t qbase = sbase + L::kQ + (ci & 1) * L::kQTile;
        for (int t = 0; t < it.T; ++t, ++ct) {
          const int s = ct % kStages;
          if (!mbar_wait(bar(kFull0 + s), (ct / kStages) & 1) || *abort_flag) {
            ok = false;
            break;
          }
          fence_proxy_async();  // the stage was written by cp.async
          tc_fence_after();
          const uint32_t kbase = sbase + L::kStage + 2u * s * L::kKTile;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ko = (kk >> 2) * L::kKBlock + (kk & 3) * 32;
            const uint32_t qo = (kk >> 2) * L::kQBlock + (kk & 3) * 32;
            mma_ss(tmem + col_s(ct & 1), sdesc(qbase + qo, 16, 1024), sdesc(kbase + ko, 16, 1024), idesc_qk,
                   kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(kSFull0 + (ct & 1)));
          if (t == it.T - 1) mma_commit(bar(kQEmpty0 + (ci & 1)));  // the item's Q is no longer read
          if (ct > 0 && !issue_pv(ct - 1, pend_ic, pend_lt)) {
            ok = false;
            break;
          }
          pend_ic = ci;
          pend_lt = t;
        }
        ++ci;
      }
      if (ok && ct > 0) ok = issue_pv(ct - 1, pend_ic, pend_lt);
      if (!ok && !*abort_flag) fail();
      // drain: every MMA issued has completed before TMEM is released
      mma_commit(bar(kDrain));
      mbar_wait(bar(kDrain), 0);
    }
    __syncwarp();
  } else if (warp >= 2 && warp <= 5) {
    // ============================ softmax rows ============================
    // tcgen05.ld / tcgen05.st are .sync.aligned: every lane of the warp issues
    // them together, so every branch around them and every loop exit below is
    // warp-uniform (padding rows compute and store zeros instead of skipping).
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    const int r = 32 * quarter + lane;
    const uint32_t tl = tmem + (uint32_t(32 * quarter) << 16);
    const float sl2 = a.scale * 1.4426950408889634f;
    int ct = 0, ci = 0;
    bool ok = true;
    while (ok) {
      const bool i_ok = mbar_wait(bar(kItemFull0 + (ci & 1)), (ci >> 1) & 1) && !*abort_flag;
      if (!__all_sync(FULL, i_ok)) {
        ok = false;
        break;
      }
      const int id = items[ci & 1];
      mbar_arrive(bar(kItemEmpty0 + (ci & 1)));
      if (id < 0) break;
      const Item it = item_of(args, id, false);
      const int rg = it.mt * kRows + r;
      const bool valid = rg < M;
      const int node = valid ? rg / G : 0;
      const uint64_t mask = valid ? a.mask_bits[size_t(it.req) * a.n + node] : 0ull;
      const uint32_t ocol = col_o(ci & 1);
      float m_ref = -INFINITY, lsum = 0.f;
      for (int t = 0; t < it.T; ++t, ++ct) {
        const int s = ct % kStages, b = ct & 1;
        const bool w_ok = mbar_wait(bar(kSFull0 + b), (ct >> 1) & 1) &&
                          mbar_wait(bar(kFull0 + s), (ct / kStages) & 1) && !*abort_flag;
        if (!__all_sync(FULL, w_ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float x[kKeys];
#pragma unroll
        for (int q = 0; q < kKeys / 32; ++q) {
          float v[32];
          tmem_ld32(tl + col_s(b) + 32 * q, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) x[32 * q + i] = v[i];
        }
        const uint32_t* f = flags + 8 * s;
        const bool all_pre = (f[4] & f[5] & f[6] & f[7]) != 0u;
        const int kbase = it.k0 + t * kKeys;
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (all_pre) {  // history keys only: all visible
#pragma unroll
          for (int c = 0; c < kKeys; ++c) {
            x[c] *= sl2;
            mx4[c & 3] = fmaxf(mx4[c & 3], x[c]);
          }
        } else {
          // visibility of the tile's keys for this row: a valid slot, and a
          // history key or a tree node on the row's ancestor mask; key c is
          // tree node c - c0
          const int c0 = it.Lp - kbase;
          const uint64_t hist = c0 <= 0 ? 0ull : (c0 >= kKeys ? ~0ull : ((1ull << c0) - 1ull));
          const uint64_t tree = c0 >= kKeys ? 0ull : (c0 >= 0 ? (mask << c0) : (mask >> (-c0)));
          const uint64_t valid = uint64_t(f[0] | (f[1] << 16)) | (uint64_t(f[2] | (f[3] << 16)) << 32);
          const uint64_t vis = valid & (hist | tree);
          const uint32_t vlo = uint32_t(vis), vhi = uint32_t(vis >> 32);
#pragma unroll
          for (int c = 0; c < kKeys; ++c) {
            const bool on = (((c < 32 ? vlo : vhi) >> (c & 31)) & 1u) != 0u;
            x[c] = on ? x[c] * sl2 : -INFINITY;
            mx4[c & 3] = fmaxf(mx4[c & 3], x[c]);
          }
        }
        const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
        // lazy rescaling: move the reference max only when it grows by > 2^8
        const bool need = valid && mx > m_ref + kRescaleLog2;
        const float factor = need ? fast_exp2(m_ref - mx) : 1.f;  // 0 when nothing was seen yet
        if (t > 0 && __any_sync(FULL, need)) {
          // O holds P V up to tile ct-1; PV(ct-2) is known complete
          const bool o_ok = mbar_wait(bar(kODone0 + ((ct - 1) & 1)), ((ct - 1) >> 1) & 1);
          if (!__all_sync(FULL, o_ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int q = 0; q < D / 32; ++q) {
            float v[32];
            tmem_ld32(tl + ocol + 32 * q, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= factor;
            tmem_st32f(tl + ocol + 32 * q, v);
          }
        }
        if (need) {
          lsum *= factor;
          m_ref = mx;
        }
        const bool live = valid && m_ref != -INFINITY;
        // P row r of buffer b: one 128-byte line, 16-byte chunk j (keys 8j..8j+7)
        // at position j ^ (r % 8)
        unsigned char* prow = sp + L::kP + b * L::kPBuf + r * 128;
        float part4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < kKeys / 8; ++j) {
          uint32_t pk[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float p0 = live ? fast_exp2(x[8 * j + 2 * i] - m_ref) : 0.f;
            const float p1 = live ? fast_exp2(x[8 * j + 2 * i + 1] - m_ref) : 0.f;
            part4[i] += p0 + p1;
            pk[i] = pack_bf16(p0, p1);
          }
          *reinterpret_cast<uint4*>(prow + ((j ^ (r & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        lsum += (part4[0] + part4[1]) + (part4[2] + part4[3]);
        fence_proxy_async();  // P is read by the MMA (async proxy)
        tc_fence_before();
        mbar_arrive(bar(kPReady0 + b));
      }
      if (!ok) break;
      // epilogue: wait for the PV of the item's last tile ct-1 (its commit
      // covers every earlier PV; PV(ct-3) is known complete from S(ct-1))
      const bool e_ok = mbar_wait(bar(kODone0 + ((ct - 1) & 1)), ((ct - 1) >> 1) & 1);
      if (!__all_sync(FULL, e_ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int head = it.g * G + rg % G;
      const size_t orow = (size_t(it.req) * a.n + node) * a.Hq + head;
      const size_t idx = orow * a.splits + it.split;
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
#pragma unroll
      for (int q = 0; q < D / 32; ++q) {
        float v[32];
        tmem_ld32(tl + ocol + 32 * q, v);
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
      tc_fence_before();
      mbar_arrive(bar(kOFree0 + (ci & 1)));  // this O buffer may take the item after next
      ++ci;
    }
    if (!ok && !*abort_flag) fail();
  }

  // ---- teardown: every role is done with TMEM ----
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
  // the CTA that finishes last puts the work counters back to zero
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(args.exit_counter, 1u) == gridDim.x - 1) {
      atomicExch(args.work_counter, 0u);
      atomicExch(args.exit_counter, 0u);
    }
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
  alignas(64) CUtensorMap tq;
  if (!encode_rows(&tq, p.q, (long long)p.b * p.n * p.Hq, D)) return SPEC_ERR_LAUNCH;
  // at least 120 KB, so that two CTAs never share an SM (each holds all 512
  // TMEM columns)
  const int smem = Smem<D>::kBytes + 1024 > 120 * 1024 ? Smem<D>::kBytes + 1024 : 120 * 1024;
  static int sm_count = 0;  // per template instance; one device per process
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(attention_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return SPEC_ERR_LAUNCH;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sm_count < 1)
      return SPEC_ERR_LAUNCH;
    attr_set = true;
  }
  const long items = long(p.splits) * p.b * p.Hkv * geo.m_tiles;
  if (items > 0x7fffffffL) return SPEC_ERR_UNSUPPORTED;
  TcArgs args{p, geo.m_tiles, geo.split_tiles, int(items), p.counters, p.counters + 1};
  const int grid = int(items < sm_count ? items : sm_count);
  attention_tc_kernel<D><<<grid, kTcThreads, smem, stream>>>(args, tq);
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
  // about four items per SM for the dynamic schedule to balance, splits of at
  // least 8 tiles (each split adds a partial per row to write and merge), at
  // most 32 splits
  long splits = (kTargetCtas + units - 1) / units;
  if (splits > tiles / 8) splits = tiles / 8;
  if (splits > 32) splits = 32;
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
