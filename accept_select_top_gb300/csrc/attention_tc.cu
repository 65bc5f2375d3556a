// attention_tc.cu -- tree-masked verify attention on the tcgen05 tensor cores.
//
// [EAGLE2 sections 4.2-4.3: the verify queries are the flattened tree nodes,
// the keys are the cached history (all visible) plus the tree nodes, of which a
// query sees only its ancestors and itself; history KV is read once and shared
// by all candidates], [SGL-XI QLEN_ONLY mask: prefix columns implicitly visible].
//
// Persistent kernel, one CTA per SM, with a stream-K partition: the units
// (request, kv head, 128 query rows -- row r is (node r / G, q head g*G + r %
// G), G = Hq/Hkv) are laid end to end in tile space (64 keys a tile: prefix
// positions, then the n tree nodes) and each CTA takes an equal contiguous
// range of tiles, cut into one piece per unit it touches.  A unit inside one
// range is written directly; a unit split over CTAs leaves one partial per
// piece and the piece arriving last merges them (no second launch).  Every
// role walks the same pieces and the same flat stream of tiles:
//   warps 0,6,7,9  copy warps, one per SM sub-partition: each looks up the
//               slots of 16 keys of every tile (req_to_token / verify_loc,
//               one tile ahead) and copies their K and V rows into a
//               four-stage ring with 16-byte cp.async, 128B-swizzled by hand
//               (the layout a swizzled TMA box would give; per-lane copies
//               keep far more scattered rows in flight than gather4 does);
//   warp 1      MMA issuer (one thread): S = Q K^T (M=128, N=64, K=D) into one
//               of two TMEM S buffers; O += P V (M=128, N=D, K=64) with both
//               operands in shared memory, into the piece's O buffer (two);
//   warps 2..5  one query row per thread: masked online softmax of the S row
//               (tcgen05.ld), P as bf16 into one of two shared-memory P
//               buffers (128B-swizzled, K-major), lazy rescaling of O in TMEM,
//               and the piece's epilogue;
//   warp 8      Q rows: copies each piece's real query rows into one of two
//               Q buffers as soon as it frees (issuing a piece's Q took the
//               copy warp ~4000 cycles under load, which drained the K/V
//               ring at every piece boundary); and counts the CTA's split
//               pieces in on their units (fence + atomic), which kept the
//               softmax rows waiting when they did it themselves.
// P goes through shared memory rather than TMEM because an MMA that reads its
// A operand from TMEM measured about three times slower on this part than the
// same MMA reading shared memory.
// TMEM columns: O0 [0,128), O1 [128,256), S0 [256,320), S1 [320,384).  Every
// mbarrier wait is bounded: on timeout the CTA sets SPEC_DEV_TIMEOUT, stops,
// drains and frees its TMEM.
#include "common.cuh"
#include "kernels.cuh"

namespace spec {

namespace {

constexpr int kRows = 128;
constexpr int kKeys = 64;
constexpr int kStages = 4;
constexpr int kTcThreads = 320;  // warps: 0 6 7 9 copy, 1 MMA, 2-5 softmax, 8 Q rows
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
  static constexpr int kFlags = kP + 2 * kPBuf;                 // per stage: 8 words of key flags
  static constexpr int kScratch = kFlags + kStages * 32;        // partition and merge scratch
  static constexpr int kBars = kScratch + 512;
  static constexpr int kBytes = kBars + 512;
};

static_assert(Smem<128>::kBytes + 1024 <= 227 * 1024, "shared memory of one CTA");

// barriers (uint64 each), by index
enum {
  kFull0 = 0,                  // + stage: K/V landed (the producer's 32 cp.async arrivals + its flags arrival)
  kEmpty0 = kFull0 + kStages,  // + stage: PV of the tile done (stage free)
  kQFull0 = kEmpty0 + kStages,
  kQEmpty0 = kQFull0 + 2,
  kSFull0 = kQEmpty0 + 2,
  kPReady0 = kSFull0 + 2,
  kOFree0 = kPReady0 + 2,
  kODone0 = kOFree0 + 2,  // + (PV index & 1): two barriers, so no wait is ever two phases behind
  kPub0 = kODone0 + 2,  // + k: the 128 softmax rows stored the CTA's k-th split piece (k < 2; one phase each)
  kDrain = kPub0 + 2,
  kQIssued,  // the first piece's Q copies are issued (the K/V copies queue behind them)
  kNumBars
};

// ------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
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
// the same bound, for a warp off the critical path that may wait a whole
// piece: it sleeps between polls so that it takes no issue slots from the
// copy and softmax warps of its sub-partition
__device__ __forceinline__ bool mbar_wait_idle(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long start = clock64();
  while (clock64() - start < kWaitCycles && !*abort_flag) {
    __nanosleep(256);
    if (mbar_try_wait(bar, parity)) return true;
  }
  return false;
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


constexpr int kMaxCtas = 192;  // upper bound of the grid (one CTA per SM); sizes the partial slots
// partial region of the workspace: [slot m, l][slot O (D <= 128)]; the
// arrival counters are the workspace's counter words (zero between calls)
constexpr size_t kSlotMLOffset = 0;
constexpr size_t kSlotOOffset = kSlotMLOffset + size_t(2) * kMaxCtas * kRows * 2 * 4;

struct TcArgs {
  AttentionParams p;
  int m_tiles;
  uint32_t* counters;   // [kMaxCtas] arrivals per split unit (workspace counter words, zero between launches)
  float* slot_o;        // [2 * kMaxCtas][128 rows][D] unnormalised O of a piece of a split unit
  float* slot_ml;       // [2 * kMaxCtas][128 rows][2]: running max (log2 domain), sum
};

// Keys, history length and pool row of request r, validated like the C ABI
// describes: a bad length is clamped, a bad pool row leaves no keys.
struct ReqInfo {
  int Lp, rq, total, tiles;
};
__device__ __forceinline__ ReqInfo req_check(const AttentionParams& a, int Lp, int rq, bool report) {
  ReqInfo q;
  q.rq = rq;
  const bool req_ok = q.rq >= 0 && q.rq < a.req_rows;
  if (Lp < 0 || Lp > a.max_seq_len || Lp > a.row_w) {
    if (report) raise_error(a.error, SPEC_DEV_LENGTH);
    Lp = max(0, min(Lp, min(a.max_seq_len, a.row_w)));
  }
  if (!req_ok && report) raise_error(a.error, SPEC_DEV_INDEX);
  q.Lp = Lp;
  q.total = req_ok ? Lp + a.n : 0;
  q.tiles = max(1, (q.total + kKeys - 1) / kKeys);  // a request without keys still owns one (empty) tile
  return q;
}
__device__ __forceinline__ ReqInfo req_info(const AttentionParams& a, int r, bool report) {
  return req_check(a, a.seq_lens[r], a.req_pool_idx[r], report);
}

// Stream-K partition.  The units (request, kv head, 128-row tile) are laid
// end to end in tile space, row tile outermost, then request, then kv head;
// unit (mt, r, g) has the tiles of request r.  CTA c takes tiles [c*T/G,
// (c+1)*T/G) and cuts them into pieces, one per unit it touches.  With the row
// tile outermost, the units that read the same keys (same request and kv head,
// other row tiles) sit T / m_tiles tiles apart, so CTAs that far apart read
// those keys at about the same time and the second read finds them in L2.
__host__ __device__ __forceinline__ long long cta_start(long long c, long long T, long long G) { return c * T / G; }
// the CTA whose range holds tile x
__host__ __device__ __forceinline__ int cta_of(long long x, long long T, long long G) {
  return int(((x + 1) * G - 1) / T);
}

struct Piece {
  int req, g, mt, t0, T, Tr, Lp, rq, k0, k1, idx;  // idx: ordinal of the piece within its CTA
  long long unit_start;                           // first tile of the unit in tile space
  bool complete;                                  // the piece is the whole unit
};

struct PieceIter {
  int r, j, mt, t0, idx;  // j: the kv head
  long long cur, end;
  int nr, nlen, nrq;  // request nr's raw seq_len and pool row, loaded one piece ahead
  __device__ __forceinline__ bool next(const AttentionParams& a, int m_tiles, Piece& p, bool report) {
    if (cur >= end) return false;
    const ReqInfo q = nr == r ? req_check(a, nlen, nrq, report && j == 0 && t0 == 0)
                              : req_info(a, r, report && j == 0 && t0 == 0);
    const long long left = end - cur;
    const int take = int(left < (long long)(q.tiles - t0) ? left : (long long)(q.tiles - t0));
    p.req = r;
    p.g = j;
    p.mt = mt;
    p.t0 = t0;
    p.T = take;
    p.Tr = q.tiles;
    p.Lp = q.Lp;
    p.rq = q.rq;
    p.k0 = t0 * kKeys;
    p.k1 = min(q.total, (t0 + take) * kKeys);
    p.idx = idx++;
    p.unit_start = cur - t0;
    p.complete = t0 == 0 && take == q.tiles;
    cur += take;
    t0 += take;
    if (t0 == q.tiles) {
      t0 = 0;
      if (++j == a.Hkv) {
        j = 0;
        if (++r == a.b) {
          r = 0;
          ++mt;
        }
      }
    }
    if (r != nr && cur < end) {  // the next piece's request: loads in flight meanwhile
      nr = r;
      nlen = a.seq_lens[r];
      nrq = a.req_pool_idx[r];
    } else if (nr != r) {
      nr = -1;
    }
    if (nr == r && r == p.req) {  // same request: keep the values already checked
      nlen = q.Lp;
      nrq = q.rq;
    }
    return true;
  }
};

// Per-stage key flags (8 words in shared memory), written by copy warp p:
//   [p]     bit j: key 16p+j of the tile has a valid slot
//   [4+p]   1 when each of keys 16p..16p+15 is a valid prefix key

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    attention_tc_kernel(const __grid_constant__ TcArgs args) {
  using L = Smem<D>;
  const AttentionParams& a = args.p;
  const int G = a.Hq / a.Hkv, M = a.n * G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned FULL = 0xffffffffu;
  const unsigned char* qbytes = static_cast<const unsigned char*>(a.q);
  const unsigned char* kbytes = static_cast<const unsigned char*>(a.k_pool);
  const unsigned char* vbytes = static_cast<const unsigned char*>(a.v_pool);

  // ---- shared memory (1024-aligned for the 128B swizzle atoms) ----
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  unsigned char* sp = smem_raw + (sbase - raw);
  uint32_t* flags = reinterpret_cast<uint32_t*>(sp + L::kFlags);  // [stage][8]
  const uint32_t bars = sbase + L::kBars;
  auto bar = [&](int i) { return bars + 8u * uint32_t(i); };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sp + L::kBars + 8 * kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sp + L::kBars + 8 * kNumBars + 8);
  long long* scratch = reinterpret_cast<long long*>(sp + L::kScratch);  // [0..15] block sums, [16..] partition
  // split units this CTA merges at the end: count, then (unit_start, Tr, req, g, mt, c1, c2, -) each
  int* merges = reinterpret_cast<int*>(sp + L::kScratch + 8 * 24);
  constexpr int kMaxMerges = 2;  // a CTA finishes at most its first and its last piece
  // split pieces of this CTA awaiting their arrival: (unit_start, Tr, req, g, mt, -, -, -) each
  int* pend = merges + 1 + 8 * kMaxMerges;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(kFull0 + i), 4 * 32 + 4);  // four copy warps: cp.async arrivals + flag arrivals
      mbar_init(bar(kEmpty0 + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kQFull0 + i), 32);  // the Q warp's cp.async arrivals
      mbar_init(bar(kQEmpty0 + i), 1);
      mbar_init(bar(kSFull0 + i), 1);
      mbar_init(bar(kPReady0 + i), kRows);
      mbar_init(bar(kOFree0 + i), kRows);
      mbar_init(bar(kODone0 + i), 1);
    }
    mbar_init(bar(kPub0), kRows);
    mbar_init(bar(kPub0 + 1), kRows);
    mbar_init(bar(kDrain), 1);
    mbar_init(bar(kQIssued), 1);
    *abort_flag = 0;
    merges[0] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }

  pdl_wait();  // nothing above reads global memory
  pdl_trigger();
  // ---- partition: total tiles T, this CTA's range, and where it starts ----
  const int upr = a.Hkv * args.m_tiles;
  const int nwarps = blockDim.x >> 5;
  {
    long long tot = 0;
    for (int r = threadIdx.x; r < a.b; r += blockDim.x) tot += (long long)req_info(a, r, false).tiles * upr;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(FULL, tot, o);
    if (lane == 0) scratch[warp] = tot;
    __syncthreads();
    if (threadIdx.x == 0) {
      long long T = 0;
      for (int w = 0; w < nwarps; ++w) T += scratch[w];
      scratch[16] = T;
    }
    __syncthreads();
    const long long T = scratch[16];
    const long long TB = T / args.m_tiles;  // the tiles of one row tile over every request and kv head
    // Ge = min(grid, T) CTAs share the tiles, so every one of them has at
    // least one (a unit's pieces are then in consecutive CTAs); the others idle
    const long long Ge = T < gridDim.x ? T : gridDim.x;
    const bool part = blockIdx.x < Ge;
    const long long S = part ? cta_start(blockIdx.x, T, Ge) : 0, E = part ? cta_start(blockIdx.x + 1, T, Ge) : 0;
    // the request holding tile S (at S' = S mod TB inside row tile S / TB):
    // chunks of blockDim requests, a block scan each
    const long long Sr = TB > 0 ? S % TB : 0;
    long long run = 0;
    for (int rb = 0; rb < a.b; rb += blockDim.x) {
      const int r = rb + threadIdx.x;
      const long long v = r < a.b ? (long long)req_info(a, r, false).tiles * a.Hkv : 0;
      long long incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(FULL, incl, o);
        if (lane >= o) incl += y;
      }
      __syncthreads();  // scratch[0..] reused
      if (lane == 31) scratch[warp] = incl;
      __syncthreads();
      long long before = run;
      for (int w = 0; w < warp; ++w) before += scratch[w];
      const long long excl = before + incl - v;
      if (r < a.b && v > 0 && excl <= Sr && Sr < excl + v) {
        const long long o = Sr - excl;  // offset inside request r
        const ReqInfo q = req_info(a, r, false);
        scratch[17] = r;
        scratch[18] = o / q.tiles;  // kv head
        scratch[19] = o % q.tiles;  // tile within the unit
        scratch[23] = TB > 0 ? S / TB : 0;  // row tile
      }
      for (int w = 0; w < nwarps; ++w) run += scratch[w];
    }
    if (threadIdx.x == 0) {
      scratch[20] = S;
      scratch[21] = E;
      scratch[22] = Ge;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const long long T_all = scratch[16], G_eff = scratch[22];
  auto start_iter = [&]() {
    PieceIter it;
    it.cur = scratch[20];
    it.end = scratch[21];
    it.r = it.cur < it.end ? int(scratch[17]) : 0;
    it.j = it.cur < it.end ? int(scratch[18]) : 0;
    it.mt = it.cur < it.end ? int(scratch[23]) : 0;
    it.t0 = it.cur < it.end ? int(scratch[19]) : 0;
    it.idx = 0;
    it.nr = -1;
    it.nlen = 0;
    it.nrq = -1;
    return it;
  };

  auto fail = [&]() {
    raise_error(a.error, SPEC_DEV_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp == 0 || warp == 6 || warp == 7 || warp == 9) {
    // ============================ producers ============================
    // Four copy warps, one per SM sub-partition (warp & 3), so the copy
    // instructions do not all land next to one softmax warp.  Copy warp
    // `part` looks up and copies keys 16*part .. 16*part+15 of every tile.
    const int part = warp & 3;
    const bool lead = warp == 0;  // reports a request's bad length or pool row
    // Key 16*part + lane (lanes 0..15) of tile t: slot load issued one tile
    // ahead (issue), value consumed after that tile's copies (finish).
    auto issue = [&](const Piece& pc, int t, int& slot, int& kind) {  // kind: 0 none, 1 prefix, 2 tree
      const int kg = pc.k0 + t * kKeys + 16 * part + lane;
      slot = -1;
      kind = 0;
      if (lane < 16 && kg < pc.k1) {
        if (kg < pc.Lp) {
          slot = a.req_to_token[size_t(pc.rq) * a.row_w + kg];
          kind = 1;
        } else {
          slot = a.verify_loc[size_t(pc.req) * a.n + (kg - pc.Lp)];
          kind = 2;
        }
      }
    };
    auto finish = [&](const Piece& pc, int slot, int kind, int& row, bool& pre) {
      const bool ok_slot = slot >= 0 && slot < a.num_slots;
      if (kind != 0 && !ok_slot) raise_error(a.error, SPEC_DEV_INDEX);
      const bool v = kind != 0 && ok_slot;
      row = v ? int(slot * a.Hkv + pc.g) : -1;  // -1: zero-filled, masked out
      pre = lane >= 16 || (v && kind == 1);
    };
    PieceIter pit = start_iter();
    Piece pc;
    int ct = 0, ci = 0;
    bool ok = true;
    // Slot lookups run kLook tiles ahead of the copies, like the copies run
    // ahead of the MMA: cur (row, pre) is the looked-up tile about to be
    // copied, ring[j] the lookup in flight for the (j+1)-th tile after it --
    // across a piece boundary, the next piece's first tiles.
    constexpr int kLook = 4;
    int row = -1;
    bool pre = true, cur_ready = false;
    int rs[kLook], rk[kLook];
    bool rv[kLook];
#pragma unroll
    for (int j = 0; j < kLook; ++j) {
      rs[j] = -1;
      rk[j] = 0;
      rv[j] = false;
    }
    while (ok && pit.next(a, args.m_tiles, pc, lead && lane == 0)) {
      int s0 = -1, k0 = 0;
      if (!cur_ready) issue(pc, 0, s0, k0);  // tile 0's lookups, unless the previous piece started them
#pragma unroll
      for (int j = 0; j < kLook; ++j)  // this piece's tiles 1..kLook not yet looked up
        if (!rv[j] && 1 + j < pc.T) {
          issue(pc, 1 + j, rs[j], rk[j]);
          rv[j] = true;
        }
      if (!cur_ready) finish(pc, s0, k0, row, pre);
      cur_ready = false;
      Piece nxt;  // the next piece: its first lookups go out during this piece's last kLook tiles
      bool has_next = false, peeked = false;
      for (int t = 0; t < pc.T; ++t, ++ct) {
        const int s = ct % kStages;
        if (!peeked && t + 1 + kLook >= pc.T) {
          PieceIter peek = pit;
          has_next = peek.next(a, args.m_tiles, nxt, false);
          peeked = true;
#pragma unroll
          for (int j = 0; j < kLook; ++j) {  // ring slots that fall in the next piece
            const int x = t + 1 + j - pc.T;
            if (!rv[j] && x >= 0 && has_next && x < nxt.T) {
              issue(nxt, x, rs[j], rk[j]);
              rv[j] = true;
            }
          }
        }
        // the lookup for the tile kLook+1 ahead
        int ns = -1, nk = 0;
        bool nv = false;
        {
          const int x = t + 1 + kLook;
          if (x < pc.T) {
            issue(pc, x, ns, nk);
            nv = true;
          } else if (has_next && x - pc.T < nxt.T) {
            issue(nxt, x - pc.T, ns, nk);
            nv = true;
          }
        }
        const bool e_ok = (ct < kStages || mbar_wait(bar(kEmpty0 + s), ((ct / kStages) - 1) & 1)) && !*abort_flag;
        if (!__all_sync(FULL, e_ok)) {
          if (!*abort_flag) fail();
          ok = false;
          break;
        }
        if (ct == 0 && !__all_sync(FULL, mbar_wait(bar(kQIssued), 0))) {
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
        // the next tile's lookup (the ring's head) becomes cur
        if (t + 1 < pc.T) {
          if (!rv[0]) issue(pc, t + 1, rs[0], rk[0]);  // (not reached: the ring holds it)
          finish(pc, rs[0], rk[0], row, pre);
        } else if (has_next) {
          if (!rv[0]) issue(nxt, 0, rs[0], rk[0]);
          finish(nxt, rs[0], rk[0], row, pre);
          cur_ready = true;
        }
#pragma unroll
        for (int j = 0; j + 1 < kLook; ++j) {
          rs[j] = rs[j + 1];
          rk[j] = rk[j + 1];
          rv[j] = rv[j + 1];
        }
        rs[kLook - 1] = ns;
        rk[kLook - 1] = nk;
        rv[kLook - 1] = nv;
      }
      ++ci;
    }
    // drain: every copy this warp issued has landed before the CTA can exit
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == 8) {
    // ============================ Q rows ============================
    // Each piece's Q rows go into Q buffer ci % 2 as soon as the MMA is done
    // with the piece two back, so neither the K/V copies nor the MMA wait
    // on them.  Only real query rows are copied (same 16-byte cp.async and
    // swizzle as K).  The rows past them keep whatever they hold: their S
    // rows are never read as output, their P rows are written as zeros (a
    // padding row is never live), so their O rows stay out of every result.
    // The first piece's Q goes out before any K/V copy, so that the first
    // QK does not wait behind four stages of K/V.
    //   The same warp counts this CTA's split pieces (its first and last at
    // most) in on their units: once the softmax rows have stored a piece's
    // partial and arrived (release, CTA scope), lane 0 adds one to the
    // unit's counter with an acquire-release atomic at GPU scope, whose
    // release covers those stores; the piece arriving last records the unit
    // (its acquire covers every other piece's partial, and the teardown
    // barrier passes that on to the whole CTA, which merges it).  A piece is counted in after the Q of the piece two
    // later is out, which is the order the two events come in.
    PieceIter pit = start_iter();
    Piece pc;
    int ci = 0;
    int nsplit = 0, npub = 0;  // split pieces seen / counted in
    int split_ci0 = 0, split_ci1 = 0;  // their piece ordinals
    auto publish = [&]() -> bool {
      const bool w = mbar_wait_idle(bar(kPub0 + npub), 0, abort_flag);
      if (!__all_sync(FULL, w)) return false;
      if (lane == 0) {
        const int* e = pend + 8 * npub;
        const int c1 = cta_of(e[0], T_all, G_eff);
        const int c2 = cta_of((long long)e[0] + e[1] - 1, T_all, G_eff);
        if (atom_add_acq_rel(args.counters + c1) == uint32_t(c2 - c1) && merges[0] < kMaxMerges) {
          int* m = merges + 1 + 8 * merges[0];
          for (int k = 0; k < 5; ++k) m[k] = e[k];
          m[5] = c1;
          m[6] = c2;
          merges[0] += 1;
        }
      }
      ++npub;
      return true;
    };
    bool q_run = true;
    constexpr int kChunks = D / 8;
    constexpr int kRowsPerOp = 32 / kChunks;
    const int c = lane % kChunks, rsub = lane / kChunks;
    while (pit.next(a, args.m_tiles, pc, false)) {
      const int b = ci & 1;
      if (!pc.complete && nsplit < kMaxMerges) {
        if (lane == 0) {
          int* e = pend + 8 * nsplit;
          e[0] = int(pc.unit_start);  // tile space fits in int: < 2^31 tiles
          e[1] = pc.Tr;
          e[2] = pc.req;
          e[3] = pc.g;
          e[4] = pc.mt;
        }
        if (nsplit == 0) split_ci0 = ci;
        else split_ci1 = ci;
        ++nsplit;
      }
      const bool q_ok = (ci < 2 || mbar_wait_idle(bar(kQEmpty0 + b), ((ci >> 1) - 1) & 1, abort_flag)) && !*abort_flag;
      if (!__all_sync(FULL, q_ok)) {
        q_run = false;
        break;
      }
      const int v = min(kRows, M - pc.mt * kRows);  // real query rows of the tile
      const uint32_t qdst = sbase + L::kQ + uint32_t(b) * L::kQTile + uint32_t(c >> 3) * L::kQBlock;
      // row r = query (token tok, head h of the group): one division per
      // piece, then stepped (a runtime divide per row cost ~200 cycles)
      const int rg0 = pc.mt * kRows + rsub;
      int tok = rg0 / G, h = rg0 - (rg0 / G) * G;
      const long long qbase = (long long)pc.req * a.n;
#pragma unroll 4
      for (int r0 = 0; r0 < v; r0 += kRowsPerOp) {
        const int r = r0 + rsub;
        if (r < v) {
          const size_t y = size_t((qbase + tok) * a.Hq + pc.g * G + h);
          const uint32_t dst = qdst + uint32_t(r) * 128u + (uint32_t((c & 7) ^ (r & 7)) << 4);
          cp_async16(dst, qbytes + y * (D * 2) + size_t(c) * 16, 16u);
        }
        h += kRowsPerOp;
        while (h >= G) {  // at most kRowsPerOp steps
          h -= G;
          ++tok;
        }
      }
      cp_async_arrive(bar(kQFull0 + b));
      if (ci == 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kQIssued));
      }
      if (npub < nsplit && (npub == 0 ? split_ci0 : split_ci1) <= ci - 2 && !publish()) {
        q_run = false;
        break;
      }
      ++ci;
    }
    if (ci == 0 && lane == 0) mbar_arrive(bar(kQIssued));  // (no piece, or stopped)
    while (q_run && npub < nsplit)
      if (!publish()) q_run = false;
    if (!q_run && !*abort_flag) fail();
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == 1) {
    // ============================ MMA issuer ============================
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(kRows, kKeys, false);
      constexpr uint32_t idesc_pv = idesc_bf16(kRows, D, true);
      // O += P V for global tile u, local tile lt of the piece with ordinal ic
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
      PieceIter pit = start_iter();
      Piece pc;
      // P V of a tile is issued after the next tile's Q K^T (so the softmax of
      // the next tile overlaps it), except at the end of a piece: there it
      // follows at once, so the piece's epilogue does not wait on the next
      // piece's first loads
      int ct = 0, ci = 0, pend_u = -1, pend_ic = 0, pend_lt = 0;
      bool ok = true;
      while (ok && pit.next(a, args.m_tiles, pc, false)) {
        if (!mbar_wait(bar(kQFull0 + (ci & 1)), (ci >> 1) & 1) || *abort_flag) {
          ok = false;
          break;
        }
        fence_proxy_async();  // Q was written by cp.async
        const uint32_t qbase = sbase + L::kQ + (ci & 1) * L::kQTile;
        for (int t = 0; t < pc.T; ++t, ++ct) {
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
          if (t == pc.T - 1) mma_commit(bar(kQEmpty0 + (ci & 1)));  // the piece's Q is no longer read
          if (pend_u >= 0 && !issue_pv(pend_u, pend_ic, pend_lt)) {
            ok = false;
            break;
          }
          pend_u = ct;
          pend_ic = ci;
          pend_lt = t;
          if (t == pc.T - 1) {
            if (!issue_pv(pend_u, pend_ic, pend_lt)) {
              ok = false;
              break;
            }
            pend_u = -1;
          }
        }
        ++ci;
      }
      if (ok && pend_u >= 0) ok = issue_pv(pend_u, pend_ic, pend_lt);
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
    PieceIter pit = start_iter();
    Piece pc;
    int ct = 0, ci = 0, nsp = 0;  // nsp: split pieces so far
    bool ok = true;
    while (ok && pit.next(a, args.m_tiles, pc, false)) {
      const int rg = pc.mt * kRows + r;
      const bool valid = rg < M;
      const int node = valid ? rg / G : 0;
      const uint64_t mask = valid ? a.mask_bits[size_t(pc.req) * a.n + node] : 0ull;
      const uint32_t ocol = col_o(ci & 1);
      float m_ref = -INFINITY, lsum = 0.f;
      for (int t = 0; t < pc.T; ++t, ++ct) {
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
        const int kbase = pc.k0 + t * kKeys;
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
          const int c0 = pc.Lp - kbase;
          const uint64_t hist = c0 <= 0 ? 0ull : (c0 >= kKeys ? ~0ull : ((1ull << c0) - 1ull));
          const uint64_t tree = c0 >= kKeys ? 0ull : (c0 >= 0 ? (mask << c0) : (mask >> (-c0)));
          const uint64_t vw = uint64_t(f[0] | (f[1] << 16)) | (uint64_t(f[2] | (f[3] << 16)) << 32);
          const uint64_t vis = vw & (hist | tree);
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
      // epilogue: wait for the PV of the piece's last tile ct-1 (its commit
      // covers every earlier PV; PV(ct-3) is known complete from S(ct-1))
      const bool e_ok = mbar_wait(bar(kODone0 + ((ct - 1) & 1)), ((ct - 1) >> 1) & 1);
      if (!__all_sync(FULL, e_ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int head = pc.g * G + rg % G;
      const size_t orow = (size_t(pc.req) * a.n + node) * a.Hq + head;
      const int slot = 2 * int(blockIdx.x) + (pc.idx == 0 ? 0 : 1);
      float* so = args.slot_o + (size_t(slot) * kRows + r) * D;
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
#pragma unroll
      for (int q = 0; q < D / 32; ++q) {
        float v[32];
        tmem_ld32(tl + ocol + 32 * q, v);
        if (valid) {
          if (pc.complete) {  // the whole unit: normalised bf16 output
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + orow * D) + 4 * q;
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(pack_bf16(v[8 * i] * inv, v[8 * i + 1] * inv),
                                  pack_bf16(v[8 * i + 2] * inv, v[8 * i + 3] * inv),
                                  pack_bf16(v[8 * i + 4] * inv, v[8 * i + 5] * inv),
                                  pack_bf16(v[8 * i + 6] * inv, v[8 * i + 7] * inv));
          } else {  // a piece of a split unit: unnormalised partial in this CTA's slot
            float4* dst = reinterpret_cast<float4*>(so) + 8 * q;
#pragma unroll
            for (int i = 0; i < 8; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(bar(kOFree0 + (ci & 1)));  // this O buffer may take the piece after next
      if (pc.complete) {
        if (valid && a.lse) a.lse[orow] = lsum > 0.f ? (m_ref + log2f(lsum)) * 0.6931471805599453f : -INFINITY;
      } else {
        // split unit: this piece's partial (O above, then m and l); the Q
        // warp, once all 128 rows arrive, fences and counts the piece in on
        // its unit, off this path
        if (valid) {
          float* sml = args.slot_ml + (size_t(slot) * kRows + r) * 2;
          sml[0] = m_ref;
          sml[1] = lsum;
        }
        if (nsp < kMaxMerges) mbar_arrive(bar(kPub0 + nsp));  // release (CTA scope): the stores above come first
        ++nsp;
      }
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

  // ---- merge the split units whose last piece this CTA finished: every
  // thread, many independent loads in flight; the K/V ring (idle now) holds
  // the per-row weights ----
  const int nmerge = *abort_flag ? 0 : merges[0];
  // [pieces][128 rows] weights, [128] 1/L, [pieces][128] sums
  float* wsm = reinterpret_cast<float*>(sp + L::kStage);
  // pieces the ring can hold per-row data for: max then weight, sum, and 1/L
  const int wcap = ((2 * kStages * L::kKTile) / (4 * kRows) - 1) / 2;
  for (int mi = 0; mi < nmerge; ++mi) {
    const int* m = merges + 1 + 8 * mi;
    const long long ustart = m[0];
    const int mreq = m[2], mg = m[3], mmt = m[4], c1 = m[5], c2 = m[6];
    const int np = c2 - c1 + 1;
    auto slot_of = [&](int c) { return 2 * c + ((c == c1 && cta_start(c1, T_all, G_eff) < ustart) ? 1 : 0); };
    const int rows = min(kRows, M - mmt * kRows);
    const float2* ml2 = reinterpret_cast<const float2*>(args.slot_ml);
    constexpr int C4 = D / 4;
    static_assert(32 % C4 == 0, "a warp instruction covers whole output rows");
    if (np <= 2) {
      // the common split (a unit over two CTAs): each warp takes a block of
      // rows and issues every load for them -- both pieces' (m, l) and O --
      // before using any, so the merge is one round trip; no shared memory,
      // no block barrier.  Lane: row offset lane / C4, 4 columns lane % C4.
      constexpr int kRPI = 32 / C4;  // rows per warp instruction
      constexpr int kRB = 8;         // warp instructions per piece per batch
      const int rsub = lane / C4, c4 = lane % C4;
      const int per_warp = (rows + kTcThreads / 32 - 1) / (kTcThreads / 32);
      const int w0 = warp * per_warp, w1 = min(rows, w0 + per_warp);
      const int s0 = slot_of(c1), s1 = np > 1 ? slot_of(c1 + 1) : s0;
      const float4* o4s = reinterpret_cast<const float4*>(args.slot_o);
      for (int r0 = w0; r0 < w1; r0 += kRPI * kRB) {
        float2 m0[kRB], m1[kRB];
        float4 o0[kRB], o1[kRB];
#pragma unroll
        for (int i = 0; i < kRB; ++i) {
          const int rr = r0 + i * kRPI + rsub;
          const bool on = rr < w1;
          m0[i] = on ? __ldcg(ml2 + size_t(s0) * kRows + rr) : make_float2(-INFINITY, 0.f);
          o0[i] = on ? __ldcg(o4s + (size_t(s0) * kRows + rr) * C4 + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
          m1[i] = on && np > 1 ? __ldcg(ml2 + size_t(s1) * kRows + rr) : make_float2(-INFINITY, 0.f);
          o1[i] = on && np > 1 ? __ldcg(o4s + (size_t(s1) * kRows + rr) * C4 + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < kRB; ++i) {
          const int rr = r0 + i * kRPI + rsub;
          if (rr < w1) {
            float Mx = -INFINITY;
            if (m0[i].y > 0.f) Mx = m0[i].x;
            if (m1[i].y > 0.f) Mx = fmaxf(Mx, m1[i].x);
            const float wa = m0[i].y > 0.f ? exp2f(m0[i].x - Mx) : 0.f;
            const float wb = m1[i].y > 0.f ? exp2f(m1[i].x - Mx) : 0.f;
            const float Ls = m0[i].y * wa + m1[i].y * wb;
            const float li = Ls > 0.f ? 1.f / Ls : 0.f;
            const float ka = wa * li, kb = wb * li;
            const int rg = mmt * kRows + rr;
            const size_t orow = (size_t(mreq) * a.n + rg / G) * a.Hq + mg * G + rg % G;
            *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + orow * D + 4 * c4) =
                make_uint2(pack_bf16(ka * o0[i].x + kb * o1[i].x, ka * o0[i].y + kb * o1[i].y),
                           pack_bf16(ka * o0[i].z + kb * o1[i].z, ka * o0[i].w + kb * o1[i].w));
            if (c4 == 0 && a.lse) a.lse[orow] = Ls > 0.f ? (Mx + log2f(Ls)) * 0.6931471805599453f : -INFINITY;
          }
        }
      }
    } else if (np <= wcap) {
      // per row: the largest running max, each piece's weight, 1 / total
      // ((m, l) pairs loaded eight pieces at a time)
      for (int rr = threadIdx.x; rr < rows; rr += blockDim.x) {
        float Mx = -INFINITY;
        for (int q0 = 0; q0 < np; q0 += 8) {
          float2 v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u)
            v[u] = q0 + u < np ? __ldcg(ml2 + size_t(slot_of(c1 + q0 + u)) * kRows + rr) : make_float2(-INFINITY, 0.f);
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            if (v[u].y > 0.f) Mx = fmaxf(Mx, v[u].x);
            if (q0 + u < np) {
              wsm[(q0 + u) * kRows + rr] = v[u].x;  // the piece's max for now
              wsm[(np + 1 + q0 + u) * kRows + rr] = v[u].y;
            }
          }
        }
        float Ls = 0.f;
        for (int q = 0; q < np; ++q) {
          const float lc = wsm[(np + 1 + q) * kRows + rr];
          const float wq = lc > 0.f ? exp2f(wsm[q * kRows + rr] - Mx) : 0.f;
          wsm[q * kRows + rr] = wq;
          Ls += lc * wq;
        }
        wsm[np * kRows + rr] = Ls > 0.f ? 1.f / Ls : 0.f;
        const int rg = mmt * kRows + rr;
        const size_t orow = (size_t(mreq) * a.n + rg / G) * a.Hq + mg * G + rg % G;
        if (a.lse) a.lse[orow] = Ls > 0.f ? (Mx + log2f(Ls)) * 0.6931471805599453f : -INFINITY;
      }
      __syncthreads();
      // every (row, 4 columns) of the output: the weighted sum over pieces;
      // each thread loads its whole share of one piece before using any of it
      constexpr int U = (kRows * C4 + kTcThreads - 1) / kTcThreads;
      const int total = rows * C4;
      float4 acc[U];
#pragma unroll
      for (int u = 0; u < U; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int q = 0; q < np; ++q) {
        const float4* src = reinterpret_cast<const float4*>(args.slot_o) + size_t(slot_of(c1 + q)) * kRows * C4;
        float4 o4[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int e = threadIdx.x + u * kTcThreads;
          o4[u] = e < total ? __ldcg(src + e) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int e = threadIdx.x + u * kTcThreads;
          const float wq = e < total ? wsm[q * kRows + e / C4] : 0.f;
          acc[u].x += wq * o4[u].x;
          acc[u].y += wq * o4[u].y;
          acc[u].z += wq * o4[u].z;
          acc[u].w += wq * o4[u].w;
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int e = threadIdx.x + u * kTcThreads;
        if (e < total) {
          const int rr = e / C4, c4 = e % C4;
          const float li = wsm[np * kRows + rr];
          const int rg = mmt * kRows + rr;
          const size_t orow = (size_t(mreq) * a.n + rg / G) * a.Hq + mg * G + rg % G;
          *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + orow * D + 4 * c4) =
              make_uint2(pack_bf16(acc[u].x * li, acc[u].y * li), pack_bf16(acc[u].z * li, acc[u].w * li));
        }
      }
    } else if (threadIdx.x < rows) {
      // more pieces than the ring holds weights for: one thread per row, two passes
      const int rr = threadIdx.x;
      float Mx = -INFINITY, Ls = 0.f;
      for (int q = 0; q < np; ++q) Mx = fmaxf(Mx, __ldcg(args.slot_ml + (size_t(slot_of(c1 + q)) * kRows + rr) * 2));
      for (int q = 0; q < np; ++q) {
        const float* ml = args.slot_ml + (size_t(slot_of(c1 + q)) * kRows + rr) * 2;
        const float lc = __ldcg(ml + 1);
        if (lc > 0.f) Ls += lc * exp2f(__ldcg(ml) - Mx);
      }
      const float linv = Ls > 0.f ? 1.f / Ls : 0.f;
      const int rg = mmt * kRows + rr;
      const size_t orow = (size_t(mreq) * a.n + rg / G) * a.Hq + mg * G + rg % G;
      for (int c4 = 0; c4 < D / 4; ++c4) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int q = 0; q < np; ++q) {
          const float* ml = args.slot_ml + (size_t(slot_of(c1 + q)) * kRows + rr) * 2;
          const float lc = __ldcg(ml + 1);
          if (!(lc > 0.f)) continue;
          const float wq = exp2f(__ldcg(ml) - Mx) * linv;
          const float4 o4 = __ldcg(reinterpret_cast<const float4*>(args.slot_o + (size_t(slot_of(c1 + q)) * kRows + rr) * D) + c4);
          acc.x += wq * o4.x;
          acc.y += wq * o4.y;
          acc.z += wq * o4.z;
          acc.w += wq * o4.w;
        }
        *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + orow * D + 4 * c4) =
            make_uint2(pack_bf16(acc.x, acc.y), pack_bf16(acc.z, acc.w));
      }
      if (a.lse) a.lse[orow] = Ls > 0.f ? (Mx + log2f(Ls)) * 0.6931471805599453f : -INFINITY;
    }
    __syncthreads();
    if (threadIdx.x == 0) atomicExch(args.counters + c1, 0u);  // ready for the next launch
  }
}

// ------------------------------------------------------------ host side

template <int D>
int launch_t(const AttentionParams& p, const TcGeometry& geo, cudaStream_t stream) {
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
  unsigned char* base = p.partials;
  TcArgs args{p, geo.m_tiles, p.counters,
              reinterpret_cast<float*>(base + kSlotOOffset),
              reinterpret_cast<float*>(base + kSlotMLOffset)};
  const int grid = sm_count < kMaxCtas ? sm_count : kMaxCtas;
  const cudaError_t e = launch_pdl(attention_tc_kernel<D>, dim3(grid), dim3(kTcThreads), smem, stream, args);
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
}

}  // namespace

TcGeometry attention_tc_geometry(int b, int n, int Hq, int Hkv, int max_seq_len) {
  (void)b;
  (void)max_seq_len;
  TcGeometry geo{};
  geo.m_tiles = (n * (Hq / Hkv) + kRows - 1) / kRows;
  geo.split_tiles = 0;
  geo.splits = 1;  // split units are merged inside the kernel: always one launch
  return geo;
}

size_t attention_partial_bytes() { return kSlotOOffset + size_t(2) * kMaxCtas * kRows * 128 * 4; }

int launch_attention_tc(const AttentionParams& p, const TcGeometry& geo, cudaStream_t stream) {
  if (p.D == 128) return launch_t<128>(p, geo, stream);
  if (p.D == 64) return launch_t<64>(p, geo, stream);
  return SPEC_ERR_UNSUPPORTED;
}

}  // namespace spec
