// stream_records.cu -- the logits streaming pass (group records); see
// stream_records.cuh.
#include "stream_records.cuh"

namespace spec {

namespace {

template <typename T>
__global__ void __launch_bounds__(kStreamThreads, kStreamPerSm) stream_records_kernel(StreamRecParams a) {
  constexpr int E = LogitTraits<T>::kVec;  // elements per 16-byte vector
  // ring: vector u of stage s of lane l of warp w at [((w * stages + s) * Vpt + u) * 32 + l]
  extern __shared__ __align__(16) uint4 ring[];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const unsigned rowU = unsigned(a.V / E);
  const unsigned U = unsigned(a.rows) * rowU;  // (the host keeps it below 2^31)
  const int nu = a.nu;                         // units in all
  const uint4* src = static_cast<const uint4*>(a.logits);
  float2* rec = a.rec;
  // c = log2(e) / T of a row: one temperature, or one a request (T = 0:
  // greedy); formed again only when the row changes
  unsigned sc_row = 0xffffffffu;
  ExpScale sc;
  bool soft = false;
  auto scale_of = [&](unsigned row) {
    if (row != sc_row) {
      const float temp = a.temperatures ? __ldg(a.temperatures + row / unsigned(a.rows_per_temp)) : a.temperature;
      soft = temp > 0.f;
      sc = soft ? ExpScale(temp) : ExpScale();
      sc_row = row;
    }
  };
  uint4* wring = ring + w * (kStreamStages * kUnitVecs) + lane;
  const unsigned long long pol = stream_read_policy();

  // Without overlap: wait for the grid before, then let the grid after (the
  // request step) launch; it waits for this grid to finish before it reads a
  // record.  With overlap the reads start at once and a lane waits before its
  // first record write.
  bool waited = !a.early;
  if (waited) pdl_wait();
  pdl_trigger();

  // Units come in chunks of cu (>= 2) consecutive ones: iteration j works on
  // unit cu * chunk(j / cu) + j % cu.  pc = chunk(j / cu), pn = chunk(j / cu +
  // 1); lane 0 holds the queue's answer for chunk(j / cu + 2).  A warp's
  // chunks are gw, gw + NW, then 2 NW + what the queue hands out.
  const int NW = gridDim.x * kStreamWarps, gw = blockIdx.x * kStreamWarps + w;
  const int cu = a.cu;
  int pc = gw, pn = gw + NW, pending = 0;
  if (lane == 0) pending = 2 * NW + int(atomicAdd(a.queue, 1u));
  auto issue = [&](int j, int unit) {  // stage j % 3 <- unit (an empty group past the last unit)
    if (unit < nu) {
      uint4* st = wring + (unsigned(j) % kStreamStages) * kUnitVecs;
      const unsigned o0 = unsigned(unit) * kUnitVecs + lane;
      if (o0 + (kStreamVpt - 1) * 32 < U) {  // the whole unit exists
#pragma unroll
        for (int u = 0; u < kStreamVpt; ++u) stream_cp16(st + u * 32, src + o0 + u * 32, 16u, pol);
      } else {
#pragma unroll
        for (int u = 0; u < kStreamVpt; ++u) {
          const unsigned o = o0 + u * 32;
          const bool ok = o < U;
          stream_cp16(st + u * 32, ok ? src + o : src, ok ? 16u : 0u, pol);
        }
      }
    }
    stream_commit();
  };
  issue(0, cu * pc);
  issue(1, cu * pc + 1);
  for (int j = 0, jc = 0;; ++j) {  // jc = j % cu
    if (j > 0 && jc == 0) {  // a new chunk
      pc = pn;
      pn = __shfl_sync(0xffffffffu, pending, 0);
      if (lane == 0) pending = 2 * NW + int(atomicAdd(a.queue, 1u));
    }
    const int unit = cu * pc + jc;
    if (unit >= nu) break;  // (a warp's units only grow: every later one is past the end too)
    issue(j + 2, jc + 2 < cu ? unit + 2 : cu * pn + jc + 2 - cu);
    if (++jc == cu) jc = 0;
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
      // (g = -inf: no element, or all -inf: every term is 0; a greedy row
      // needs no sum: 1 marks the group as holding elements)
      scale_of(row);
      const float s = soft ? (g > -INFINITY ? batch_exp_sum<T>(x, sc, g) : 0.f) : 1.f;
      if (!waited) {
        pdl_wait();
        waited = true;
      }
      if (rec) __stcg(&rec[stream_slot(unit, row & 1, lane)], make_float2(g, any ? s : -1.f));
      if (a.usum) {  // the unit summary of this row: over its groups, the maximum and the sum relative to it
        const float gu = warp_max(g);
        const float su = warp_sum(any && s > 0.f ? s * fast_exp2(sc.times(g - gu)) : 0.f);
        if (lane == 0) __stcg(&a.usum[unit * 2 + (row & 1)], make_float2(gu, su));
      }
      cur = seg;
      ++row;
    }
  }
  stream_wait_group<0>();  // no copy of this lane is left in flight (the last groups are empty)
}

}  // namespace

// The streaming split: G CTAs (kStreamPerSm a SM) over the units.  None where
// a row is shorter than a unit (a unit then could span more than two rows),
// where a row has more than kRowRecordsMax records (the request steps hold a
// row's records in shared memory), or where the vector count reaches 2^31.
// bytes: the records alone.
StreamGeometry stream_geometry(long rows, int V, int vec, int sms) {
  const long long rowU = V / vec;
  if (rows < 1 || rowU < kUnitVecs) return StreamGeometry{0, 0, 0};
  if ((rowU / kUnitVecs + 2) * 32 > kRowRecordsMax) return StreamGeometry{0, 0, 0};
  const long long U = rows * rowU;
  if (U >= (1LL << 31) - kUnitVecs) return StreamGeometry{0, 0, 0};
  const long long nu = (U + kUnitVecs - 1) / kUnitVecs;
  long long G = (long long)kStreamPerSm * sms;
  const long long need = (nu + 2 * kStreamWarps - 1) / (2 * kStreamWarps);  // CTAs whose warps get a pair each
  if (G > need) G = need;
  if (G < 1) G = 1;
  const size_t bytes = align256(size_t(nu) * 2 * 32 * sizeof(float2));
  return StreamGeometry{int(G), int(nu), bytes};
}

int launch_stream_records(const StreamRecParams& p0, int ctas, int dtype, cudaStream_t stream) {
  constexpr size_t smem = size_t(kStreamWarps) * kStreamStages * kUnitVecs * 16;
  // units a queue answer hands out: about four answers a warp, 2 to 16 units
  StreamRecParams p = p0;
  const long long nw = (long long)ctas * kStreamWarps;
  long long cu = p.nu / (4 * nw);
  p.cu = int(cu < 2 ? 2 : cu > 16 ? 16 : cu);
  cudaError_t e;
  if (dtype == SPEC_F32) {
    e = cudaFuncSetAttribute(stream_records_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e == cudaSuccess) e = launch_pdl(stream_records_kernel<float>, dim3(ctas), dim3(kStreamThreads), smem, stream, p);
  } else {
    e = cudaFuncSetAttribute(stream_records_kernel<uint16_t>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e == cudaSuccess)
      e = launch_pdl(stream_records_kernel<uint16_t>, dim3(ctas), dim3(kStreamThreads), smem, stream, p);
  }
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
}

}  // namespace spec
