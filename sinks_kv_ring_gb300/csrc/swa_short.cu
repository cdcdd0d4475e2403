// swa_short.cu -- windowed attention for short chunks: a few tokens per
// sequence checked in one pass, as in the verification of a multi-token-
// prediction draft (the Chinese Xiaomi article, section
// "Decode加速与多模态优化").
//
// Row i of chunk s (position P0 + i of sequence seq) attends positions
// (P0 + i - 128, P0 + i] (gaudi-cookbook "MiMo-V2.6-Flash on Gaudi 2", "What
// was built": exactly the last 128 positions), with the per-head sink in the
// denominator only (colibri "MiMo-V2.6 (Xiaomi)", "What the engine
// implements").  Positions below P0 come from the sequence's ring (its state
// before the chunk, slot tags checked: colibri "System One mode and prompt
// reuse"), positions from P0 on from the chunk's own rows in the staging
// buffer.  A ring cannot hold both: the draft's slots still hold positions
// that the draft's earlier rows need.
//
// A unit is one (chunk, KV head): the whole ring of that (sequence, KV head)
// -- 128 slots, 48 KB of K and 32 KB of V -- plus the chunk's first 16 staged
// rows, brought into shared memory by four TMA boxes (3-D boxes of whole ring
// rows, 4-D boxes of 16 tokens of one KV head).  Its query rows are the
// chunk's (token, head) pairs, C * G <= 32 of them, in m-tiles of 16.  The
// kernel is persistent with two CTAs per SM (one 90 KB stage each), so one
// CTA's products overlap the other's loads; the next unit's query rows and
// slot tags are prefetched into registers.  Per m-tile, with 8 warps:
//   1. warp w: S = Q K^T for ring slots 16w..16w+15; warps 0 and 1 also for
//      the 16 staged rows (8 each); masked per row (ring slot: tag in (P0 + i - 128, P0);
//      staged row d: d <= i and d < C); row maxima;
//   2. M = max(sink, row maxima), P = e^{s - M} as bf16 in shared memory
//      ([16][144] keys), row sums;
//   3. warp w: O[:, 16w..16w+15] = P V over the 144 keys, divided by
//      e^{sink - M} + sum of P.
#include <cuda.h>

#include "launch.h"
#include "tc_ptx.cuh"
#include "warp_attn.cuh"

namespace kvr {
namespace {

using namespace tc;

constexpr int SS_WARPS = 8;
constexpr int SS_THREADS = SS_WARPS * 32;
constexpr int SS_ROWS = SWA_SHORT_ROWS;                    // query rows of a unit (2 m-tiles)
constexpr int SS_DRAFT = SWA_SHORT_MAX_C;                  // staged rows per unit
constexpr int SS_RK = WIN * DQK * 2;                       // ring K, 48 KB
constexpr int SS_RV = WIN * DV * 2;                        // ring V, 32 KB
constexpr int SS_DK = SS_DRAFT * DQK * 2;                  // staged K, 6 KB
constexpr int SS_DVB = SS_DRAFT * DV * 2;                  // staged V, 4 KB
constexpr int SS_STAGE = SS_RK + SS_RV + SS_DK + SS_DVB;   // 90 KB, every part 1024-aligned
constexpr int SS_NSTAGE = 1;
constexpr int SS_CTAS = 2;                                 // CTAs per SM
constexpr int SS_OFF_Q = SS_NSTAGE * SS_STAGE;             // [32][192] bf16, swz<DQK>
constexpr int SS_OFF_TAG = SS_OFF_Q + SS_ROWS * DQK * 2;   // [128] int32
constexpr int SS_PROW = 192;                               // P row stride (24 chunks: the swizzle stays in the row)
constexpr int SS_OFF_P = SS_OFF_TAG + WIN * 4;             // [16][192] bf16
constexpr int SS_OFF_RED = SS_OFF_P + 16 * SS_PROW * 2;    // [8][16] row maxima, then [8][16] row sums
constexpr int SS_OFF_SINK = SS_OFF_RED + 2 * SS_WARPS * 16 * 4;  // [32] the rows' sinks (x log2 e)
constexpr int SS_OFF_BAR = SS_OFF_SINK + SS_ROWS * 4;
constexpr int SS_SMEM = SS_OFF_BAR + 8 * SS_NSTAGE + 16 + 1024;
constexpr unsigned ST_TIMEOUT = 8u;

struct SsArgs {
  const uint16_t *q;
  const float *sinks;
  const float *table;
  const int32_t *slot_pos;
  uint16_t *out;
  unsigned *status;
  VarlenPlan plan;
  int hq, G, hkv;
  int draft_rows;     // rows of one staged box (16, or T when T < 16)
  float scale_log2;
};

struct Unit {
  long long c0, P0;
  int C, seq, kv;
};

__device__ __forceinline__ Unit get_unit(const SsArgs &a, int u) {
  Unit U;
  const int s = a.plan.short_list[u / a.hkv];
  U.kv = u % a.hkv;
  U.c0 = a.plan.cu_rows[s];
  U.C = (int)(a.plan.cu_rows[s + 1] - U.c0);
  U.P0 = a.plan.P0[s];
  U.seq = a.plan.seq[s];
  return U;
}

// One unit's rotated query rows and slot tags, held in registers between
// their global loads and their shared-memory stores.  Thread t covers row
// t / 8: pass-through chunks 8 + 2 (t % 8) and 9 + 2 (t % 8), and, for
// t % 8 < 4, the rotated pair (t % 8, t % 8 + 4).
struct ShortPrefetch {
  uint4 pass[2];
  uint4 r1, r2;
  float4 cs[4];
  int tag;
  float sink;  // row tid's sink (x log2 e), threads 0..31
};

__device__ __forceinline__ void ss_prefetch(const SsArgs &a, const Unit &U, int tid, ShortPrefetch &pf) {
  const int r = tid >> 3, qd = tid & 7;
  const bool live = r < U.C * a.G;
  const long long i = live ? r / a.G : 0;
  const int g = live ? r % a.G : 0;
  const uint4 *q4 = reinterpret_cast<const uint4 *>(a.q + ((U.c0 + i) * a.hq + (long long)U.kv * a.G + g) * DQK);
  const uint4 zero = make_uint4(0, 0, 0, 0);
  pf.pass[0] = live ? q4[8 + 2 * qd] : zero;
  pf.pass[1] = live ? q4[9 + 2 * qd] : zero;
  const bool rot = live && qd < 4;
  pf.r1 = rot ? q4[qd] : zero;
  pf.r2 = rot ? q4[qd + 4] : zero;
  const float4 *tr = reinterpret_cast<const float4 *>(a.table + (U.P0 + i) * 64 + 16 * (qd & 3));
#pragma unroll
  for (int k = 0; k < 4; ++k) pf.cs[k] = rot ? tr[k] : make_float4(0.f, 0.f, 0.f, 0.f);
  pf.tag = tid < WIN ? a.slot_pos[(long long)U.seq * WIN + tid] : -1;
  pf.sink = tid < SS_ROWS && tid < U.C * a.G ? a.sinks[U.kv * a.G + tid % a.G] * LOG2E : 0.f;
}

__device__ __forceinline__ void ss_store(const ShortPrefetch &pf, int tid, uint8_t *sQ, int32_t *sTag,
                                         float *sSink) {
  const int r = tid >> 3, qd = tid & 7;
  *reinterpret_cast<uint4 *>(sQ + swz<DQK>(r, 8 + 2 * qd)) = pf.pass[0];
  *reinterpret_cast<uint4 *>(sQ + swz<DQK>(r, 9 + 2 * qd)) = pf.pass[1];
  if (qd < 4) {
    float cs[16];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      cs[4 * k] = pf.cs[k].x; cs[4 * k + 1] = pf.cs[k].y; cs[4 * k + 2] = pf.cs[k].z; cs[4 * k + 3] = pf.cs[k].w;
    }
    uint4 o1, o2;
    rope_pair8(pf.r1, pf.r2, cs, o1, o2);
    *reinterpret_cast<uint4 *>(sQ + swz<DQK>(r, qd)) = o1;
    *reinterpret_cast<uint4 *>(sQ + swz<DQK>(r, qd + 4)) = o2;
  }
  if (tid < WIN) sTag[tid] = pf.tag;
  if (tid < SS_ROWS) sSink[tid] = pf.sink;
}

__global__ void __launch_bounds__(SS_THREADS, SS_CTAS)
    swa_short_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                     const __grid_constant__ CUtensorMap tdk, const __grid_constant__ CUtensorMap tdv,
                     const SsArgs a) {
  extern __shared__ uint8_t smem_raw[];
  // launched as a programmatic dependent (launch_pdl): the plan it reads is
  // the kernel before it's output
  pdl_wait();
  pdl_trigger();
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *g = smem_raw + (base - raw);
  const uint32_t sBar = base + SS_OFF_BAR;
  volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(g + SS_OFF_BAR + 8 * SS_NSTAGE);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int units = a.plan.short_list[a.plan.n] * a.hkv;
  const int nmine = units > (int)blockIdx.x ? (units - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
  if (nmine == 0) return;
  auto unit_id = [&](int k) { return (int)blockIdx.x + k * (int)gridDim.x; };
  const int G = a.G;
  const uint32_t stage_bytes = SS_RK + SS_RV + (uint32_t)a.draft_rows * (DQK + DV) * 2;

  uint8_t *sQ = g + SS_OFF_Q;
  int32_t *sTag = reinterpret_cast<int32_t *>(g + SS_OFF_TAG);
  uint8_t *sP = g + SS_OFF_P;
  float *sMax = reinterpret_cast<float *>(g + SS_OFF_RED);  // [8][16]
  float *sSum = sMax + SS_WARPS * 16;                      // [8][16]
  float *sSink = reinterpret_cast<float *>(g + SS_OFF_SINK);

  // Thread 0: the four boxes of unit k (described by U) into its stage.
  auto issue = [&](int k, const Unit &U) {
    const uint32_t bar = sBar + 8 * (k % SS_NSTAGE);
    const uint32_t dst = base + (k % SS_NSTAGE) * SS_STAGE;
    const int row = (U.seq * a.hkv + U.kv) * WIN;
    mbar_expect_tx(bar, stage_bytes);
    tma_load_3d(dst, &tmk, 0, 0, row, bar);
    tma_load_3d(dst + SS_RK, &tmv, 0, 0, row, bar);
    tma_load_4d(dst + SS_RK + SS_RV, &tdk, 0, 0, U.kv, (int)U.c0, bar);
    tma_load_4d(dst + SS_RK + SS_RV + SS_DK, &tdv, 0, 0, U.kv, (int)U.c0, bar);
  };
  static_assert(SS_NSTAGE == 1, "the next unit's description is carried one unit ahead");
  int issued = -1;
  // the unit being computed; the next one's description is loaded during it
  Unit U = get_unit(a, unit_id(0));
  if (tid == 0) {
    for (int i = 0; i < SS_NSTAGE; ++i) mbar_init(sBar + 8 * i, 1);
    *abort_flag = 0;
    fence_mbar_init();
    issue(0, U);
    issued = 0;
  }
  {
    ShortPrefetch pf;
    ss_prefetch(a, U, tid, pf);
    ss_store(pf, tid, sQ, sTag, sSink);
  }
  __syncthreads();

  const int qr = lane >> 2;  // this thread's rows within an m-tile: qr and qr + 8
  const int r0 = 16 * warp;  // this warp's ring slots in phase 1
  bool alive = true;
  for (int k = 0; k < nmine && alive; ++k) {
    const bool has_next = k + 1 < nmine;
    ShortPrefetch nx;
    // the next unit's description: its loads go out now, its query rows and
    // tags are fetched after the first m-tile (the description's latency
    // hides behind that m-tile, theirs behind the rest of the unit)
    const Unit Un = has_next ? get_unit(a, unit_id(k + 1)) : U;
    const int st = k % SS_NSTAGE;
    if (!__syncthreads_and(mbar_wait(sBar + 8 * st, (uint32_t)(k / SS_NSTAGE) & 1u, abort_flag))) {
      alive = false;
      break;
    }
    uint8_t *sK = g + st * SS_STAGE;
    uint8_t *sV = sK + SS_RK;
    uint8_t *sDK = sV + SS_RV;
    uint8_t *sDV = sDK + SS_DK;
    const long long P0 = U.P0;
    const int R = U.C * G;

    // V rows no row of the unit may see are zeroed (stale bytes must not
    // reach the product: 0 * NaN is not 0): ring slots whose tag is outside
    // (P0 - 128, P0), staged rows from C on.
    {
      bool in = false;
      if (lane < 16) {
        const int sp = sTag[r0 + lane];
        in = sp >= 0 && sp < P0 && sp > P0 - WIN;
      }
      unsigned bad = __ballot_sync(0xffffffffu, !in) & 0xffffu;
      while (bad) {
        const int r = r0 + __ffs(bad) - 1;
        bad &= bad - 1;
        if (lane < 16) *reinterpret_cast<uint4 *>(sV + swrow<2>(r, lane)) = make_uint4(0, 0, 0, 0);
      }
      for (int idx = U.C * 16 + tid; idx < SS_DRAFT * 16; idx += SS_THREADS)
        *reinterpret_cast<uint4 *>(sDV + swrow<2>(idx >> 4, idx & 15)) = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();

    for (int mt = 0; mt * 16 < R; ++mt) {
      // This thread's two rows: token i, head h; rows past R are padding.
      const int ra = 16 * mt + qr, rb = ra + 8;
      const int ia = ra < R ? ra / G : -1, ib = rb < R ? rb / G : -1;
      const long long pa = P0 + ia, pb = P0 + ib;
      // Phase 1: S over ring slots r0..r0+15 (and the staged rows in warp 0).
      // The Q fragments are loaded per k-step (m-tile rows start on a
      // multiple of 8, so the tile's swizzle applies unchanged).
      float S[2][4], D[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) S[j][e] = D[j][e] = 0.f;
      {
        const uint32_t qb = smem_u32(sQ) + 16 * mt * DQK * 2;
        const uint32_t kb = smem_u32(sK), db = smem_u32(sDK);
        const int csel = lane >> 3;
#pragma unroll
        for (int kk = 0; kk < 12; kk += 2) {
          uint32_t qa[4], qc[4];
          ldsm_x4(qb + swz<DQK>(lane & 15, 2 * kk + (lane >> 4)), qa[0], qa[1], qa[2], qa[3]);
          ldsm_x4(qb + swz<DQK>(lane & 15, 2 * kk + 2 + (lane >> 4)), qc[0], qc[1], qc[2], qc[3]);
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int row = 8 * j + (lane & 7);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kb + swrow<3>(r0 + row, 2 * kk + csel), b0, b1, b2, b3);
            mma_bf16(S[j], qa, b0, b1);
            mma_bf16(S[j], qc, b2, b3);
            if (warp == j) {  // the staged rows' two 8-row halves: warps 0 and 1
              ldsm_x4(db + swrow<3>(row, 2 * kk + csel), b0, b1, b2, b3);
              mma_bf16(D[j], qa, b0, b1);
              mma_bf16(D[j], qc, b2, b3);
            }
          }
        }
      }
      float x0 = NEG_INF, x1 = NEG_INF;
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = 8 * j + 2 * (lane & 3) + (e & 1);
          const int i = e < 2 ? ia : ib;
          const long long pr = e < 2 ? pa : pb;
          const int sp = sTag[r0 + key];
          const bool ok = i >= 0 && sp >= 0 && sp < P0 && sp > pr - WIN;
          S[j][e] = ok ? S[j][e] * a.scale_log2 : NEG_INF;
          const bool okd = warp == j && i >= 0 && key < U.C && key <= i;
          D[j][e] = okd ? D[j][e] * a.scale_log2 : NEG_INF;
          const float m = fmaxf(S[j][e], D[j][e]);
          if (e < 2) x0 = fmaxf(x0, m); else x1 = fmaxf(x1, m);
        }
      x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, 1));
      x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, 2));
      x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, 1));
      x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, 2));
      if ((lane & 3) == 0) {
        sMax[warp * 16 + qr] = x0;
        sMax[warp * 16 + qr + 8] = x1;
      }
      __syncthreads();
      // Phase 2: M = max(sink, all keys); P = e^{s - M}; row sums.
      const float ska = sSink[ra < R ? ra : 0], skb = sSink[rb < R ? rb : 0];
      float M0 = ska, M1 = skb;
#pragma unroll
      for (int w = 0; w < SS_WARPS; ++w) {
        M0 = fmaxf(M0, sMax[w * 16 + qr]);
        M1 = fmaxf(M1, sMax[w * 16 + qr + 8]);
      }
      {
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float p0 = ex2(S[j][0] - M0), p1 = ex2(S[j][1] - M0);
          const float p2 = ex2(S[j][2] - M1), p3 = ex2(S[j][3] - M1);
          s0 += p0 + p1;
          s1 += p2 + p3;
          const int k0 = r0 + 8 * j + 2 * (lane & 3);
          *reinterpret_cast<uint32_t *>(sP + swz<SS_PROW>(qr, k0 >> 3) + (k0 & 7) * 2) = pack_bf16(p0, p1);
          *reinterpret_cast<uint32_t *>(sP + swz<SS_PROW>(qr + 8, k0 >> 3) + (k0 & 7) * 2) = pack_bf16(p2, p3);
        }
        if (warp < 2) {
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            if (j != warp) continue;  // warp j holds the staged rows' half j
            const float p0 = ex2(D[j][0] - M0), p1 = ex2(D[j][1] - M0);
            const float p2 = ex2(D[j][2] - M1), p3 = ex2(D[j][3] - M1);
            s0 += p0 + p1;
            s1 += p2 + p3;
            const int k0 = WIN + 8 * j + 2 * (lane & 3);
            *reinterpret_cast<uint32_t *>(sP + swz<SS_PROW>(qr, k0 >> 3) + (k0 & 7) * 2) = pack_bf16(p0, p1);
            *reinterpret_cast<uint32_t *>(sP + swz<SS_PROW>(qr + 8, k0 >> 3) + (k0 & 7) * 2) = pack_bf16(p2, p3);
          }
        }
        s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
        s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
        s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
        s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
        if ((lane & 3) == 0) {
          sSum[warp * 16 + qr] = s0;
          sSum[warp * 16 + qr + 8] = s1;
        }
      }
      __syncthreads();
      // Phase 3: warp w's value columns 16w..16w+15 over the 144 keys.
      float L0 = ex2(ska - M0), L1 = ex2(skb - M1);
#pragma unroll
      for (int w = 0; w < SS_WARPS; ++w) {
        L0 += sSum[w * 16 + qr];
        L1 += sSum[w * 16 + qr + 8];
      }
      float O[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j) O[j][0] = O[j][1] = O[j][2] = O[j][3] = 0.f;
      {
        const uint32_t pb0 = smem_u32(sP);
        const int vrow = (lane & 7) + (((lane >> 3) & 1) << 3);
        const int vch = 2 * warp + (lane >> 4);
#pragma unroll
        for (int ks = 0; ks < 9; ++ks) {
          uint32_t af[4], b0, b1, b2, b3;
          ldsm_x4(pb0 + swz<SS_PROW>(lane & 15, 2 * ks + (lane >> 4)), af[0], af[1], af[2], af[3]);
          const uint32_t vb = ks < 8 ? smem_u32(sV) + swrow<2>(16 * ks + vrow, vch) : smem_u32(sDV) + swrow<2>(vrow, vch);
          ldsm_x4_t(vb, b0, b1, b2, b3);
          mma_bf16(O[0], af, b0, b1);
          mma_bf16(O[1], af, b2, b3);
        }
      }
      {
        const float i0 = 1.f / L0, i1 = 1.f / L1;  // L >= e^{sink - M} > 0
        const int dcol = 16 * warp + 2 * (lane & 3);
        if (ia >= 0) {
          uint16_t *o = a.out + ((U.c0 + ia) * a.hq + (long long)U.kv * G + ra % G) * DV + dcol;
#pragma unroll
          for (int j = 0; j < 2; ++j)
            *reinterpret_cast<uint32_t *>(o + 8 * j) = pack_bf16(O[j][0] * i0, O[j][1] * i0);
        }
        if (ib >= 0) {
          uint16_t *o = a.out + ((U.c0 + ib) * a.hq + (long long)U.kv * G + rb % G) * DV + dcol;
#pragma unroll
          for (int j = 0; j < 2; ++j)
            *reinterpret_cast<uint32_t *>(o + 8 * j) = pack_bf16(O[j][2] * i1, O[j][3] * i1);
        }
      }
      __syncthreads();  // P and the row arrays are reused by the next m-tile
      if (mt == 0 && has_next) ss_prefetch(a, Un, tid, nx);
    }
    // The unit is done: its query tile, tags and stage are free.
    if (has_next) ss_store(nx, tid, sQ, sTag, sSink);
    fence_proxy_async_smem();  // zeroed V rows (generic writes) before the stage is refilled by TMA
    __syncthreads();
    if (tid == 0 && k + SS_NSTAGE < nmine) {
      issue(k + SS_NSTAGE, Un);
      issued = k + SS_NSTAGE;
    }
    U = Un;
  }

  if (*abort_flag) {
    if (tid == 0) {
      flag(a.status, ST_TIMEOUT);
      // Let the loads already issued land before the CTA exits (time bound only).
      for (int k = issued; k >= 0 && k > issued - SS_NSTAGE; --k) {
        volatile uint32_t local = 0;
        mbar_wait(sBar + 8 * (k % SS_NSTAGE), (uint32_t)(k / SS_NSTAGE) & 1u, &local, 1000000000ull);
      }
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_swa_short(const uint16_t *q, const VarlenPlan &plan, int n, long long T, int hq,
                             const KvView &chunk, const KvView &ring, const float *sinks, const float *table,
                             float softmax_scale, uint16_t *out, unsigned *status, cudaStream_t st) {
  const int hkv = ring.hkv;
  const long long rows = (long long)ring.num_seqs * hkv * WIN;
  if (rows >= (1LL << 31) || T >= (1LL << 31)) return cudaErrorInvalidValue;
  const int draft_rows = T < SS_DRAFT ? (int)T : SS_DRAFT;
  CUtensorMap mk, mv, dk, dv;
  if (!make_tma_map_rows3d(&mk, ring.k, rows, DQK, WIN) || !make_tma_map_rows3d(&mv, ring.v, rows, DV, WIN) ||
      !make_tma_map_tokens4d(&dk, chunk.k, T, hkv, DQK, draft_rows) ||
      !make_tma_map_tokens4d(&dv, chunk.v, T, hkv, DV, draft_rows))
    return cudaErrorInvalidValue;
  cudaError_t e = ensure_smem_limit(6, (const void *)swa_short_kernel, SS_SMEM);
  if (e != cudaSuccess) return e;
  SsArgs a;
  a.q = q;
  a.sinks = sinks;
  a.table = table;
  a.slot_pos = ring.slot_pos;
  a.out = out;
  a.status = status;
  a.plan = plan;
  a.hq = hq;
  a.G = hq / hkv;
  a.hkv = hkv;
  a.draft_rows = draft_rows;
  a.scale_log2 = softmax_scale * LOG2E;
  long long units = (long long)n * hkv;
  int grid = SS_CTAS * num_sms();
  if (grid > units) grid = (int)units;
  return launch_pdl(swa_short_kernel, dim3((unsigned)grid), dim3(SS_THREADS), (size_t)SS_SMEM, st, mk, mv, dk, dv, a);
}

}  // namespace kvr
