// swa_decode.cu -- one-token decode over a windowed layer: 128-slot ring,
// per-head sink, the GQA group of one KV head per unit.
//
// colibri "MiMo-V2.6 (Xiaomi)", "What the engine implements": the sink joins
// the softmax denominator and nothing else; "System One mode and prompt
// reuse": position p sits in slot p mod 128 and the ring records the position
// each slot holds.  gaudi-cookbook "MiMo-V2.6-Flash on Gaudi 2", "What was
// built": the window is exactly the last 128 positions.  Decode is
// memory-bound (Xiaomi "Full-Pipeline Inference Optimization", section 1.2).
//
// A unit is one (sequence, KV head): 128 ring slots, 48 KB of K and 32 KB of
// V, contiguous in the ring, brought into shared memory by two 3-D TMA boxes
// that read whole K and V rows.  The kernel is persistent with two CTAs per
// SM (one 80 KB stage each), so one CTA's products overlap the other's loads;
// the ring rows of all of a CTA's units are staged first, and the next unit's
// query rows and slot tags are prefetched into registers.  Per unit (the code
// can also stream a unit in parts with online rescaling; one part measured
// fastest), with 8 warps:
//   1. warp w: S = Q K^T for slots 16w..16w+15 (m16n8k16, the G query heads
//      are the 16 MMA rows), masked by the slot tags; row maxima;
//   2. the row maximum over all slots and the sink, P = e^{s-M} as bf16 in
//      shared memory, row sums;
//   3. warp w: O[:, 16w..16w+15] = P V over all 128 slots -- the value
//      columns are split across warps, so no warp merges another warp's
//      numerators -- normalised by the full denominator, in which the sink
//      is counted once.
#include <cuda.h>

#include "launch.h"
#include "tc_ptx.cuh"
#include "warp_attn.cuh"

namespace kvr {
namespace {

using namespace tc;

constexpr int SD_WARPS = 8;
constexpr int SD_THREADS = SD_WARPS * 32;
constexpr int SD_CTAS = 2;                               // CTAs per SM
constexpr int SD_SPW = WIN / SD_WARPS;                   // slots per warp in phase 1
constexpr int SD_NT = SD_SPW / 8;                        // 8-key MMA tiles per warp
constexpr int SD_HK = WIN * DQK * 2;                     // K bytes of a unit (48 KB)
constexpr int SD_HV = WIN * DV * 2;                      // V bytes of a unit (32 KB)
constexpr int SD_OFF_Q = SD_HK + SD_HV;                  // two [16][192] query tiles
constexpr int SD_QTILE = 16 * DQK * 2;
constexpr int SD_OFF_TAG = SD_OFF_Q + 2 * SD_QTILE;      // two [128] int32 tag arrays
constexpr int SD_OFF_SINK = SD_OFF_TAG + 2 * WIN * 4;    // [hq] sinks * log2(e)
constexpr int SD_MAX_HQ = 1024;
constexpr int SD_OFF_P = SD_OFF_SINK + SD_MAX_HQ * 4;    // [16][128] bf16 probabilities
constexpr int SD_OFF_RED = SD_OFF_P + 16 * WIN * 2;      // [8 warps][16] row max, then row sums
constexpr int SD_MAX_UNITS = 256;                        // units per CTA whose ring rows are staged
constexpr int SD_OFF_ROW = SD_OFF_RED + 2 * SD_WARPS * 16 * 4;
constexpr int SD_OFF_BAR = SD_OFF_ROW + SD_MAX_UNITS * 4;  // K barrier, V barrier, abort flag
constexpr int SD_SMEM = SD_OFF_BAR + 16 + 32 + 1024;
constexpr unsigned ST_TIMEOUT = 8u;

struct SdArgs {
  const uint16_t *q;
  const int64_t *pos;
  const int32_t *seq;
  const int32_t *slot_pos;
  const float *sinks;
  const float *table;
  uint16_t *out;
  unsigned *status;
  int B, hq, G, hkv, num_seqs;
  long long max_pos;
  float scale_log2;
};

// One unit's query rows and slot tags, held in registers between their global
// loads and their shared-memory stores.
struct UnitPrefetch {
  uint4 pass;    // one of the 16 x 16 plain chunks (dims 64..191)
  uint4 r1, r2;  // one of the 16 x 4 rotated chunk pairs (threads 0..63)
  float4 cs[4];  // its 16 table values
  int tag;       // one slot tag (threads 0..127)
};

__device__ __forceinline__ bool unit_valid(const SdArgs &a, int u, long long &p, int &s) {
  const int b = u / a.hkv;
  p = a.pos[b];
  s = a.seq[b];
  return p >= 0 && p < a.max_pos && s >= 0 && s < a.num_seqs;
}

__device__ __forceinline__ void prefetch_unit(const SdArgs &a, int u, int tid, UnitPrefetch &pf) {
  long long p;
  int s;
  const bool ok = unit_valid(a, u, p, s);
  const int b = u / a.hkv, kv = u % a.hkv;
  const uint16_t *qb = a.q + ((long long)b * a.hq + (long long)kv * a.G) * DQK;
  const int r = tid >> 4, ch = 8 + (tid & 15);
  // The query rows depend only on the unit, so they are loaded without
  // waiting for the position / sequence checks (an invalid unit is skipped).
  pf.pass = r < a.G ? reinterpret_cast<const uint4 *>(qb + r * DQK)[ch] : make_uint4(0, 0, 0, 0);
  pf.r1 = pf.r2 = make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int k = 0; k < 4; ++k) pf.cs[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (tid < 64) {
    const int rr = tid >> 2, c = tid & 3;
    if (rr < a.G) {
      const uint4 *s4 = reinterpret_cast<const uint4 *>(qb + rr * DQK);
      pf.r1 = s4[c];
      pf.r2 = s4[c + 4];
      if (ok) {
        const float4 *tr = reinterpret_cast<const float4 *>(a.table + p * 64 + 16 * c);
#pragma unroll
        for (int k = 0; k < 4; ++k) pf.cs[k] = tr[k];
      }
    }
  }
  pf.tag = -1;
  if (tid < WIN && ok) pf.tag = a.slot_pos[(long long)s * WIN + tid];
}

// Rotate (threads 0..63) and store a prefetched unit into a Q tile / tag buffer.
__device__ __forceinline__ void store_unit(const UnitPrefetch &pf, int tid, uint8_t *sQ, int32_t *sTag) {
  const int r = tid >> 4, ch = 8 + (tid & 15);
  *reinterpret_cast<uint4 *>(sQ + swz<DQK>(r, ch)) = pf.pass;
  if (tid < 64) {
    const int rr = tid >> 2, c = tid & 3;
    float cs[16];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      cs[4 * k] = pf.cs[k].x; cs[4 * k + 1] = pf.cs[k].y; cs[4 * k + 2] = pf.cs[k].z; cs[4 * k + 3] = pf.cs[k].w;
    }
    uint4 o1, o2;
    rope_pair8(pf.r1, pf.r2, cs, o1, o2);
    *reinterpret_cast<uint4 *>(sQ + swz<DQK>(rr, c)) = o1;
    *reinterpret_cast<uint4 *>(sQ + swz<DQK>(rr, c + 4)) = o2;
  }
  if (tid < WIN) sTag[tid] = pf.tag;
}

__global__ void __launch_bounds__(SD_THREADS, SD_CTAS)
    swa_decode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                      const SdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *g = smem_raw + (base - raw);
  const uint32_t kBar = base + SD_OFF_BAR, vBar = kBar + 8;
  volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(g + SD_OFF_BAR + 16);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int units = a.B * a.hkv;
  const int nmine = units > (int)blockIdx.x ? (units - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
  const int G = a.G;
  auto unit_id = [&](int n) { return (int)blockIdx.x + n * (int)gridDim.x; };
  if (nmine == 0) return;

  float *sSink = reinterpret_cast<float *>(g + SD_OFF_SINK);
  uint8_t *sP = g + SD_OFF_P;
  float *sMax = reinterpret_cast<float *>(g + SD_OFF_RED);  // [8][16]
  float *sSum = sMax + SD_WARPS * 16;                       // [8][16]
  int32_t *sRow = reinterpret_cast<int32_t *>(g + SD_OFF_ROW);
  uint8_t *sK = g, *sV = g + SD_HK;

  // Ring row of this CTA's n-th unit (-1: invalid unit).
  auto ring_row = [&](int n) {
    long long p;
    int s;
    const int u = unit_id(n);
    return unit_valid(a, u, p, s) ? (s * a.hkv + u % a.hkv) * WIN : -1;
  };
  auto row_of = [&](int n) { return n < SD_MAX_UNITS ? sRow[n] : ring_row(n); };
  // Thread 0: the K rows / the V rows of unit n, as one 3-D TMA box of whole
  // rows each, on their own barriers.  An invalid unit still completes the
  // barrier's phase (no bytes).
  auto issue_k = [&](int row) {
    if (row >= 0) {
      mbar_expect_tx(kBar, SD_HK);
      tma_load_3d(base, &tmk, 0, 0, row, kBar);
    } else {
      mbar_arrive(kBar);
    }
  };
  auto issue_v = [&](int row) {
    if (row >= 0) {
      mbar_expect_tx(vBar, SD_HV);
      tma_load_3d(base + SD_HK, &tmv, 0, 0, row, vBar);
    } else {
      mbar_arrive(vBar);
    }
  };

  // The first loads go out before anything else.
  int issued_k = -1, issued_v = -1;  // last unit whose K / V load was issued (thread 0)
  if (tid == 0) {
    mbar_init(kBar, 1);
    mbar_init(vBar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    issue_k(ring_row(0));  // V(0) goes out once K(0) is in (below)
    issued_k = 0;
  }
  for (int n = tid; n < nmine && n < SD_MAX_UNITS; n += SD_THREADS) sRow[n] = ring_row(n);
  for (int h = tid; h < a.hq; h += SD_THREADS) sSink[h] = a.sinks[h] * LOG2E;
  {
    UnitPrefetch pf;
    prefetch_unit(a, unit_id(0), tid, pf);
    store_unit(pf, tid, g + SD_OFF_Q, reinterpret_cast<int32_t *>(g + SD_OFF_TAG));
  }
  __syncthreads();

  const int qr = lane >> 2;  // this thread's MMA rows: qr and qr + 8
  const int r0 = SD_SPW * warp;  // this warp's ring slots in phase 1
  bool alive = true;
  for (int n = 0; n < nmine && alive; ++n) {
    const int u = unit_id(n);
    const int b = u / a.hkv, kv = u % a.hkv;
    long long p;
    int s;
    const bool ok = unit_valid(a, u, p, s);
    const bool has_next = n + 1 < nmine;
    UnitPrefetch nx;
    if (has_next) prefetch_unit(a, unit_id(n + 1), tid, nx);
    uint16_t *orow = a.out + ((long long)b * a.hq + (long long)kv * G) * DV;
    const uint8_t *sQ = g + SD_OFF_Q + (n & 1) * SD_QTILE;
    const int32_t *sTag = reinterpret_cast<const int32_t *>(g + SD_OFF_TAG) + (n & 1) * WIN;
    // The softmax state of this thread's two rows starts at the sink: it is
    // the running maximum and contributes e^{sink - M} = 1 to the sum.
    const float sk0 = qr < G ? sSink[kv * G + qr] : NEG_INF;
    const float sk1 = qr + 8 < G ? sSink[kv * G + qr + 8] : NEG_INF;
    float S[SD_NT][4];

    if (!__syncthreads_and(mbar_wait(kBar, (uint32_t)n & 1u, abort_flag))) {
      alive = false;
      break;
    }
    // All CTAs start at once: their first K rows alone come in sooner than K
    // and V together would, and V(0) then loads during this unit's S = Q K^T.
    if (n == 0 && tid == 0) {
      issue_v(row_of(0));
      issued_v = 0;
    }
    if (ok) {
      // Phase 1: warp w: S = Q K^T for slots 16w .. 16w+15; slots whose tag is
      // outside (p - 128, p] are masked; row maxima.
      uint32_t qf[12][4];
      load_q_frags(sQ, lane, qf);
#pragma unroll
      for (int j = 0; j < SD_NT; ++j) S[j][0] = S[j][1] = S[j][2] = S[j][3] = 0.f;
      const uint32_t kb = smem_u32(sK);
#pragma unroll
      for (int j = 0; j < SD_NT; ++j) {
        const int row = r0 + 8 * j + (lane & 7);
        const int csel = lane >> 3;  // an x4 load covers chunks 2kk .. 2kk+3 (two k-steps)
#pragma unroll
        for (int kk = 0; kk < 12; kk += 2) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kb + swrow<3>(row, 2 * kk + csel), b0, b1, b2, b3);
          mma_bf16(S[j], qf[kk], b0, b1);
          mma_bf16(S[j], qf[kk + 1], b2, b3);
        }
      }
#pragma unroll
      for (int j = 0; j < SD_NT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int sp = sTag[r0 + 8 * j + 2 * (lane & 3) + (e & 1)];
          const bool in = sp >= 0 && sp <= p && sp > p - WIN;
          S[j][e] = in ? S[j][e] * a.scale_log2 : NEG_INF;
        }
      float x0 = NEG_INF, x1 = NEG_INF;
#pragma unroll
      for (int j = 0; j < SD_NT; ++j) {
        x0 = fmaxf(x0, fmaxf(S[j][0], S[j][1]));
        x1 = fmaxf(x1, fmaxf(S[j][2], S[j][3]));
      }
      x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, 1));
      x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, 2));
      x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, 1));
      x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, 2));
      if ((lane & 3) == 0) {
        sMax[warp * 16 + qr] = x0;
        sMax[warp * 16 + qr + 8] = x1;
      }
    }
    __syncthreads();
    // Every warp is done with this unit's K: the next unit's K rows come in
    // while this unit's P.V runs.
    if (tid == 0 && has_next) {
      fence_proxy_async_smem();
      issue_k(row_of(n + 1));
      issued_k = n + 1;
    }
    float M0 = sk0, M1 = sk1;
    if (ok) {
      // Phase 2: the row maximum over all slots and the sink, P = e^{s - M}
      // (bf16) and row sums.
#pragma unroll
      for (int w = 0; w < SD_WARPS; ++w) {
        M0 = fmaxf(M0, sMax[w * 16 + qr]);
        M1 = fmaxf(M1, sMax[w * 16 + qr + 8]);
      }
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int j = 0; j < SD_NT; ++j) {
        const float p0 = ex2(S[j][0] - M0), p1 = ex2(S[j][1] - M0);
        const float p2 = ex2(S[j][2] - M1), p3 = ex2(S[j][3] - M1);
        s0 += p0 + p1;
        s1 += p2 + p3;
        const int k0 = r0 + 8 * j + 2 * (lane & 3);  // P tile [16 rows][128 slots], chunks swizzled by row
        *reinterpret_cast<uint32_t *>(sP + swz<WIN>(qr, k0 >> 3) + (k0 & 7) * 2) = pack_bf16(p0, p1);
        *reinterpret_cast<uint32_t *>(sP + swz<WIN>(qr + 8, k0 >> 3) + (k0 & 7) * 2) = pack_bf16(p2, p3);
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
    if (!__syncthreads_and(mbar_wait(vBar, (uint32_t)n & 1u, abort_flag))) {
      alive = false;
      break;
    }
    if (ok) {
      // V rows of stale slots are zeroed so that their bytes cannot reach the
      // product (P is 0 there, but 0 * NaN is not 0).
      bool valid = false;
      if (lane < SD_SPW) {
        const int sp = sTag[r0 + lane];
        valid = sp >= 0 && sp <= p && sp > p - WIN;
      }
      unsigned bad = __ballot_sync(0xffffffffu, !valid) & ((1u << SD_SPW) - 1u);
      while (bad) {
        const int r = r0 + __ffs(bad) - 1;
        bad &= bad - 1;
        if (lane < 16) *reinterpret_cast<uint4 *>(sV + swrow<2>(r, lane)) = make_uint4(0, 0, 0, 0);
      }
    }
    __syncthreads();
    if (ok) {
      // Phase 3: warp w: O[:, 16w..16w+15] = P V over the 128 slots, divided
      // by the sum (in which the sink counts once).
      const float L0 = (qr < G ? ex2(sk0 - M0) : 0.f), L1 = (qr + 8 < G ? ex2(sk1 - M1) : 0.f);
      float l0 = L0, l1 = L1;
#pragma unroll
      for (int w = 0; w < SD_WARPS; ++w) {
        l0 += sSum[w * 16 + qr];
        l1 += sSum[w * 16 + qr + 8];
      }
      float O[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j) O[j][0] = O[j][1] = O[j][2] = O[j][3] = 0.f;
      const uint32_t pb = smem_u32(sP), vb = smem_u32(sV);
      const int vrow = (lane & 7) + (((lane >> 3) & 1) << 3);
      const int vch = 2 * warp + (lane >> 4);
#pragma unroll
      for (int ks = 0; ks < WIN / 16; ++ks) {
        uint32_t af[4], b0, b1, b2, b3;
        ldsm_x4(pb + swz<WIN>(lane & 15, 2 * ks + (lane >> 4)), af[0], af[1], af[2], af[3]);
        ldsm_x4_t(vb + swrow<2>(16 * ks + vrow, vch), b0, b1, b2, b3);
        mma_bf16(O[0], af, b0, b1);
        mma_bf16(O[1], af, b2, b3);
      }
      const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
      const int dcol = 16 * warp + 2 * (lane & 3);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        if (qr < G)
          *reinterpret_cast<uint32_t *>(orow + qr * DV + dcol + 8 * j) = pack_bf16(O[j][0] * i0, O[j][1] * i0);
        if (qr + 8 < G)
          *reinterpret_cast<uint32_t *>(orow + (qr + 8) * DV + dcol + 8 * j) =
              pack_bf16(O[j][2] * i1, O[j][3] * i1);
      }
    } else {
      for (int idx = tid; idx < G * DV; idx += SD_THREADS) orow[idx] = 0;
      if (tid == 0) flag(a.status, (p < 0 || p >= a.max_pos) ? ST_BAD_POS : ST_BAD_SEQ);
    }
    if (has_next) {
      const int nb = (n + 1) & 1;  // that query tile / tag buffer served unit n - 1
      store_unit(nx, tid, g + SD_OFF_Q + nb * SD_QTILE, reinterpret_cast<int32_t *>(g + SD_OFF_TAG) + nb * WIN);
    }
    fence_proxy_async_smem();  // the zeroed V rows (generic writes) before the next TMA writes there
    __syncthreads();
    // Every warp is done with this unit's V: the next unit's V rows.
    if (tid == 0 && has_next) {
      issue_v(row_of(n + 1));
      issued_v = n + 1;
    }
  }

  if (*abort_flag) {
    if (tid == 0) {
      flag(a.status, ST_TIMEOUT);
      // Let the loads already issued land before the CTA exits (time bound only).
      volatile uint32_t local = 0;
      if (issued_k >= 0) mbar_wait(kBar, (uint32_t)issued_k & 1u, &local, 1000000000ull);
      local = 0;
      if (issued_v >= 0) mbar_wait(vBar, (uint32_t)issued_v & 1u, &local, 1000000000ull);
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_swa_decode(const uint16_t *q, const int64_t *pos, const int32_t *seq, int B, int hq,
                              const KvView &ring, const float *sinks, const float *table,
                              int64_t max_pos, float softmax_scale, uint16_t *out, unsigned *status,
                              cudaStream_t st) {
  const int hkv = ring.hkv;
  const long long rows = (long long)ring.num_seqs * hkv * WIN;
  if (rows >= (1LL << 31)) return cudaErrorInvalidValue;
  CUtensorMap mk, mv;
  if (!make_tma_map_rows3d(&mk, ring.k, rows, DQK, WIN) || !make_tma_map_rows3d(&mv, ring.v, rows, DV, WIN))
    return cudaErrorInvalidValue;
  cudaError_t e = ensure_smem_limit(1, (const void *)swa_decode_kernel, SD_SMEM);
  if (e != cudaSuccess) return e;
  SdArgs a;
  a.q = q;
  a.pos = pos;
  a.seq = seq;
  a.slot_pos = ring.slot_pos;
  a.sinks = sinks;
  a.table = table;
  a.out = out;
  a.status = status;
  a.B = B;
  a.hq = hq;
  a.G = hq / hkv;
  a.hkv = hkv;
  a.num_seqs = ring.num_seqs;
  a.max_pos = max_pos;
  a.scale_log2 = softmax_scale * LOG2E;
  const int units = B * hkv;
  int grid = SD_CTAS * num_sms();
  if (grid > units) grid = units;
  swa_decode_kernel<<<grid, SD_THREADS, SD_SMEM, st>>>(mk, mv, a);
  return cudaGetLastError();
}

}  // namespace kvr
