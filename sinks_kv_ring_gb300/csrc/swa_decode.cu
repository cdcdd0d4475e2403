// swa_decode.cu -- one-token decode over a windowed layer: 128-slot ring,
// per-head sink, the GQA group of one KV head per unit.
//
// colibri "MiMo-V2.6 (Xiaomi)", "What the engine implements": the sink joins
// the softmax denominator and nothing else; "System One mode and prompt
// reuse": position p sits in slot p mod 128 and the ring records the position
// each slot holds.  gaudi-cookbook "MiMo-V2.6-Flash on Gaudi 2", "What was
// built": the window is exactly the last 128 positions.
//
// A unit is one (sequence, KV head): 128 ring slots = 48 KB of K + 32 KB of V,
// contiguous in the ring.  The kernel is persistent (two CTAs per SM, each
// with one K/V stage, so one CTA's products and merge overlap the other's
// loads): 8 warps compute unit n (16 slots each; the G query heads are the 16
// rows of an m16n8k16 bf16 MMA) from five 128-byte-swizzled TMA boxes, while
// the threads already hold unit n+1's rotated query rows and slot tags in
// registers.  Each warp keeps
// its own softmax state; the 8 states and the sink are merged once at the
// end of the unit.  Decode is memory-bound (Xiaomi "Full-Pipeline Inference
// Optimization", section 1.2): the point of the design is to keep the ring
// bytes streaming while the small products run.
#include <cuda.h>

#include "launch.h"
#include "tc_ptx.cuh"
#include "warp_attn.cuh"

namespace kvr {
namespace {

using namespace tc;

constexpr int SD_WARPS = 8;
constexpr int SD_THREADS = SD_WARPS * 32;
constexpr int SD_BOX = 16384;                        // 128 rows x 128 bytes
constexpr int SD_STAGE = 5 * SD_BOX;                 // K: 3 boxes, V: 2 boxes (80 KB)
constexpr int SD_NSTAGE = 1;                        // K/V stages per CTA (2 CTAs share an SM)
constexpr int SD_OFF_Q = SD_NSTAGE * SD_STAGE;       // two [16][192] query tiles
constexpr int SD_QTILE = 16 * DQK * 2;
constexpr int SD_OFF_TAG = SD_OFF_Q + 2 * SD_QTILE;  // two [128] int32 tag arrays
constexpr int SD_OFF_SINK = SD_OFF_TAG + 2 * WIN * 4;  // [hq] sinks * log2(e)
constexpr int SD_MAX_HQ = 1024;
constexpr int SD_OFF_FAC = SD_OFF_SINK + SD_MAX_HQ * 4;  // [16][8] merge factors, [16] 1/L
constexpr int SD_OFF_BAR = SD_OFF_FAC + 16 * (SD_WARPS + 1) * 4;
constexpr int SD_SMEM = SD_OFF_BAR + 64 + 1024;
constexpr unsigned ST_TIMEOUT = 8u;
static_assert(SD_WARPS * 16 * (MO_STRIDE + 2) * 4 <= SD_STAGE, "merge area fits in a stage");

// Byte offset of 16-byte chunk ch of row r in a [boxes][128 rows][128 B] tile
// written by TMA with the 128-byte swizzle (chunk bits 4..6 ^ row bits 0..2).
__device__ __forceinline__ uint32_t sw128(int r, int ch) {
  return (uint32_t)((ch >> 3) * SD_BOX + r * 128 + (((ch & 7) ^ (r & 7)) << 4));
}

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
  pf.pass = (ok && r < a.G) ? reinterpret_cast<const uint4 *>(qb + r * DQK)[ch] : make_uint4(0, 0, 0, 0);
  pf.r1 = pf.r2 = make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int k = 0; k < 4; ++k) pf.cs[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (tid < 64) {
    const int rr = tid >> 2, c = tid & 3;
    if (ok && rr < a.G) {
      const uint4 *s4 = reinterpret_cast<const uint4 *>(qb + rr * DQK);
      pf.r1 = s4[c];
      pf.r2 = s4[c + 4];
      const float4 *tr = reinterpret_cast<const float4 *>(a.table + p * 64 + 16 * c);
#pragma unroll
      for (int k = 0; k < 4; ++k) pf.cs[k] = tr[k];
    }
  }
  pf.tag = -1;
  if (tid < WIN && ok) pf.tag = a.slot_pos[(long long)s * WIN + tid];
}

// Rotate (threads 0..63) and store a prefetched unit into Q tile / tag buffer.
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

__global__ void __launch_bounds__(SD_THREADS, 2)
    swa_decode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                      const SdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *g = smem_raw + (base - raw);
  const uint32_t sBar = base + SD_OFF_BAR;
  volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(g + SD_OFF_BAR + 32);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int units = a.B * a.hkv;
  const int nmine = units > (int)blockIdx.x ? (units - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
  const int G = a.G;
  auto unit_id = [&](int n) { return (int)blockIdx.x + n * (int)gridDim.x; };

  if (tid == 0) {
    mbar_init(sBar, 1);
    mbar_init(sBar + 8, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  float *sSink = reinterpret_cast<float *>(g + SD_OFF_SINK);
  float *sFac = reinterpret_cast<float *>(g + SD_OFF_FAC);  // [16][8] per-warp factors / L, then [16] 1/L
  for (int h = tid; h < a.hq; h += SD_THREADS) sSink[h] = a.sinks[h] * LOG2E;
  __syncthreads();
  if (nmine == 0) return;

  // Thread 0: the five boxes of unit u into stage st.  An invalid unit still
  // completes its barrier phase (no bytes).
  auto issue = [&](int u, int st) {
    long long p;
    int s;
    const uint32_t bar = sBar + 8 * st;
    if (unit_valid(a, u, p, s)) {
      const int row = (s * a.hkv + u % a.hkv) * WIN;
      const uint32_t dst = base + st * SD_STAGE;
      mbar_expect_tx(bar, SD_STAGE);
      for (int kb = 0; kb < 3; ++kb) tma_load_2d(dst + kb * SD_BOX, &tmk, 64 * kb, row, bar);
      for (int db = 0; db < 2; ++db) tma_load_2d(dst + (3 + db) * SD_BOX, &tmv, 64 * db, row, bar);
    } else {
      mbar_arrive(bar);
    }
  };

  int issued = -1;  // highest unit index whose stage load was issued (thread 0)
  if (tid == 0) {
    for (int n = 0; n < SD_NSTAGE && n < nmine; ++n) {
      issue(unit_id(n), n);
      issued = n;
    }
  }
  {
    UnitPrefetch pf;
    prefetch_unit(a, unit_id(0), tid, pf);
    store_unit(pf, tid, g + SD_OFF_Q, reinterpret_cast<int32_t *>(g + SD_OFF_TAG));
  }
  __syncthreads();

  for (int n = 0; n < nmine; ++n) {
    const int st = n % SD_NSTAGE;
    const int u = unit_id(n);
    const int b = u / a.hkv, kv = u % a.hkv;
    long long p;
    int s;
    const bool ok = unit_valid(a, u, p, s);
    const bool has_next = n + 1 < nmine;
    UnitPrefetch nx;
    if (has_next) prefetch_unit(a, unit_id(n + 1), tid, nx);

    const bool landed =
        __syncthreads_and(mbar_wait(sBar + 8 * st, (uint32_t)(n / SD_NSTAGE) & 1u, abort_flag));
    if (!landed) break;
    uint16_t *orow = a.out + ((long long)b * a.hq + (long long)kv * G) * DV;
    uint8_t *sK = g + st * SD_STAGE;
    uint8_t *sV = sK + 3 * SD_BOX;
    const uint8_t *sQ = g + SD_OFF_Q + (n & 1) * SD_QTILE;
    const int32_t *sTag = reinterpret_cast<const int32_t *>(g + SD_OFF_TAG) + (n & 1) * WIN;

    if (ok) {
      // A slot is in the window iff it holds a position in (p - 128, p].
      // Zero the V rows of slots outside it so that stale bytes cannot
      // reach the product (their P is 0, but 0 * NaN is not).
      const int r0 = 16 * warp;
      bool valid = false;
      if (lane < 16) {
        const int sp = sTag[r0 + lane];
        valid = sp >= 0 && sp <= p && sp > p - WIN;
      }
      unsigned bad = __ballot_sync(0xffffffffu, !valid) & 0xffffu;
      while (bad) {
        const int r = r0 + __ffs(bad) - 1;
        bad &= bad - 1;
        if (lane < 16) *reinterpret_cast<uint4 *>(sV + sw128(r, lane)) = make_uint4(0, 0, 0, 0);
      }
      __syncwarp();

      uint32_t qf[12][4];
      load_q_frags(sQ, lane, qf);
      float S[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j) S[j][0] = S[j][1] = S[j][2] = S[j][3] = 0.f;
      const uint32_t kb = smem_u32(sK), vb = smem_u32(sV);
      {
        const int row = r0 + (lane & 7) + ((lane >> 4) << 3);
        const int csel = (lane >> 3) & 1;
#pragma unroll
        for (int kk = 0; kk < 12; ++kk) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kb + sw128(row, 2 * kk + csel), b0, b1, b2, b3);
          mma_bf16(S[0], qf[kk], b0, b1);
          mma_bf16(S[1], qf[kk], b2, b3);
        }
      }
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int slot = r0 + 8 * j + 2 * (lane & 3) + (e & 1);
          const int sp = sTag[slot];
          const bool in = sp >= 0 && sp <= p && sp > p - WIN;
          S[j][e] = in ? S[j][e] * a.scale_log2 : NEG_INF;
        }
      float O[16][4];
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) O[nt][0] = O[nt][1] = O[nt][2] = O[nt][3] = 0.f;
      float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;
      softmax_update(S, m0, m1, l0, l1, O);
      {
        uint32_t pa[4];
        pa[0] = pack_bf16(S[0][0], S[0][1]);
        pa[1] = pack_bf16(S[0][2], S[0][3]);
        pa[2] = pack_bf16(S[1][0], S[1][1]);
        pa[3] = pack_bf16(S[1][2], S[1][3]);
        const int row = r0 + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int csel = lane >> 4;
#pragma unroll
        for (int dp = 0; dp < 8; ++dp) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vb + sw128(row, 2 * dp + csel), b0, b1, b2, b3);
          mma_bf16(O[2 * dp], pa, b0, b1);
          mma_bf16(O[2 * dp + 1], pa, b2, b3);
        }
      }
      __syncthreads();  // every warp is done with the stage: reuse it as the merge area
      float *mml = reinterpret_cast<float *>(sK);   // [8][16][2]
      float *mo = mml + SD_WARPS * 32;              // [8][16][MO_STRIDE]
      stash_warp_state(mml + warp * 32, mo + warp * 16 * MO_STRIDE, lane, m0, m1, l0, l1, O);
      __syncthreads();
      // Per query row: the merged max M (sink included), denominator L, and
      // each warp's weight e^{m_w - M} / L.
      if (tid < G) {
        const float sk = sSink[kv * G + tid];
        float M = sk;
#pragma unroll
        for (int w = 0; w < SD_WARPS; ++w) M = fmaxf(M, mml[w * 32 + tid * 2]);
        float f[SD_WARPS];
        float L = ex2(sk - M);
#pragma unroll
        for (int w = 0; w < SD_WARPS; ++w) {
          const float mw = mml[w * 32 + tid * 2];
          f[w] = mw == NEG_INF ? 0.f : ex2(mw - M);
          L += mml[w * 32 + tid * 2 + 1] * f[w];
        }
        const float inv = 1.f / L;
#pragma unroll
        for (int w = 0; w < SD_WARPS; ++w) sFac[tid * SD_WARPS + w] = f[w] * inv;
      }
      __syncthreads();
      for (int idx = tid; idx < G * DV; idx += SD_THREADS) {
        const int gq = idx >> 7, d = idx & (DV - 1);
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < SD_WARPS; ++w) acc += mo[(w * 16 + gq) * MO_STRIDE + d] * sFac[gq * SD_WARPS + w];
        orow[idx] = f2bf(acc);
      }
    } else {
      for (int idx = tid; idx < G * DV; idx += SD_THREADS) orow[idx] = 0;
      if (tid == 0) flag(a.status, (p < 0 || p >= a.max_pos) ? ST_BAD_POS : ST_BAD_SEQ);
    }
    __syncthreads();  // stage st, query tile st and tags st are free again
    if (has_next) {
      const int nb = (n + 1) & 1;
      store_unit(nx, tid, g + SD_OFF_Q + nb * SD_QTILE, reinterpret_cast<int32_t *>(g + SD_OFF_TAG) + nb * WIN);
    }
    if (tid == 0 && n + SD_NSTAGE < nmine) {
      fence_proxy_async_smem();  // the merge area's generic accesses before the TMA writes
      issue(unit_id(n + SD_NSTAGE), st);
      issued = n + SD_NSTAGE;
    }
    __syncthreads();
  }

  if (*abort_flag) {
    if (tid == 0) {
      flag(a.status, ST_TIMEOUT);
      // Let the loads already issued land before the CTA exits (time bound only).
      for (int m = issued; m >= 0 && m > issued - SD_NSTAGE; --m) {
        volatile uint32_t local = 0;
        mbar_wait(sBar + 8 * (m % SD_NSTAGE), (uint32_t)(m / SD_NSTAGE) & 1u, &local, 1000000000ull);
      }
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
  if (!make_tma_map_2d(&mk, ring.k, rows, DQK, WIN) || !make_tma_map_2d(&mv, ring.v, rows, DV, WIN))
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
  int grid = 2 * num_sms();
  if (grid > units) grid = units;
  swa_decode_kernel<<<grid, SD_THREADS, SD_SMEM, st>>>(mk, mv, a);
  return cudaGetLastError();
}

}  // namespace kvr
