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
// -- 128 slots -- plus the chunk's first 16 staged rows: nine 16-key
// subtiles.  Its query rows are the chunk's (token, head) pairs, C * G <= 32
// of them, in column tiles of 8.  One persistent CTA per SM.  Two producer
// warps stream the CTA's units through two stage sets: one the unit's
// query rows (a 4-D TMA box of the chunk's tokens x the group's heads), its
// RoPE rows and its slot tags; the other its ring K and V (one 128-row TMA box
// each) and its staged rows (a 4-D box of 16 tokens of one KV head).  Two
// groups of four consumer warps take alternate units (group g uses set g).
// In a group, warp w takes column tile w (query rows 8w .. 8w+7) over all
// nine subtiles, so its rows need no merge with another warp's:
//   S^T[16 keys x 8 rows] = K Q^T (m16n8k16, keys as the MMA rows, two
//   accumulation chains), RoPE applied to the Q^T B fragments in registers
//   with each row's own position; masked per row (ring slot: tag in
//   (P0 + i - 128, P0); staged row d: d <= i); online softmax per row across
//   the lanes of one column pair; P^T into B fragments by movmatrix;
//   O^T[128 x 8] += V^T P^T; then the sink joins the denominator, and the
//   accumulators are transposed back (movmatrix) for the row stores.
// V rows no row of the unit may see are zeroed first (0 * NaN is not 0).
//
// Every wait on an mbarrier is bounded: a wait that gives up sets the CTA's
// abort flag and KVR_DEV_TIMEOUT; the consumers stop together at their next
// unit, and the producers wait (bounded) for their loads still in flight.
#include <cuda.h>

#include "launch.h"
#include "tc_ptx.cuh"
#include "warp_attn.cuh"

namespace kvr {
namespace {

constexpr unsigned SS_ST_TIMEOUT = 8u;  // KVR_DEV_TIMEOUT
constexpr int SS_CWARPS = 8;                      // consumer warps, two groups of four
constexpr int SS_GWARPS = 4;
constexpr int SS_GTHREADS = SS_GWARPS * 32;
constexpr int SS_THREADS = SS_CWARPS * 32 + 64;   // + two producer warps
constexpr int SS_ROWS = SWA_SHORT_ROWS;           // query rows of a unit (4 column tiles of 8)
constexpr int SS_DRAFT = SWA_SHORT_MAX_C;         // staged rows per unit
constexpr int SS_RK = WIN * DQK * 2;              // ring K [128][3][128 B], 48 KB
constexpr int SS_RV = WIN * DV * 2;               // ring V [128][2][128 B], 32 KB
constexpr int SS_DK = SS_DRAFT * DQK * 2;         // staged K [16][3][128 B], 6 KB
constexpr int SS_DV = SS_DRAFT * DV * 2;          // staged V [16][2][128 B], 4 KB
// a stage set, from a 1024-byte boundary: the K/V boxes, then the query rows
// [32][3][128 B], the RoPE rows [16][64] fp32 and the slot tags [128]
constexpr int SS_OFF_RV = SS_RK;
constexpr int SS_OFF_DK = SS_OFF_RV + SS_RV;
constexpr int SS_OFF_DV = SS_OFF_DK + SS_DK;
constexpr int SS_OFF_Q = SS_OFF_DV + SS_DV;
constexpr int SS_OFF_CS = SS_OFF_Q + SS_ROWS * DQK * 2;
constexpr int SS_OFF_TAG = SS_OFF_CS + SS_DRAFT * 256;
constexpr int SS_SET = (SS_OFF_TAG + WIN * 4 + 1023) / 1024 * 1024;
// after the two sets: per set the unit record and its rows' sinks (x log2 e),
// then the barriers (kv[2], q[2], free[2], one nothing arrives on: the test
// hook's stall) and the abort flag
constexpr int SS_OFF_REC = 2 * SS_SET;
constexpr int SS_OFF_SINK = SS_OFF_REC + 2 * 32;
constexpr int SS_OFF_BAR = SS_OFF_SINK + 2 * SS_ROWS * 4;
constexpr int SS_OFF_ABORT = SS_OFF_BAR + 7 * 8;
constexpr int SS_SMEM = SS_OFF_ABORT + 16 + 1024;
static_assert(SS_SMEM <= 232448, "one CTA per SM");
static_assert(SS_OFF_RV % 1024 == 0 && SS_OFF_DK % 1024 == 0 && SS_OFF_DV % 1024 == 0 && SS_OFF_Q % 1024 == 0,
              "TMA boxes with the 128-byte swizzle start on 1024-byte boundaries");

struct SsArgs {
  const int64_t *pos_unused;
  const float *sinks;
  const float *table;
  const int32_t *slot_pos;
  const uint16_t *q;
  uint16_t *out;
  unsigned *status;
  VarlenPlan plan;
  int hq, G, hkv;
  int draft_rows;     // rows of one staged box (16, or T when T < 16)
  int q_tokens;       // tokens of one query box (SS_ROWS / G, at most 16, at most T)
  float scale_log2;
  unsigned long long stall_ns;  // test hook: group 0 stalls on its first unit (0 = never)
};

// one unit as the producers find it in the plan and pass it on
struct SsUnit {
  long long c0, P0;
  int C, seq, kv, pad;
};

__device__ __forceinline__ SsUnit ss_unit(const SsArgs &a, int u) {
  SsUnit U;
  const int s = a.plan.short_list[u / a.hkv];
  U.kv = u % a.hkv;
  U.c0 = a.plan.cu_rows[s];
  U.C = (int)(a.plan.cu_rows[s + 1] - U.c0);
  U.P0 = a.plan.P0[s];
  U.seq = a.plan.seq[s];
  U.pad = 0;
  return U;
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// B fragments of Q^T (16 dims x 8 query rows per k-step) for the 12 k-steps,
// from rows r0 .. r0+7 of a [rows][3][128 B] query box: lane l gets row r0 + l/4,
// dims 2(l%4) ..
__device__ __forceinline__ void ss_q_frags(uint32_t qbase, int r0, int lane, uint32_t (&qf)[12][2]) {
#pragma unroll
  for (int kk = 0; kk < 12; kk += 2)
    ldsm_x4(qbase + swrow<3>(r0 + (lane & 7), 2 * kk + (lane >> 3)), qf[kk][0], qf[kk][1], qf[kk + 1][0],
            qf[kk + 1][1]);
}

// Rotate-half RoPE of dims 0..63 on the Q^T B fragments in registers (dims d
// and d + 32 sit in k-steps kk and kk + 2 of the same lane), with the table
// row cs ([32][2] fp32) of this lane's query row; rounded to bf16 as a
// rotated query tile would be.
__device__ __forceinline__ void ss_rope(uint32_t (&qf)[12][2], const float *cs, int lane) {
  const int t = lane & 3;
#pragma unroll
  for (int kk = 0; kk < 2; ++kk)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int d = 16 * kk + 8 * r + 2 * t;
      const float4 c = *reinterpret_cast<const float4 *>(cs + 2 * d);  // (cos, sin) of d and d + 1
      const uint32_t x1 = qf[kk][r], x2 = qf[kk + 2][r];
      const float u0 = bf2f((uint16_t)(x1 & 0xffffu)), u1 = bf2f((uint16_t)(x1 >> 16));
      const float v0 = bf2f((uint16_t)(x2 & 0xffffu)), v1 = bf2f((uint16_t)(x2 >> 16));
      qf[kk][r] = pack_bf16(u0 * c.x - v0 * c.y, u1 * c.z - v1 * c.w);
      qf[kk + 2][r] = pack_bf16(v0 * c.x + u0 * c.y, v1 * c.z + u1 * c.w);
    }
}

// S^T[16 keys x 8 rows] = K Q^T for NS subtiles at once: K rows r0[u] ..
// r0[u]+15 of the [rows][3][128 B] box at kbase[u]; two accumulation chains
// per subtile (even and odd k-steps), all interleaved, so the dependent MMAs
// of one hide the others'.
template <int NS>
__device__ __forceinline__ void ss_qk(const uint32_t (&qf)[12][2], const uint32_t (&kbase)[NS],
                                      const int (&r0)[NS], int lane, float (&s)[NS][4]) {
  float e[NS][4], o[NS][4];
#pragma unroll
  for (int u = 0; u < NS; ++u)
#pragma unroll
    for (int r = 0; r < 4; ++r) e[u][r] = o[u][r] = 0.f;
  const int csel = lane >> 4;
#pragma unroll
  for (int kk = 0; kk < 12; ++kk)
#pragma unroll
    for (int u = 0; u < NS; ++u) {
      uint32_t a[4];
      ldsm_x4(kbase[u] + swrow<3>(r0[u] + (lane & 15), 2 * kk + csel), a[0], a[1], a[2], a[3]);
      mma_bf16(kk & 1 ? o[u] : e[u], a, qf[kk][0], qf[kk][1]);
    }
#pragma unroll
  for (int u = 0; u < NS; ++u)
#pragma unroll
    for (int r = 0; r < 4; ++r) s[u][r] = e[u][r] + o[u][r];
}

// O^T[128 x 8] += V^T P^T for V rows r0 .. r0+15 of a [rows][2][128 B] box;
// pb0 / pb1 are P^T's B fragments for keys 0..7 / 8..15.
__device__ __forceinline__ void ss_pv(uint32_t vbase, int r0, int lane, uint32_t pb0, uint32_t pb1,
                                      float (&O)[8][4]) {
  const int row = r0 + (lane & 7) + ((lane >> 4) << 3), csel = (lane >> 3) & 1;
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    uint32_t a[4];
    ldsm_x4_t(vbase + swrow<2>(row, 2 * m + csel), a[0], a[1], a[2], a[3]);
    mma_bf16(O[m], a, pb0, pb1);
  }
}

// The output row of query row `row` (token row / G, head row % G) of unit U.
__device__ __forceinline__ uint16_t *out_row(const SsArgs &a, const SsUnit &U, int row, bool live) {
  if (!live) return nullptr;
  const int i = row / a.G, h = row % a.G;
  return a.out + ((U.c0 + i) * a.hq + (long long)U.kv * a.G + h) * DV;
}

__global__ void __launch_bounds__(SS_THREADS, 1)
    swa_short_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                     const __grid_constant__ CUtensorMap tdk, const __grid_constant__ CUtensorMap tdv,
                     const __grid_constant__ CUtensorMap tmq, const SsArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + (((smem_u32(smem_raw) + 1023u) & ~1023u) - smem_u32(smem_raw));
  const uint32_t base = smem_u32(smem);
  const uint32_t bar0 = base + SS_OFF_BAR;
  auto kvbar = [&](int set) -> uint32_t { return bar0 + 8 * set; };         // ring and staged K/V landed
  auto qbar = [&](int set) -> uint32_t { return bar0 + 16 + 8 * set; };     // query rows, RoPE rows, tags landed
  auto freebar = [&](int set) -> uint32_t { return bar0 + 32 + 8 * set; };  // the group has read the set
  const uint32_t stallBar = bar0 + 48;                                      // nothing arrives on it
  volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + SS_OFF_ABORT);
  SsUnit *rec = reinterpret_cast<SsUnit *>(smem + SS_OFF_REC);
  float *sSink = reinterpret_cast<float *>(smem + SS_OFF_SINK);  // [2][32]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int set = 0; set < 2; ++set) {
      tc::mbar_init(kvbar(set), 1);
      tc::mbar_init(qbar(set), 1);
      tc::mbar_init(freebar(set), SS_GWARPS);
    }
    tc::mbar_init(stallBar, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  // launched as a programmatic dependent (launch_pdl): the plan read below is
  // the output of the kernel before this one
  pdl_wait();
  __syncthreads();
  pdl_trigger();
  const long long units = (long long)a.plan.short_list[a.plan.n] * a.hkv;

  if (warp >= SS_CWARPS) {
    // ------------------------------------------------------------ producers
    // warp 0 of them: the unit record, its query rows, RoPE rows and slot
    // tags; warp 1: its ring K and V and staged rows.  A unit's description
    // is read from the plan one unit ahead.
    const int pw = warp - SS_CWARPS;
    if (lane == 0) {
      if (pw == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmq) : "memory");
      } else {
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmk) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmv) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tdk) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tdv) : "memory");
      }
    }
    int k = 0;  // units issued
    long long u = blockIdx.x;
    SsUnit Un;
    if (u < units) Un = ss_unit(a, (int)u);
    for (; u < units; u += gridDim.x, ++k) {
      const SsUnit U = Un;
      if (u + gridDim.x < units) Un = ss_unit(a, (int)(u + gridDim.x));
      const int set = k & 1;
      // the set is free once its group has read it for unit k - 2
      if (k >= 2 && !__all_sync(0xffffffffu, tc::mbar_wait(freebar(set), (uint32_t)((k >> 1) - 1) & 1u, abort_flag)))
        break;
      uint8_t *sset = smem + set * SS_SET;
      if (pw == 0) {
        if (lane == 0) rec[set] = U;
        if (lane < U.C * a.G) sSink[set * SS_ROWS + lane] = a.sinks[U.kv * a.G + lane % a.G] * LOG2E;
        __syncwarp();  // the record and sinks before the barrier's arrival
        const uint32_t qb = qbar(set);
        tc::mbar_expect_tx_elect(qb, (uint32_t)(a.q_tokens * a.G * DQK * 2 + U.C * 256 + WIN * 4));
        tc::tma_load_4d_elect(smem_u32(sset + SS_OFF_Q), &tmq, 0, 0, U.kv * a.G, (int)U.c0, qb);
        tc::bulk_load_elect(smem_u32(sset + SS_OFF_CS), a.table + U.P0 * 64, (uint32_t)U.C * 256, qb);
        tc::bulk_load_elect(smem_u32(sset + SS_OFF_TAG), a.slot_pos + (long long)U.seq * WIN, WIN * 4, qb);
      } else {
        const uint32_t kb = kvbar(set);
        const int row = (U.seq * a.hkv + U.kv) * WIN;
        tc::mbar_expect_tx_elect(kb, (uint32_t)(SS_RK + SS_RV + a.draft_rows * (DQK + DV) * 2));
        tc::tma_load_3d_elect(smem_u32(sset), &tmk, 0, 0, row, kb);
        tc::tma_load_3d_elect(smem_u32(sset + SS_OFF_RV), &tmv, 0, 0, row, kb);
        tc::tma_load_4d_elect(smem_u32(sset + SS_OFF_DK), &tdk, 0, 0, U.kv, (int)U.c0, kb);
        tc::tma_load_4d_elect(smem_u32(sset + SS_OFF_DV), &tdv, 0, 0, U.kv, (int)U.c0, kb);
      }
    }
    // before leaving, wait (bounded, whatever the abort flag says) for this
    // warp's loads of the last unit issued into each set
    uint32_t never = 0;
    for (int set = 0; set < 2; ++set) {
      const int n = (k + 1 - set) / 2;  // units issued into this set
      if (n > 0) tc::mbar_wait(pw == 0 ? qbar(set) : kvbar(set), (uint32_t)(n - 1) & 1u, &never);
    }
    if (*abort_flag && lane == 0) flag(a.status, SS_ST_TIMEOUT);
    return;
  }
  // ------------------------------------------------------------ consumers
  // group gr (warps 4gr .. 4gr+3) takes units k = gr, gr + 2, ... from set gr;
  // warp gw of it the query rows 8gw .. 8gw+7 of each unit
  const int gr = warp / SS_GWARPS, gw = warp % SS_GWARPS, ltid = tid % SS_GTHREADS, set = gr;
  const int g = lane >> 2, t = lane & 3;
  const int barA = 1 + 2 * gr, barB = barA + 1;  // the group's named barriers
  uint8_t *sset = smem + set * SS_SET;
  const uint32_t kbase = smem_u32(sset), vbase = kbase + SS_OFF_RV;
  const uint32_t dkbase = kbase + SS_OFF_DK, dvbase = kbase + SS_OFF_DV, qbase = kbase + SS_OFF_Q;
  const float *sCS = reinterpret_cast<const float *>(sset + SS_OFF_CS);
  const int32_t *sTag = reinterpret_cast<const int32_t *>(sset + SS_OFF_TAG);
  const int G = a.G;
  for (long long u = blockIdx.x + (long long)gr * gridDim.x, k = gr; u < units; u += 2LL * gridDim.x, k += 2) {
    const uint32_t par = (uint32_t)(k >> 1) & 1u;
    const bool got_q = __all_sync(0xffffffffu, tc::mbar_wait(qbar(set), par, abort_flag));
    // the group's warps: the unit's record and rows are in, the previous
    // unit's reads of the set are done; a wait that gave up stops them here
    if (!tc::named_bar_and(barA, SS_GTHREADS, got_q && *abort_flag == 0)) break;
    // test hook (stall_ns != 0): group 0 waits on a barrier nothing completes,
    // with the unit's loads in flight; its limit sets the abort flag
    if (a.stall_ns && k == 0) tc::mbar_wait(stallBar, 0, abort_flag, a.stall_ns);
    const SsUnit U = rec[set];
    const int R = U.C * G;
    const long long P0 = U.P0;
    // this thread's S^T / O^T columns (query rows c0r, c0r + 1) and their
    // tokens (-1: padding); the row its B fragments hold
    const int c0r = 8 * gw + 2 * t, c1r = c0r + 1, rowB = 8 * gw + g;
    const int ia = c0r < R ? c0r / G : -1, ib = c1r < R ? c1r / G : -1;
    const bool active = 8 * gw < R;
    const float sk0 = ia >= 0 ? sSink[set * SS_ROWS + c0r] : 0.f;
    const float sk1 = ib >= 0 ? sSink[set * SS_ROWS + c1r] : 0.f;
    uint32_t qf[12][2];
    if (active) {
      ss_q_frags(qbase, 8 * gw, lane, qf);
      ss_rope(qf, sCS + (rowB < R ? rowB / G : 0) * 64, lane);
    }
    const bool got_kv = __all_sync(0xffffffffu, tc::mbar_wait(kvbar(set), par, abort_flag));
    if (got_kv) {
      // V rows no row of the unit may see are zeroed: ring slots whose tag is
      // outside (P0 - 128, P0), staged rows from C on
      const int sp = sTag[ltid];
      if (!(sp >= 0 && sp < P0 && sp > P0 - WIN)) {
#pragma unroll
        for (int ch = 0; ch < 16; ++ch)
          *reinterpret_cast<uint4 *>(smem + (vbase - base) + swrow<2>(ltid, ch)) = make_uint4(0, 0, 0, 0);
      }
      for (int idx = U.C * 16 + ltid; idx < SS_DRAFT * 16; idx += SS_GTHREADS)
        *reinterpret_cast<uint4 *>(smem + (dvbase - base) + swrow<2>(idx >> 4, idx & 15)) = make_uint4(0, 0, 0, 0);
    }
    tc::named_bar_sync(barB, SS_GTHREADS);

    float O[8][4];
#pragma unroll
    for (int m = 0; m < 8; ++m) O[m][0] = O[m][1] = O[m][2] = O[m][3] = 0.f;
    float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;
    if (active && got_kv) {
      // three steps of three subtiles (the last one the staged rows): their
      // scores together, one online-softmax update for all 48 keys, then
      // their P.V
#pragma unroll 1
      for (int j0 = 0; j0 < 9; j0 += 3) {
        uint32_t kb[3];
        int r0[3];
        bool v[3][4];  // key g / g + 8, column 0 / 1 (va0, va1, vb0, vb1)
#pragma unroll
        for (int u = 0; u < 3; ++u) {
          const int jj = j0 + u;
          const bool staged = jj == 8;
          r0[u] = staged ? 0 : 16 * jj;
          kb[u] = staged ? dkbase : kbase;
          if (staged) {
            v[u][0] = ia >= 0 && g <= ia;
            v[u][1] = ib >= 0 && g <= ib;
            v[u][2] = ia >= 0 && g + 8 <= ia;
            v[u][3] = ib >= 0 && g + 8 <= ib;
          } else {
            const long long ta = sTag[r0[u] + g], tb = sTag[r0[u] + g + 8];
            const bool ra = ta >= 0 && ta < P0, rb = tb >= 0 && tb < P0;
            v[u][0] = ia >= 0 && ra && ta > P0 + ia - WIN;
            v[u][1] = ib >= 0 && ra && ta > P0 + ib - WIN;
            v[u][2] = ia >= 0 && rb && tb > P0 + ia - WIN;
            v[u][3] = ib >= 0 && rb && tb > P0 + ib - WIN;
          }
        }
        float sc[3][4];  // per subtile: keys r0 + g, r0 + g + 8 (rows) x query rows c0r, c1r (columns)
        ss_qk<3>(qf, kb, r0, lane, sc);
        float x0 = NEG_INF, x1 = NEG_INF;
#pragma unroll
        for (int u = 0; u < 3; ++u) {
#pragma unroll
          for (int r = 0; r < 4; ++r) sc[u][r] = v[u][r] ? sc[u][r] * a.scale_log2 : NEG_INF;
          x0 = fmaxf(x0, fmaxf(sc[u][0], sc[u][2]));
          x1 = fmaxf(x1, fmaxf(sc[u][1], sc[u][3]));
        }
        // online softmax per column over these 48 keys (the lanes with this t)
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, off));
          x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, off));
        }
        const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
        const float b0f = n0 == NEG_INF ? 0.f : n0, b1f = n1 == NEG_INF ? 0.f : n1;
        const float f0 = ex2(m0 - b0f), f1 = ex2(m1 - b1f);
        m0 = n0;
        m1 = n1;
        l0 *= f0;
        l1 *= f1;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          O[m][0] *= f0;
          O[m][1] *= f1;
          O[m][2] *= f0;
          O[m][3] *= f1;
        }
#pragma unroll
        for (int u = 0; u < 3; ++u) {
          const float p0 = ex2(sc[u][0] - b0f), p1 = ex2(sc[u][1] - b1f);
          const float p2 = ex2(sc[u][2] - b0f), p3 = ex2(sc[u][3] - b1f);
          l0 += p0 + p2;
          l1 += p1 + p3;
          // P^T as B fragments: each 8x8 block [keys][columns] transposed in registers
          const uint32_t pb0 = movmatrix_t(pack_bf16(p0, p1)), pb1 = movmatrix_t(pack_bf16(p2, p3));
          ss_pv(j0 + u == 8 ? dvbase : vbase, r0[u], lane, pb0, pb1, O);
        }
      }
    }
    // the warp is done with the set: hand it back; its generic writes there
    // (zeroed rows) come before the next TMA writes into it
    tc::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(freebar(set));

    if (active && got_kv) {
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
      }
      // the sink joins each row's denominator only
      const float M0 = fmaxf(m0, sk0), M1 = fmaxf(m1, sk1);
      const float e0 = m0 == NEG_INF ? 0.f : ex2(m0 - M0), e1 = m1 == NEG_INF ? 0.f : ex2(m1 - M1);
      const float s0 = e0 / (l0 * e0 + ex2(sk0 - M0)), s1 = e1 / (l1 * e1 + ex2(sk1 - M1));
      // back to [row][value dim]: each 8x8 block of O^T transposed in
      // registers, lane l then holds row 8gw + l/4, dims 2(l%4), 2(l%4) + 1
      const bool store = rowB < R;
      uint16_t *orow = out_row(a, U, rowB, store);
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const uint32_t y0 = movmatrix_t(pack_bf16(O[m][0] * s0, O[m][1] * s1));
        const uint32_t y1 = movmatrix_t(pack_bf16(O[m][2] * s0, O[m][3] * s1));
        if (store) {
          *reinterpret_cast<uint32_t *>(orow + 16 * m + 2 * t) = y0;
          *reinterpret_cast<uint32_t *>(orow + 16 * m + 8 + 2 * t) = y1;
        }
      }
    }
  }
  if (*abort_flag && ltid == 0) flag(a.status, SS_ST_TIMEOUT);
}

}  // namespace

cudaError_t launch_swa_short(const uint16_t *q, const VarlenPlan &plan, int n, long long T, int hq,
                             const KvView &chunk, const KvView &ring, const float *sinks, const float *table,
                             float softmax_scale, uint16_t *out, unsigned *status, cudaStream_t st) {
  const int hkv = ring.hkv, G = hq / hkv;
  const long long rows = (long long)ring.num_seqs * hkv * WIN;
  if (rows >= (1LL << 31) || T >= (1LL << 31) || G > SS_ROWS) return cudaErrorInvalidValue;
  const int draft_rows = T < SS_DRAFT ? (int)T : SS_DRAFT;
  int q_tokens = SS_ROWS / G < SS_DRAFT ? SS_ROWS / G : SS_DRAFT;
  if (q_tokens > T) q_tokens = (int)T;
  CUtensorMap mk, mv, dk, dv, mq;
  if (!make_tma_map_rows3d(&mk, ring.k, rows, DQK, WIN) || !make_tma_map_rows3d(&mv, ring.v, rows, DV, WIN) ||
      !make_tma_map_tokens4d(&dk, chunk.k, T, hkv, DQK, draft_rows) ||
      !make_tma_map_tokens4d(&dv, chunk.v, T, hkv, DV, draft_rows) ||
      !make_tma_map_tokens4d(&mq, q, T, hq, DQK, q_tokens, false, G))
    return cudaErrorInvalidValue;
  cudaError_t e = ensure_smem_limit(6, (const void *)swa_short_kernel, SS_SMEM);
  if (e != cudaSuccess) return e;
  SsArgs a;
  a.pos_unused = nullptr;
  a.q = q;
  a.sinks = sinks;
  a.table = table;
  a.slot_pos = ring.slot_pos;
  a.out = out;
  a.status = status;
  a.plan = plan;
  a.hq = hq;
  a.G = G;
  a.hkv = hkv;
  a.draft_rows = draft_rows;
  a.q_tokens = q_tokens;
  a.scale_log2 = softmax_scale * LOG2E;
  a.stall_ns = take_stall();
  const long long units = (long long)n * hkv;
  int grid = num_sms();
  if (grid > units) grid = (int)units;
  return launch_pdl(swa_short_kernel, dim3((unsigned)grid), dim3(SS_THREADS), (size_t)SS_SMEM, st, mk, mv, dk, dv, mq, a);
}

}  // namespace kvr
