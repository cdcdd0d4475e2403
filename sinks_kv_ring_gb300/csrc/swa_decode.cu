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
// V, contiguous in the ring.  One persistent CTA per SM.  A producer warp
// streams the CTA's units, in the order they are needed, through a ring of
// 16 KB chunks: per unit the three 64-dim parts of K and the two 64-dim
// parts of V, each [128 slots][128 B] with the 128-byte swizzle (one TMA box
// each), plus a small entry holding the unit's G query rows, its 128 slot
// tags and its RoPE table row.  Each chunk goes back to the producer as soon
// as its readers are done with it, so the next unit of a group loads while
// the group still computes on the one before.
//
// Two consumer groups of four warps take alternate units, so that one
// group's chain of dependent steps (products, cross-warp reductions,
// barriers) runs while the other's does.  Per unit, with the ring slots as
// the MMA rows (the G query heads, padded to 8 or 16, are the MMA columns,
// so no product is spent on padding rows at G = 8):
//   1. warp w: S^T = K q^T for slots 32w..32w+31 (m16n8k16: A = K rows, B =
//      the rotated query heads; RoPE is applied to the B fragments in
//      registers), masked by the slot tags; per-head maxima over its slots;
//   2. the per-head maximum over all slots and the sink, P = e^{s-M}: each
//      8x8 block of the S^T accumulators is transposed in registers
//      (movmatrix) into the [head][slot] layout that P.V reads, stored as
//      bf16; per-head sums;
//   3. warp w: O^T[32w..32w+31][heads] = V^T P^T over the 128 slots (A = V
//      rows read transposed, B = P), normalised by the full denominator, in
//      which the sink is counted once; the accumulators are transposed back
//      to [head][value dim] for the stores.
#include <cuda.h>

#include "launch.h"
#include "tc_ptx.cuh"
#include "warp_attn.cuh"

namespace kvr {
namespace {

using namespace tc;

constexpr int SD_GWARPS = 4;                        // warps per consumer group
constexpr int SD_SPW = WIN / SD_GWARPS;             // slots per consumer warp in S (32)
constexpr int SD_CHUNK = WIN * 64 * 2;              // one 64-dim part of 128 rows (16 KB)
constexpr int SD_KPARTS = DQK / 64, SD_VPARTS = DV / 64;
constexpr int SD_UCHUNKS = SD_KPARTS + SD_VPARTS;   // chunks per unit
constexpr int SD_TAGS = WIN * 4;                    // one sequence's slot tags
constexpr int SD_TAB = 32 * 2 * 4;                  // one RoPE table row
constexpr int SD_MAX_UNITS = 128;                   // units per CTA whose ring rows are staged at start
constexpr unsigned ST_TIMEOUT = 8u;

// Shape of the kernel for NT column tiles of 8 query heads (G <= 8 * NT):
// NG_ consumer groups (each with its own producer warp), R chunks of ring per
// group.  A group's ring places only ever pass between that group's units,
// which it takes in order, so every wait on a place is for the phase right
// after the one the group saw last.  At G <= 8 the CTA has four groups (one
// CTA per SM) or two (two CTAs per SM; see launch_nt).
template <int NT, int NG_>
struct SdLayout {
  static constexpr int NG = NG_;
  static constexpr int CTAS = NT == 1 && NG <= 2 ? 2 : 1;  // resident CTAs per SM
  // ring places per group: a one-group CTA holds a whole unit (five chunks)
  static constexpr int R = NT == 1 ? (NG == 1 ? SD_UCHUNKS : 3) : 6;
  static constexpr int WARPS = NG * (SD_GWARPS + 1);
  static constexpr int THREADS = WARPS * 32;
  static constexpr int QROWS = 8 * NT;
  static constexpr int QBYTES = QROWS * DQK * 2;        // a multiple of 1024 (swizzle atoms)
  static constexpr int META = QBYTES + 1024;            // q rows | tags | table row (one entry per group)
  static constexpr int GRP = QROWS * WIN * 2 + 2 * SD_GWARPS * 16 * 4 + SD_GWARPS * 4;
  static constexpr int OFF_C = 0;
  static constexpr int OFF_M = OFF_C + NG * R * SD_CHUNK;
  static constexpr int OFF_G = OFF_M + NG * META;       // per group: P [QROWS][128] bf16, max, sum, stale masks
  static constexpr int OFF_INFO = OFF_G + NG * GRP;     // per group: (position, ring row) of its entry
  static constexpr int OFF_ROW = OFF_INFO + NG * 8;     // [SD_MAX_UNITS] (ring row, position)
  static constexpr int OFF_GO = OFF_ROW + SD_MAX_UNITS * 8;  // [NG] int: producer gi has queued its first K parts
  static constexpr int OFF_BAR = OFF_GO + 64;
  static constexpr int NBAR = NG * (2 * R + 2) + 1;     // per group: chunk full/empty, entry full/empty; stall
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 8 + 1024;
  static_assert(OFF_M % 1024 == 0 && META % 1024 == 0, "swizzled tiles need 1024-byte alignment");
  static_assert(GRP % 16 == 0 && OFF_BAR % 8 == 0, "alignment");
  static_assert(SMEM <= 232448, "shared memory per CTA");
  static_assert(NG + 1 <= 16, "named barriers");
};

struct SdArgs {
  const uint16_t *k, *v;  // ring rows (for the L2 prefetch only; the loads go through the tensor maps)
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
  unsigned long long stall_ns;  // test hook: group 0 stalls on its first unit (0 = never)
};

// Ring row of unit u (its first K/V row) and its position.  Row -1: the
// position is outside the table; -2: the sequence id is outside the ring.
__device__ __forceinline__ int unit_row(const SdArgs &a, int u, int &p32) {
  const int b = u / a.hkv;
  const long long p = a.pos[b];
  const int s = a.seq[b];
  p32 = 0;
  if (p < 0 || p >= a.max_pos) return -1;
  if (s < 0 || s >= a.num_seqs) return -2;
  p32 = (int)p;
  return (s * a.hkv + u % a.hkv) * WIN;
}

// The K and V rows of the unit whose first ring row is `row` into L2.
__device__ __forceinline__ void prefetch_unit(const SdArgs &a, long long row) {
  prefetch_l2(a.k + row * DQK, WIN * DQK * 2);
  prefetch_l2(a.v + row * DV, WIN * DV * 2);
}

__device__ __forceinline__ void prefetch_tmap(const void *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// Transpose of an 8x8 bf16 block held as m16n8 accumulator pairs: thread t
// holds row t/4, columns 2(t%4), 2(t%4)+1 before and after.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

__device__ __forceinline__ bool in_window(int t, int p) { return t >= 0 && t <= p && t > p - WIN; }

template <int NT, int NG_>
__global__ void __launch_bounds__(SdLayout<NT, NG_>::THREADS, SdLayout<NT, NG_>::CTAS)
    swa_decode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                      const __grid_constant__ CUtensorMap tmq, const SdArgs a) {
  using L = SdLayout<NT, NG_>;
  constexpr int NG = L::NG, R = L::R;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *g = smem_raw + (base - raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int units = a.B * a.hkv;
  const int grid = (int)gridDim.x;
  const int nmine = units > (int)blockIdx.x ? (units - (int)blockIdx.x + grid - 1) / grid : 0;
  if (nmine == 0) return;
  auto unit_id = [&](int n) { return (int)blockIdx.x + n * grid; };
  const int G = a.G;

  // Barriers: per group gi, ring places gi*R .. gi*R+R-1 (full, empty) and
  // its entry (full, empty).
  const uint32_t bar0 = base + L::OFF_BAR;
  auto cFull = [&](int pl) { return bar0 + 8u * pl; };
  auto cEmpty = [&](int pl) { return bar0 + 8u * (NG * R + pl); };
  auto mFull = [&](int gi) { return bar0 + 8u * (2 * NG * R + gi); };
  auto mEmpty = [&](int gi) { return bar0 + 8u * (2 * NG * R + NG + gi); };
  const uint32_t stallBar = bar0 + 8u * (2 * NG * R + 2 * NG);  // nothing arrives on it
  volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(g + L::OFF_BAR + 8 * L::NBAR);
  int2 *sRow = reinterpret_cast<int2 *>(g + L::OFF_ROW);
  int2 *sInfo = reinterpret_cast<int2 *>(g + L::OFF_INFO);
  volatile int *sGo = reinterpret_cast<volatile int *>(g + L::OFF_GO);
  const bool producer = warp >= NG * SD_GWARPS;
  // Launched as a programmatic dependent (launch_pdl): the set-up below
  // overlaps the end of the kernel before it on the stream; before pdl_wait
  // global memory is only read to choose an L2 prefetch (ld_early_s32).

  if (tid == 0) {
    for (int pl = 0; pl < NG * R; ++pl) {
      mbar_init(cFull(pl), 1);
      mbar_init(cEmpty(pl), SD_GWARPS);
    }
    for (int gi = 0; gi < NG; ++gi) {
      mbar_init(mFull(gi), 1);
      mbar_init(mEmpty(gi), SD_GWARPS);
    }
    mbar_init(stallBar, 1);
    *abort_flag = 0;
    for (int gi = 0; gi < NG; ++gi) sGo[gi] = 0;
    fence_mbar_init();
  }
  if (producer) {
    const int pw = warp - NG * SD_GWARPS;
    if (pw == 0 && lane == 0) {
      prefetch_tmap(&tmk);
      prefetch_tmap(&tmv);
      prefetch_tmap(&tmq);
    }
    // While the kernel ahead may still run, the ring rows of group pw's first
    // unit are requested into L2 from a sequence id read early (see
    // ld_early_s32): the DRAM then streams across the boundary between the
    // two kernels instead of idling through this CTA's start.  Ids outside
    // the ring are not prefetched.  (Only the first units: a prefetch of
    // each next unit inside the loop, which occupies the TMA unit ahead of
    // the loads that fill the ring, made batch 256 slower, 30 -> 37 us.)
    if (lane == 0 && pw < nmine) {
      const int u = unit_id(pw);
      const int s = ld_early_s32(a.seq + u / a.hkv);
      if (s >= 0 && s < a.num_seqs) prefetch_unit(a, ((long long)s * a.hkv + u % a.hkv) * WIN);
    }
    pdl_wait();
    // One round of independent loads for the ring rows of the CTA's units.
    for (int n = pw * 32 + lane; n < nmine && n < SD_MAX_UNITS; n += NG * 32) {
      int p;
      const int row = unit_row(a, unit_id(n), p);
      sRow[n] = make_int2(row, p);
    }
  } else {
    pdl_wait();
    // Query rows G..QROWS-1 of every entry stay zero (the loads bring G rows).
    const int per = (L::QROWS - G) * (DQK / 8);
    for (int i = tid; i < NG * per; i += NG * SD_GWARPS * 32) {
      const int e = i / per, r = G + (i % per) / (DQK / 8), ch = (i % per) % (DQK / 8);
      *reinterpret_cast<uint4 *>(g + L::OFF_M + e * L::META + swrow<3>(r, ch)) = make_uint4(0, 0, 0, 0);
    }
  }
  __syncthreads();
  pdl_trigger();  // (every thread has passed pdl_wait)

  if (producer) {
    // ------------------------------------------------------------ producer
    // Group gi's units in order: the entry (q rows, tags, table row), then
    // the K parts, then the V parts, each as soon as its place is free.
    const int gi = warp - NG * SD_GWARPS;
    const uint32_t mbytes = (uint32_t)G * DQK * 2 + SD_TAGS + SD_TAB;
    const uint32_t mdst = base + L::OFF_M + gi * L::META;
    int issued_c = 0, issued_m = 0;
    bool alive = true;
    for (int m = 0; alive; ++m) {
      const int n = NG * m + gi;
      if (n >= nmine) break;
      int2 rp;
      if (n < SD_MAX_UNITS) {
        rp = sRow[n];
      } else {
        int p;
        const int row = unit_row(a, unit_id(n), p);
        rp = make_int2(row, p);
      }
      const int row = rp.x, p = rp.y;
      const int u = unit_id(n);
      if (m == 0 && gi > 0) {
        // The first units' loads queue in unit order (group gi - 1's K parts
        // before group gi's), so they land, and are computed, one after the
        // other rather than all at the end.
        const uint64_t t0 = global_ns();
        while (!sGo[gi - 1] && !*abort_flag) {
          __nanosleep(32);
          if (global_ns() - t0 > 2000000000ull) *abort_flag = 1;
        }
      }
      if (m >= 1 && !mbar_wait(mEmpty(gi), (uint32_t)(m - 1) & 1u, abort_flag)) break;
      if (lane == 0) sInfo[gi] = make_int2(p, row);
      __syncwarp();
      if (row >= 0) {
        const int b = u / a.hkv, kv = u % a.hkv;
        const int s = row / (WIN * a.hkv);
        mbar_expect_tx_elect(mFull(gi), mbytes);
        tma_load_3d_elect(mdst, &tmq, 0, 0, b * a.hq + kv * G, mFull(gi));
        bulk_load_elect(mdst + L::QBYTES, a.slot_pos + (long long)s * WIN, SD_TAGS, mFull(gi));
        bulk_load_elect(mdst + L::QBYTES + SD_TAGS, a.table + (long long)p * 64, SD_TAB, mFull(gi));
      } else if (lane == 0) {
        mbar_arrive(mFull(gi));
      }
      issued_m = m + 1;
      for (int j = 0; j < SD_UCHUNKS; ++j) {
        const int cg = SD_UCHUNKS * m + j, pl = gi * R + cg % R;
        if (cg >= R && !mbar_wait(cEmpty(pl), (uint32_t)((cg / R) - 1) & 1u, abort_flag)) {
          alive = false;
          break;
        }
        if (row >= 0) {
          mbar_expect_tx_elect(cFull(pl), SD_CHUNK);
          if (j < SD_KPARTS)
            tma_load_3d_elect(base + L::OFF_C + pl * SD_CHUNK, &tmk, 0, j, row, cFull(pl));
          else
            tma_load_3d_elect(base + L::OFF_C + pl * SD_CHUNK, &tmv, 0, j - SD_KPARTS, row, cFull(pl));
        } else if (lane == 0) {
          mbar_arrive(cFull(pl));
        }
        issued_c = cg + 1;
        if (m == 0 && j == SD_KPARTS - 1 && lane == 0) sGo[gi] = 1;
      }
    }
    if (lane == 0) sGo[gi] = 1;  // (also when this group has no unit or gave up)
    // Every load issued lands before this warp exits, so none can outlive
    // the CTA's shared memory even if the consumers give up (time bound
    // only: these waits do not look at the abort flag).
    __syncwarp();
    volatile uint32_t local = 0;
    for (int cg = issued_c - R; cg < issued_c; ++cg)
      if (cg >= 0) mbar_wait(cFull(gi * R + cg % R), (uint32_t)(cg / R) & 1u, &local, 1000000000ull);
    if (issued_m > 0) mbar_wait(mFull(gi), (uint32_t)(issued_m - 1) & 1u, &local, 1000000000ull);
    if (*abort_flag && lane == 0) flag(a.status, ST_TIMEOUT);
    return;
  }

  // -------------------------------------------------------------- consumers
  const int grp = warp / SD_GWARPS, wg = warp % SD_GWARPS;
  const int gtid = tid - grp * SD_GWARPS * 32;
  const int gbar = 1 + grp;  // the group's named barrier
  const int qd = lane & 3, qr = lane >> 2;
  const int r0 = SD_SPW * wg;  // this warp's ring slots in S
  uint8_t *gb = g + L::OFF_G + grp * L::GRP;
  uint8_t *sP = gb;                                                    // [QROWS][128] bf16
  float *sMax = reinterpret_cast<float *>(gb + L::QROWS * WIN * 2);     // [4][16]
  float *sSum = sMax + SD_GWARPS * 16;                                  // [4][16]
  unsigned *sBad = reinterpret_cast<unsigned *>(sSum + SD_GWARPS * 16);  // [4]
  const uint32_t pbase = smem_u32(sP);
  const uint8_t *meta = g + L::OFF_M + grp * L::META;
  auto place = [&](int cg) { return grp * R + cg % R; };

  for (int m = 0;; ++m) {
    const int n = NG * m + grp;
    if (n >= nmine) break;
    const int u = unit_id(n);
    const int b = u / a.hkv, kv = u % a.hkv;
    const int c0 = SD_UCHUNKS * m;
    // sinks of this thread's heads (8 nt + 2 qd + i), in log2 units; -inf
    // for padding heads
    float snk[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int h = 8 * nt + 2 * qd + i;
        snk[nt][i] = h < G ? __ldg(a.sinks + kv * G + h) * LOG2E : NEG_INF;
      }

    // A warp hands a chunk or entry back only when every lane saw it land:
    // after an abort, a place whose load may still be landing is kept.
    const bool got_m = __all_sync(0xffffffffu, mbar_wait(mFull(grp), (uint32_t)m & 1u, abort_flag));
    bool ok = got_m;
    if (a.stall_ns && grp == 0 && m == 0) ok = mbar_wait(stallBar, 0, abort_flag, a.stall_ns) && ok;
    const int2 info = sInfo[grp];
    const int p = info.x;
    const bool valid = ok && info.y >= 0;
    float S[2][NT][4];  // [m-tile][n-tile]: slots r0 + 16 mt + qr (+8), heads 8 nt + 2 qd (+1)
    if (valid) {
      // B fragments of q^T (k = dims, n = heads) for the 12 k-steps; lanes
      // 8j..8j+7 address head rows for chunk 2kk + j.
      uint32_t qf[NT][12][2];
      const uint32_t qbase = smem_u32(meta);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int kk = 0; kk < 12; kk += 2)
          ldsm_x4(qbase + swrow<3>(8 * nt + (lane & 7), 2 * kk + (lane >> 3)), qf[nt][kk][0], qf[nt][kk][1],
                  qf[nt][kk + 1][0], qf[nt][kk + 1][1]);
      // Rotate-half RoPE of dims 0..63: dim d of k-step kk < 2 pairs with
      // d + 32, which sits in the same register of k-step kk + 2.
      const float *tab = reinterpret_cast<const float *>(meta + L::QBYTES + SD_TAGS);
#pragma unroll
      for (int kk = 0; kk < 2; ++kk)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const float4 cs = *reinterpret_cast<const float4 *>(tab + 2 * (16 * kk + 8 * r + 2 * qd));
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const uint32_t x1 = qf[nt][kk][r], x2 = qf[nt][kk + 2][r];
            const float a0 = bf_lo(x1), a1 = bf_hi(x1), b0 = bf_lo(x2), b1 = bf_hi(x2);
            qf[nt][kk][r] = pack_bf16(a0 * cs.x - b0 * cs.y, a1 * cs.z - b1 * cs.w);
            qf[nt][kk + 2][r] = pack_bf16(b0 * cs.x + a0 * cs.y, b1 * cs.z + a1 * cs.w);
          }
        }
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) S[mt][nt][i] = 0.f;
      // S^T for slots r0..r0+31, one K part (four k-steps) per chunk.
      const int arow = r0 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
      for (int j = 0; j < SD_KPARTS; ++j) {
        const int cg = c0 + j, pl = place(cg);
        const bool got = __all_sync(0xffffffffu, mbar_wait(cFull(pl), (uint32_t)(cg / R) & 1u, abort_flag));
        ok = got && ok;
        const uint32_t kb = base + L::OFF_C + pl * SD_CHUNK;
#pragma unroll
        for (int kl = 0; kl < 4; ++kl) {
          const int kk = 4 * j + kl;
          uint32_t a0[4], a1[4];
          ldsm_x4(kb + swrow<1>(arow, 2 * kl + (lane >> 4)), a0[0], a0[1], a0[2], a0[3]);
          ldsm_x4(kb + swrow<1>(arow + 16, 2 * kl + (lane >> 4)), a1[0], a1[1], a1[2], a1[3]);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma_bf16(S[0][nt], a0, qf[nt][kk][0], qf[nt][kk][1]);
            mma_bf16(S[1][nt], a1, qf[nt][kk][0], qf[nt][kk][1]);
          }
        }
        __syncwarp();
        if (lane == 0 && got) mbar_arrive(cEmpty(pl));
      }
    } else {
      // nothing to compute: hand the K parts back as they come
#pragma unroll
      for (int j = 0; j < SD_KPARTS; ++j) {
        const int cg = c0 + j, pl = place(cg);
        const bool got = __all_sync(0xffffffffu, mbar_wait(cFull(pl), (uint32_t)(cg / R) & 1u, abort_flag));
        ok = got && ok;
        if (lane == 0 && got) mbar_arrive(cEmpty(pl));
      }
    }
    if (valid) {
      // Slot tags: a slot counts iff its tag lies in (p - 128, p].
      const int *tags = reinterpret_cast<const int *>(meta + L::QBYTES);
      const unsigned badw = ~__ballot_sync(0xffffffffu, in_window(tags[r0 + lane], p));
      if (lane == 0) sBad[wg] = badw;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        const bool i0 = !((badw >> (16 * mt + qr)) & 1u), i1 = !((badw >> (16 * mt + qr + 8)) & 1u);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          S[mt][nt][0] = i0 ? S[mt][nt][0] * a.scale_log2 : NEG_INF;
          S[mt][nt][1] = i0 ? S[mt][nt][1] * a.scale_log2 : NEG_INF;
          S[mt][nt][2] = i1 ? S[mt][nt][2] * a.scale_log2 : NEG_INF;
          S[mt][nt][3] = i1 ? S[mt][nt][3] * a.scale_log2 : NEG_INF;
        }
      }
    }
    // This warp is done with the entry (q rows, tags, table row).
    __syncwarp();
    if (lane == 0 && got_m) mbar_arrive(mEmpty(grp));
    if (valid) {
      // per-head maxima over this warp's 32 slots
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float m0 = fmax3(S[0][nt][0], S[0][nt][2], fmaxf(S[1][nt][0], S[1][nt][2]));
        float m1 = fmax3(S[0][nt][1], S[0][nt][3], fmaxf(S[1][nt][1], S[1][nt][3]));
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
          m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
        }
        if (qr == 0) *reinterpret_cast<float2 *>(sMax + wg * 16 + 8 * nt + 2 * qd) = make_float2(m0, m1);
      }
    }
    if (!named_bar_and(gbar, SD_GWARPS * 32, ok)) {
      if (gtid == 0) flag(a.status, ST_TIMEOUT);
      break;
    }

    float M[NT][2];
    if (valid) {
      // Per-head maximum over all slots and the sink; P = e^{s - M} as bf16
      // in [head][slot] (8x8 blocks transposed in registers); per-head sums.
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float m0 = snk[nt][0], m1 = snk[nt][1];
#pragma unroll
        for (int ww = 0; ww < SD_GWARPS; ++ww) {
          const float2 x = *reinterpret_cast<const float2 *>(sMax + ww * 16 + 8 * nt + 2 * qd);
          m0 = fmaxf(m0, x.x);
          m1 = fmaxf(m1, x.y);
        }
        M[nt][0] = m0 == NEG_INF ? 0.f : m0;  // only a padding head can have no finite term
        M[nt][1] = m1 == NEG_INF ? 0.f : m1;
        float s0 = 0.f, s1 = 0.f;
        const int hrow = 8 * nt + qr;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          const float p0 = ex2(S[mt][nt][0] - M[nt][0]), p1 = ex2(S[mt][nt][1] - M[nt][1]);
          const float p2 = ex2(S[mt][nt][2] - M[nt][0]), p3 = ex2(S[mt][nt][3] - M[nt][1]);
          s0 += p0 + p2;
          s1 += p1 + p3;
          // block [slot][heads 2qd, 2qd+1] -> [head qr][slots 2qd, 2qd+1]
          const uint32_t x0 = movmatrix_t(pack_bf16(p0, p1));
          const uint32_t x1 = movmatrix_t(pack_bf16(p2, p3));
          const int ca = r0 + 16 * mt + 2 * qd, cb = ca + 8;
          *reinterpret_cast<uint32_t *>(sP + swz<WIN>(hrow, ca >> 3) + (ca & 7) * 2) = x0;
          *reinterpret_cast<uint32_t *>(sP + swz<WIN>(hrow, cb >> 3) + (cb & 7) * 2) = x1;
        }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          s0 += __shfl_xor_sync(0xffffffffu, s0, o);
          s1 += __shfl_xor_sync(0xffffffffu, s1, o);
        }
        if (qr == 0) *reinterpret_cast<float2 *>(sSum + wg * 16 + 8 * nt + 2 * qd) = make_float2(s0, s1);
      }
    }
    // This warp reads value dims 32wg..32wg+31: V part wg/2.
    const int vp = wg >> 1;
    const int cv = c0 + SD_KPARTS + vp, sv = place(cv);
    const bool got_v = __all_sync(0xffffffffu, mbar_wait(cFull(sv), (uint32_t)(cv / R) & 1u, abort_flag));
    ok = got_v && ok;
    uint8_t *sV = g + L::OFF_C + sv * SD_CHUNK;
    if (valid && ok) {
      // V rows of stale slots are zeroed so that their bytes cannot reach the
      // product (P is 0 there, but 0 * NaN is not 0): each of the part's two
      // warps takes 64 slots; then ordered before the next TMA write there.
      const unsigned bb0 = sBad[2 * (wg & 1)], bb1 = sBad[2 * (wg & 1) + 1];
      if (bb0 | bb1) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          unsigned bb = h ? bb1 : bb0;
          while (bb) {
            const int r = 64 * (wg & 1) + 32 * h + __ffs(bb) - 1;
            bb &= bb - 1;
            if (lane < 8) *reinterpret_cast<uint4 *>(sV + swrow<1>(r, lane)) = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
      }
    }
    if (!named_bar_and(gbar, SD_GWARPS * 32, ok)) {
      if (gtid == 0) flag(a.status, ST_TIMEOUT);
      break;
    }

    uint16_t *orow = a.out + ((long long)b * a.hq + (long long)kv * G) * DV;
    if (valid) {
      // O^T[32wg..32wg+31][heads] = V^T P^T over the 128 slots; value dims
      // 32(wg&1) + 16mt.. of this part.
      float O[2][NT][4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) O[mt][nt][i] = 0.f;
      const uint32_t vbase = smem_u32(sV);
      const int vrow = (lane & 7) + ((lane >> 4) << 3);
      const int vch = 4 * (wg & 1) + ((lane >> 3) & 1);
#pragma unroll
      for (int ks = 0; ks < WIN / 16; ks += 2) {
        uint32_t pb[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          ldsm_x4(pbase + swz<WIN>(8 * nt + (lane & 7), 2 * ks + (lane >> 3)), pb[nt][0], pb[nt][1], pb[nt][2],
                  pb[nt][3]);
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2) {
          uint32_t v0[4], v1[4];
          ldsm_x4_t(vbase + swrow<1>(16 * (ks + k2) + vrow, vch), v0[0], v0[1], v0[2], v0[3]);
          ldsm_x4_t(vbase + swrow<1>(16 * (ks + k2) + vrow, vch + 2), v1[0], v1[1], v1[2], v1[3]);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma_bf16(O[0][nt], v0, pb[nt][2 * k2], pb[nt][2 * k2 + 1]);
            mma_bf16(O[1][nt], v1, pb[nt][2 * k2], pb[nt][2 * k2 + 1]);
          }
        }
      }
      // The part's two readers hand it back (two arrivals each: a ring
      // place takes four whatever it holds).
      __syncwarp();
      if (lane == 0 && got_v) mbar_arrive_cnt(cEmpty(sv), SD_GWARPS / SD_VPARTS);
      // Normalise by the denominator (sink once + all slots), transpose each
      // 8x8 block back to [head][value dim] and store.
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float l0 = ex2(snk[nt][0] - M[nt][0]), l1 = ex2(snk[nt][1] - M[nt][1]);
#pragma unroll
        for (int ww = 0; ww < SD_GWARPS; ++ww) {
          const float2 x = *reinterpret_cast<const float2 *>(sSum + ww * 16 + 8 * nt + 2 * qd);
          l0 += x.x;
          l1 += x.y;
        }
        const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
        const int h = 8 * nt + qr;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          const uint32_t y0 = movmatrix_t(pack_bf16(O[mt][nt][0] * i0, O[mt][nt][1] * i1));
          const uint32_t y1 = movmatrix_t(pack_bf16(O[mt][nt][2] * i0, O[mt][nt][3] * i1));
          if (h < G) {
            uint16_t *o = orow + (long long)h * DV + 32 * wg + 16 * mt + 2 * qd;
            *reinterpret_cast<uint32_t *>(o) = y0;
            *reinterpret_cast<uint32_t *>(o + 8) = y1;
          }
        }
      }
    } else {
      __syncwarp();
      if (lane == 0 && got_v) mbar_arrive_cnt(cEmpty(sv), SD_GWARPS / SD_VPARTS);
      for (int i = gtid; i < G * DV / 8; i += SD_GWARPS * 32)
        reinterpret_cast<uint4 *>(orow)[i] = make_uint4(0, 0, 0, 0);
      if (gtid == 0 && ok) flag(a.status, info.y == -1 ? ST_BAD_POS : ST_BAD_SEQ);
    }
  }
}

template <int NT, int NG>
cudaError_t launch_nt(const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mq, const SdArgs &a,
                      int units, int per, cudaStream_t st) {
  using L = SdLayout<NT, NG>;
  cudaError_t e = ensure_smem_limit(NT == 2 ? 12 : NG == 4 ? 1 : NG == 2 ? 14 : 5,
                                    (const void *)swa_decode_kernel<NT, NG>, L::SMEM, L::CTAS > 1);
  if (e != cudaSuccess) return e;
  const int grid = (units + per - 1) / per;
  return launch_pdl(swa_decode_kernel<NT, NG>, dim3((unsigned)grid), dim3(L::THREADS), (size_t)L::SMEM, st, mk, mv,
                    mq, a);
}

}  // namespace

cudaError_t launch_swa_decode(const uint16_t *q, const int64_t *pos, const int32_t *seq, int B, int hq,
                              const KvView &ring, const float *sinks, const float *table,
                              int64_t max_pos, float softmax_scale, uint16_t *out, unsigned *status,
                              cudaStream_t st) {
  const int hkv = ring.hkv;
  const int G = hq / hkv;
  const long long rows = (long long)ring.num_seqs * hkv * WIN;
  if (rows >= (1LL << 31) || (long long)B * hq >= (1LL << 31) || G > 16) return cudaErrorInvalidValue;
  CUtensorMap mk, mv, mq;
  if (!make_tma_map_rows3d(&mk, ring.k, rows, DQK, WIN, true) ||
      !make_tma_map_rows3d(&mv, ring.v, rows, DV, WIN, true) ||
      !make_tma_map_rows3d(&mq, q, (long long)B * hq, DQK, G))
    return cudaErrorInvalidValue;
  SdArgs a;
  a.k = ring.k;
  a.v = ring.v;
  a.pos = pos;
  a.seq = seq;
  a.slot_pos = ring.slot_pos;
  a.sinks = sinks;
  a.table = table;
  a.out = out;
  a.status = status;
  a.B = B;
  a.hq = hq;
  a.G = G;
  a.hkv = hkv;
  a.num_seqs = ring.num_seqs;
  a.max_pos = max_pos;
  a.scale_log2 = softmax_scale * LOG2E;
  a.stall_ns = take_stall();
  const int units = B * hkv;
  // Units per CTA: as few CTAs as give every CTA the same number of units
  // (or one fewer), so that no SM is left with an extra unit at the end.
  const int sms = num_sms();
  const int per1 = (units + sms - 1) / sms, per2 = (units + 2 * sms - 1) / (2 * sms);
  if (G > 8) return launch_nt<2, 2>(mk, mv, mq, a, units, per1, st);
  // G <= 8: two CTAs of two groups per SM when each CTA then has an even
  // number of units (both of its groups equally loaded) and no SM more units
  // than with one CTA of four groups; the next launch's CTAs can then start
  // on an SM beside this one's last.  (Batch 64 over 8 KV heads: 8.7 -> 8.5
  // us in graph replay; batch 96, three units per CTA: 12.1 -> 12.6 us, so
  // not there.)
  if (per2 % 2 == 0 && 2 * per2 <= per1) return launch_nt<1, 2>(mk, mv, mq, a, units, per2, st);
  // At most one unit per SM: one unit per CTA of one group, whose ring holds
  // all five of the unit's chunks, so none waits for another to be read
  // (batch 16 over 8 KV heads: 4.09 -> 4.02 us).
  if (per1 == 1) return launch_nt<1, 1>(mk, mv, mq, a, units, 1, st);
  return launch_nt<1, 4>(mk, mv, mq, a, units, per1, st);
}

}  // namespace kvr
