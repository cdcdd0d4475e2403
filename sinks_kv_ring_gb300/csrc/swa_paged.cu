// swa_paged.cu -- windowed decode over a paged pool for GQA groups of up to
// eight q heads (the windowed layers' 64 q / 8 KV heads): one new token per
// sequence attends over keys p-127..p, with a per-head sink.
//
// colibri "MiMo-V2.6 (Xiaomi)", "What the engine implements": the sink joins
// the softmax denominator and nothing else.  gaudi-cookbook "MiMo-V2.6-Flash
// on Gaudi 2", "What was built": the window is exactly the last 128
// positions; "Windowed KV groups" and Xiaomi "Full-Pipeline Inference
// Optimization", section 2.1: the windowed layer's cache kept in pages.
// Decode is memory-bound (Xiaomi section 1.2).
//
// Layout of the work: one item per (sequence, KV head); persistent CTAs,
// two per SM, each of one group of four consumer warps, take items
// round-robin.  An item's window is at most nine 16-key
// subtiles (the window starts on any key; subtiles start on 16-key
// boundaries, so a 16-multiple block size never splits one).  Each group
// streams the subtiles of its items, in order, through a ring of eight
// places (one subtile's K and V, one TMA box of all parts x 16 rows each, on
// a barrier of the place's own): a place goes back to its producer as soon
// as the warp that read it is done, so the next subtiles, of this item or
// the next, are already loading while the group computes.  Two producer
// warps fill the ring's places of one parity each; one of them
// also loads each item's G query rows and RoPE table row (bulk copies) into
// one of two item slots.  In a group, warp w takes subtiles w, w + 4, w + 8
// of each item.  (An earlier design held a whole window per group, two
// groups per CTA, and gave it back only when the group was done with it:
// 13.8 us at batch 64 against 12.05 us now.)  The kernel is written for
// NGR groups per CTA; one is what runs.
//
// The products run transposed, keys as the MMA rows: S^T[16 keys x 8 heads] =
// K Q^T (m16n8k16, the group's heads as the 8 columns) and O^T[128 x 8] +=
// V^T P^T, P^T moved into the B-fragment layout by movmatrix.  A group of 8
// heads fills the 8 columns; the query-rows formulation would leave half of
// 16 MMA rows empty, so this takes half the tensor-core work per key.  A
// group's warps then merge their (m, l, O) per head in a shared-memory area
// of the group's own (not over the ring, which already holds the next subtiles).
//
// Every wait on an mbarrier is bounded: a wait that gives up sets the CTA's
// abort flag and KVR_DEV_TIMEOUT, the consumers stop together at their next
// item, and the producer waits (bounded) for its loads still in flight.
#include <cuda.h>

#include "launch.h"
#include "tc_ptx.cuh"
#include "warp_attn.cuh"

namespace kvr {
namespace {

constexpr unsigned SP_ST_TIMEOUT = 8u;  // KVR_DEV_TIMEOUT
constexpr int SP_GWARPS = 4;                     // consumer warps per group
constexpr int SP_GTHREADS = SP_GWARPS * 32;
constexpr int SP_SUB_K = 16 * DQK * 2;           // 6144 B: [16][3 parts][128 B]
constexpr int SP_SUB_V = 16 * DV * 2;            // 4096 B: [16][2 parts][128 B]
constexpr int SP_STAGE = SP_SUB_K + SP_SUB_V;    // one subtile's place
constexpr int SP_NP = 8;                         // places in a group's ring
constexpr int SP_RING = SP_NP * SP_STAGE;
constexpr int SP_NB = 16;  // block ids of one window (blocks of >= 16 keys)
static_assert((WIN + 15 + 15) / 16 + 1 <= SP_NB, "block ids of one window");
constexpr int SP_OSTRIDE = DV + 4;  // merge rows: the 8 x 4 lanes of a stash store hit 32 banks
constexpr int SP_MERGE_G = (SP_GWARPS * 8 * 2 + SP_GWARPS * 8 * SP_OSTRIDE + SP_GWARPS * 8) * 4;  // per group
// query tile rows padded to 400 bytes: the eight rows an ldmatrix reads then
// start in eight different 16-byte bank groups (384-byte rows would all start
// in the same one)
constexpr int SP_QROW = DQK * 2 + 16;
constexpr int SP_QTILE = 8 * SP_QROW;
static_assert(SP_STAGE % 1024 == 0, "places start on 1024-byte boundaries");

// Shape of a CTA of NGR groups (each: four consumer warps, two producer
// warps).  Shared memory from a 1024-byte aligned base (the TMA boxes'
// 128-byte swizzle wants it): the groups' rings, their merge areas (per
// warp and head: (m, l), O row, factor), then per group and item slot (two
// per group) the query tile [8][192] (rows padded to 400 bytes), the table row, the
// window's block ids and the item record; the barriers -- full[group][place],
// empty[group][place], qfull[group][slot], qempty[group][slot], one nothing
// arrives on (the test hook's stall) -- and the abort flag.
template <int NGR>
struct SpL {
  static constexpr int CWARPS = SP_GWARPS * NGR, PWARPS = 2 * NGR;
  static constexpr int THREADS = (CWARPS + PWARPS) * 32;
  static constexpr int CTAS = NGR == 1 ? 2 : 1;  // resident CTAs per SM
  static constexpr int OFF_MERGE = NGR * SP_RING;
  static constexpr int OFF_Q = OFF_MERGE + NGR * SP_MERGE_G;
  static constexpr int OFF_CS = OFF_Q + 2 * NGR * SP_QTILE;
  static constexpr int OFF_NB = OFF_CS + 2 * NGR * 256;
  static constexpr int OFF_REC = OFF_NB + 2 * NGR * SP_NB * 4;
  static constexpr int OFF_BAR = OFF_REC + 2 * NGR * 16;
  static constexpr int B_EMPTY = NGR * SP_NP, B_QFULL = 2 * NGR * SP_NP, B_QEMPTY = B_QFULL + 2 * NGR,
                       B_STALL = B_QEMPTY + 2 * NGR, NBAR = B_STALL + 1;
  static constexpr int OFF_ABORT = OFF_BAR + 8 * NBAR;
  static constexpr int SMEM = OFF_ABORT + 16 + 1024;
  static_assert(CTAS * (SMEM + 1024) <= 233472, "shared memory per SM");
};
// item record written by the producer: position, then the sequence id (-1: bad item)
struct SpRec {
  long long p;
  int s;
  int pad;
};

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// B fragments of Q^T (16 dims x 8 heads per k-step) for the 12 k-steps, from
// the [8][192] query tile (rows SP_QROW bytes apart): lane l gets head l/4, dims 2(l%4)..
__device__ __forceinline__ void load_qt_frags(const uint8_t *sQ, int lane, uint32_t (&qf)[12][2]) {
  const uint32_t base = smem_u32(sQ) + (lane & 7) * SP_QROW;
#pragma unroll
  for (int kk = 0; kk < 12; kk += 2)
    ldsm_x4(base + (2 * kk + (lane >> 3)) * 16, qf[kk][0], qf[kk][1], qf[kk + 1][0], qf[kk + 1][1]);
}

// Rotate-half RoPE of dims 0..63 on the Q^T B fragments in registers: dims d
// and d + 32 (d < 32) sit in k-steps kk and kk + 2 of the same lane; cs is the
// table row ([32][2] fp32, (cos, sin) per frequency); the results are rounded
// to bf16, as a rotated query tile would be.
__device__ __forceinline__ void rope_qt_frags(uint32_t (&qf)[12][2], const float *cs, int lane) {
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

// S^T[16 keys x 8 heads] = K Q^T for a TMA-written K subtile ([16][3][128 B]).
// Two accumulation chains (even and odd k-steps) halve the dependent MMAs.
__device__ __forceinline__ void qk_t(const uint32_t (&qf)[12][2], uint32_t kbase, int lane, float (&s)[4]) {
  float e[4] = {0.f, 0.f, 0.f, 0.f}, o[4] = {0.f, 0.f, 0.f, 0.f};
  const int row = lane & 15, csel = lane >> 4;
#pragma unroll
  for (int kk = 0; kk < 12; ++kk) {
    uint32_t a[4];
    ldsm_x4(kbase + swrow<3>(row, 2 * kk + csel), a[0], a[1], a[2], a[3]);
    mma_bf16(kk & 1 ? o : e, a, qf[kk][0], qf[kk][1]);
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) s[r] = e[r] + o[r];
}

// O^T[128 x 8] += V^T P^T for a TMA-written V subtile ([16][2][128 B]); pb0 /
// pb1 are P^T's B fragments for keys 0..7 / 8..15.
__device__ __forceinline__ void pv_t(uint32_t vbase, int lane, uint32_t pb0, uint32_t pb1, float (&O)[8][4]) {
  const int row = (lane & 7) + ((lane >> 4) << 3), csel = (lane >> 3) & 1;
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    uint32_t a[4];
    ldsm_x4_t(vbase + swrow<2>(row, 2 * m + csel), a[0], a[1], a[2], a[3]);
    mma_bf16(O[m], a, pb0, pb1);
  }
}


// The window of an item at position p: keys key_min .. p, read as nsub
// 16-key subtiles from key_lo (16-aligned), the first block b0 = key_lo / bsz.
struct SpWin {
  long long key_min, key_lo, b0;
  int nsub;
};
__device__ __forceinline__ SpWin sp_window(long long p, int bsz) {
  SpWin w;
  w.key_min = max(0LL, p - WIN + 1);
  w.key_lo = w.key_min & ~15LL;
  w.nsub = (int)((p + 1 - w.key_lo + 15) / 16);
  w.b0 = w.key_lo / bsz;
  return w;
}

// The window rows of item w (keys max(0, p - 127) rounded down to 16 .. p,
// block by block) into L2, by one warp (lane j: the window's j-th block),
// from a position, sequence id and block ids read before pdl_wait (see
// ld_early_s32: a stale value only wastes a prefetch); anything outside the
// pool is skipped.
__device__ __forceinline__ void prefetch_window_early(long long w, const int64_t *pos, const int32_t *seq,
                                                      const KvView &pool, int64_t max_pos, int lane) {
  const int hkv = pool.hkv, bsz = pool.block_size;
  const long long b = w / hkv;
  const int kv = (int)(w % hkv);
  const long long p = ld_early_s64(pos + b);
  const int s = ld_early_s32(seq + b);
  if (p < 0 || p >= max_pos || s < 0 || s >= pool.num_seqs) return;
  const long long key_lo = max(0LL, p - WIN + 1) & ~15LL, b0 = key_lo / bsz;
  if (lane > p / bsz - b0 || b0 + lane >= pool.max_blocks) return;
  const int blk = ld_early_s32(pool.block_table + (long long)s * pool.max_blocks + b0 + lane);
  if (blk < 0 || blk >= pool.num_blocks) return;
  const long long lo = max(key_lo, (b0 + lane) * bsz), hi = min(p, (b0 + lane + 1) * bsz - 1);
  const long long row = ((long long)blk * hkv + kv) * bsz + lo % bsz;
  prefetch_l2(pool.k + row * DQK, (uint32_t)(hi - lo + 1) * DQK * 2);
  prefetch_l2(pool.v + row * DV, (uint32_t)(hi - lo + 1) * DV * 2);
}

template <int NGR>
__global__ void __launch_bounds__(SpL<NGR>::THREADS, SpL<NGR>::CTAS)
    swa_paged_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                     const uint16_t *__restrict__ q, const int64_t *__restrict__ pos,
                     const int32_t *__restrict__ seq, int B, int hq, int G, KvView pool,
                     const float *__restrict__ table, int64_t max_pos, float scale_log2, long long max_ctx,
                     unsigned *status, const float *__restrict__ sinks, uint16_t *__restrict__ out,
                     unsigned long long stall_ns) {
  using L = SpL<NGR>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + (((smem_u32(smem_raw) + 1023u) & ~1023u) - smem_u32(smem_raw));
  const uint32_t sBar = smem_u32(smem + L::OFF_BAR);
  auto full_bar = [&](int gr, int pl) -> uint32_t { return sBar + 8 * (gr * SP_NP + pl); };
  auto empty_bar = [&](int gr, int pl) -> uint32_t { return sBar + 8 * (L::B_EMPTY + gr * SP_NP + pl); };
  auto qfull_bar = [&](int gr, int sl) -> uint32_t { return sBar + 8 * (L::B_QFULL + 2 * gr + sl); };
  auto qempty_bar = [&](int gr, int sl) -> uint32_t { return sBar + 8 * (L::B_QEMPTY + 2 * gr + sl); };
  const uint32_t stallBar = sBar + 8 * L::B_STALL;
  SpRec *rec = reinterpret_cast<SpRec *>(smem + L::OFF_REC);      // [group * 2 + slot]
  int32_t *sNB = reinterpret_cast<int32_t *>(smem + L::OFF_NB);   // [group * 2 + slot][SP_NB]
  volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + L::OFF_ABORT);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hkv = pool.hkv, bsz = pool.block_size;
  const long long nitems = (long long)B * hkv;
  const long long grid = gridDim.x;

  if (tid == 0) {
    for (int j = 0; j < 2 * NGR * SP_NP; ++j) tc::mbar_init(sBar + 8 * j, 1);
    for (int gr = 0; gr < NGR; ++gr)
      for (int sl = 0; sl < 2; ++sl) {
        tc::mbar_init(qfull_bar(gr, sl), 1);
        tc::mbar_init(qempty_bar(gr, sl), SP_GWARPS);
      }
    tc::mbar_init(stallBar, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  // rows G..7 of every query tile stay zero (the copies write rows 0..G-1)
  for (int e = tid; e < 2 * NGR * SP_QTILE / 16; e += L::THREADS)
    *reinterpret_cast<uint4 *>(smem + L::OFF_Q + 16 * e) = make_uint4(0, 0, 0, 0);
  tc::fence_proxy_async_smem();  // the zeroing before the bulk copies into the same tiles
  // launched as a programmatic dependent (launch_pdl): the set-up above
  // overlaps the end of the kernel before it; before pdl_wait nothing global
  // is touched but the early reads that choose the first item's window to
  // bring into L2 (by the first producer warp of each group), when no group
  // has more than two items (batch 64 over 8 KV heads: 12.1 -> 11.8 us; at
  // batch 256, seven items per group, it cost 2%)
  if (nitems <= 2LL * NGR * gridDim.x && warp >= L::CWARPS && ((warp - L::CWARPS) & 1) == 0) {
    const long long w = blockIdx.x + (long long)((warp - L::CWARPS) >> 1) * gridDim.x;
    if (w < nitems) prefetch_window_early(w, pos, seq, pool, max_pos, lane);
  }
  pdl_wait();
  __syncthreads();
  pdl_trigger();

  if (warp >= L::CWARPS) {
    // ---------------------------------------------------------- producers
    // Group gr's items are m = 0, 1, .. (item w = blockIdx.x + (gr + NGR m) *
    // grid); their subtiles form one stream, subtile j of item m being
    // number base_m + j, which goes to ring place (base_m + j) mod SP_NP.
    // Producer pw of the group fills the places of parity pw, so a place is
    // always filled by the same warp, its uses in order: each wait on a
    // place's empty barrier is for the phase right after the one this warp
    // saw last.  (Subtiles 0 and 8 of a nine-subtile window share a place:
    // a ring of nine, with the smaller two-round merge it needs, measured
    // slower.)  Producer 0 also writes each item's record and
    // block ids and loads its query rows and table row into the item's slot
    // (m mod 2), once the group is done with item m - 2.
    const int pq = warp - L::CWARPS, gr = pq >> 1, pw = pq & 1;
    if (pq == 0 && lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(&kmap) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(&vmap) : "memory");
    }
    uint8_t *ring = smem + gr * SP_RING;
    long long base = 0;
    constexpr int NPW = (SP_NP + 1) / 2;
    int lastu[NPW];  // last use issued of this warp's places pw, pw + 2, ..
#pragma unroll
    for (int k = 0; k < NPW; ++k) lastu[k] = -1;
    int m = 0;
    bool alive = true;
    for (long long w = blockIdx.x + gr * grid; w < nitems && alive; w += NGR * grid, ++m) {
      const int b = (int)(w / hkv), kv = (int)(w % hkv);
      const long long p = pos[b];
      const int s = seq[b];
      const unsigned bad = (p < 0 || p >= max_pos || p + 1 > max_ctx ? ST_BAD_POS : 0u) |
                           (s < 0 || s >= pool.num_seqs ? ST_BAD_SEQ : 0u);
      SpWin win{};
      int blk_l = -1;
      if (!bad) {
        win = sp_window(p, bsz);
        if (lane < p / bsz - win.b0 + 1) blk_l = pool.block_table[(long long)s * pool.max_blocks + win.b0 + lane];
      }
      const int sl = m & 1;
      if (pw == 0) {
        if (m >= 2 && !__all_sync(0xffffffffu, tc::mbar_wait(qempty_bar(gr, sl), ((m >> 1) - 1) & 1u, abort_flag)))
          break;
        if (!bad && lane < p / bsz - win.b0 + 1) sNB[(gr * 2 + sl) * SP_NB + lane] = blk_l;
        if (lane == 0) {
          rec[gr * 2 + sl].p = p;
          rec[gr * 2 + sl].s = s;
          rec[gr * 2 + sl].pad = (int)bad;
        }
        __syncwarp();  // the record and block ids before the barrier's arrival
        const uint32_t qb = qfull_bar(gr, sl);
        if (bad) {
          if (lane == 0) tc::mbar_arrive(qb);
        } else {
          tc::mbar_expect_tx_elect(qb, G * DQK * 2 + 256);
          __syncwarp();
          if (lane < G)  // one padded row per lane
            tc::bulk_load(smem_u32(smem + L::OFF_Q + (gr * 2 + sl) * SP_QTILE + lane * SP_QROW),
                          q + ((long long)b * hq + (long long)kv * G + lane) * DQK, DQK * 2, qb);
          tc::bulk_load_elect(smem_u32(smem + L::OFF_CS + (gr * 2 + sl) * 256), table + p * 64, 256, qb);
        }
      }
      for (int j = 0; j < win.nsub; ++j) {
        const long long su = base + j;
        const int pl = (int)(su % SP_NP);
        if ((pl & 1) != pw) continue;
        const int u = (int)(su / SP_NP);
        if (u >= 1 && !__all_sync(0xffffffffu, tc::mbar_wait(empty_bar(gr, pl), (uint32_t)(u - 1) & 1u, abort_flag))) {
          alive = false;
          break;
        }
        const long long key0 = win.key_lo + 16LL * j;
        const int blk = __shfl_sync(0xffffffffu, blk_l, (int)(key0 / bsz - win.b0));
        const uint32_t fb = full_bar(gr, pl);
        if (blk >= 0 && blk < pool.num_blocks) {
          const int hrow = (int)(((long long)blk * hkv + kv) * bsz + key0 % bsz);
          const uint32_t dst = smem_u32(ring + pl * SP_STAGE);
          tc::mbar_expect_tx_elect(fb, SP_STAGE);
          tc::tma_load_3d_elect(dst, &kmap, 0, 0, hrow, fb);
          tc::tma_load_3d_elect(dst + SP_SUB_K, &vmap, 0, 0, hrow, fb);
        } else if (lane == 0) {
          flag(status, ST_BAD_BLOCK);
          tc::mbar_arrive(fb);
        }
        lastu[pl >> 1] = u;
      }
      base += win.nsub;
    }
    // before leaving, wait (bounded, whatever the abort flag says) for the
    // last load this warp issued into each of its places, and producer 0 for
    // the last query rows
    uint32_t never = 0;
#pragma unroll
    for (int k = 0; k < NPW; ++k)
      if (2 * k + pw < SP_NP && lastu[k] >= 0) tc::mbar_wait(full_bar(gr, 2 * k + pw), (uint32_t)lastu[k] & 1u, &never);
    if (pw == 0 && m > 0) {
      const int ml = m - 1;  // (an item whose slot wait gave up issued nothing: m was not advanced past it)
      tc::mbar_wait(qfull_bar(gr, ml & 1), (uint32_t)(ml >> 1) & 1u, &never);
    }
    if (*abort_flag && lane == 0) flag(status, SP_ST_TIMEOUT);
    return;
  }
  // ------------------------------------------------------------ consumers
  // group gr (warps 4gr..4gr+3) takes its items m = 0, 1, .. from its ring
  // (see the producers); warp gw of it the item's subtiles j = gw, gw + 4, ..
  // Every use of a place is handed back by the one warp that read it.
  const int g = lane >> 2, t = lane & 3;
  const int gr = warp / SP_GWARPS, gw = warp % SP_GWARPS, ltid = tid % SP_GTHREADS;
  const int bar0 = 1 + 4 * gr;  // the group's named barriers bar0 .. bar0 + 3
  float *mml = reinterpret_cast<float *>(smem + L::OFF_MERGE + gr * SP_MERGE_G);  // [4 warps][8 heads][2]
  float *mo = mml + SP_GWARPS * 16;                                               // [4][8][SP_OSTRIDE]
  float *fac = mo + SP_GWARPS * 8 * SP_OSTRIDE;                                   // [4][8]
  uint8_t *ring = smem + gr * SP_RING;
  long long base = 0;
  int m = 0;
  for (long long w = blockIdx.x + gr * grid; w < nitems; w += NGR * grid, ++m) {
    const int sl = m & 1;
    const bool got_q = __all_sync(0xffffffffu, tc::mbar_wait(qfull_bar(gr, sl), (uint32_t)(m >> 1) & 1u, abort_flag));
    // the group's warps: the item's record is in and the previous item's
    // merge area is free; a wait that gave up stops them here
    if (!tc::named_bar_and(bar0, SP_GTHREADS, got_q && *abort_flag == 0)) break;
    // test hook (stall_ns != 0): group 0 waits on a barrier nothing completes,
    // with the item's loads in flight; its limit sets the abort flag
    if (stall_ns && m == 0) tc::mbar_wait(stallBar, 0, abort_flag, stall_ns);
    const int b = (int)(w / hkv), kv = (int)(w % hkv);
    const long long p = rec[gr * 2 + sl].p;
    const unsigned bad = (unsigned)rec[gr * 2 + sl].pad;
    if (bad) {  // a bad position or sequence id: zero rows, flagged once per sequence (no subtiles)
      if (kv == 0 && ltid == 0) flag(status, bad);
      uint16_t *o = out + ((long long)b * hq + (long long)kv * G) * DV;
      for (int e = ltid; e < G * DV; e += SP_GTHREADS) o[e] = 0;
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(qempty_bar(gr, sl));
      continue;
    }
    const SpWin win = sp_window(p, bsz);
    const long long key_hi = p + 1;
    uint32_t qf[12][2];
    load_qt_frags(smem + L::OFF_Q + (gr * 2 + sl) * SP_QTILE, lane, qf);
    rope_qt_frags(qf, reinterpret_cast<const float *>(smem + L::OFF_CS + (gr * 2 + sl) * 256), lane);
    const int32_t *nb = sNB + (gr * 2 + sl) * SP_NB;

    // per thread: O^T[dims 16m + g (+8)][heads 2t, 2t+1]; (m, l) of heads 2t, 2t+1
    float O[8][4];
#pragma unroll
    for (int mm = 0; mm < 8; ++mm) O[mm][0] = O[mm][1] = O[mm][2] = O[mm][3] = 0.f;
    float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;
    for (int j = gw; j < win.nsub; j += SP_GWARPS) {
      const long long su = base + j;
      const int pl = (int)(su % SP_NP);
      const long long key0 = win.key_lo + 16LL * j;
      const int blk = nb[key0 / bsz - win.b0];
      const bool blk_ok = blk >= 0 && blk < pool.num_blocks;
      const bool got = __all_sync(0xffffffffu, tc::mbar_wait(full_bar(gr, pl), (uint32_t)(su / SP_NP) & 1u, abort_flag));
      if (!got) continue;  // gave up: the subtile counts as masked (its place is not handed back), and the CTA stops
      uint8_t *st = ring + pl * SP_STAGE;
      // rows outside the window (or of a bad block) hold other keys' values:
      // zero them, as their zero weights must not meet a non-finite value
      if (!blk_ok || key0 < win.key_min || key0 + 16 > key_hi) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int c = lane + 32 * u, r = c >> 4, ch = c & 15;
          const long long key = key0 + r;
          if (!(blk_ok && key < key_hi && key >= win.key_min))
            *reinterpret_cast<uint4 *>(st + SP_SUB_K + swrow<2>(r, ch)) = make_uint4(0, 0, 0, 0);
        }
      }
      __syncwarp();
      float sc[4];  // S^T: keys g, g + 8 (rows) x heads 2t, 2t + 1 (columns)
      qk_t(qf, smem_u32(st), lane, sc);
      const long long ka = key0 + g, kb = key0 + g + 8;
      const bool va = blk_ok && ka >= win.key_min && ka < key_hi, vb = blk_ok && kb >= win.key_min && kb < key_hi;
      sc[0] = va ? sc[0] * scale_log2 : NEG_INF;
      sc[1] = va ? sc[1] * scale_log2 : NEG_INF;
      sc[2] = vb ? sc[2] * scale_log2 : NEG_INF;
      sc[3] = vb ? sc[3] * scale_log2 : NEG_INF;
      // online softmax per head over the 16 keys (the lanes with this t)
      float x0 = fmaxf(sc[0], sc[2]), x1 = fmaxf(sc[1], sc[3]);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, off));
        x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, off));
      }
      const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
      const float b0f = n0 == NEG_INF ? 0.f : n0, b1f = n1 == NEG_INF ? 0.f : n1;
      const float c0 = ex2(m0 - b0f), c1 = ex2(m1 - b1f);
      m0 = n0;
      m1 = n1;
      const float p0 = ex2(sc[0] - b0f), p1 = ex2(sc[1] - b1f), p2 = ex2(sc[2] - b0f), p3 = ex2(sc[3] - b1f);
      l0 = l0 * c0 + p0 + p2;
      l1 = l1 * c1 + p1 + p3;
#pragma unroll
      for (int mm = 0; mm < 8; ++mm) {
        O[mm][0] *= c0;
        O[mm][1] *= c1;
        O[mm][2] *= c0;
        O[mm][3] *= c1;
      }
      // P^T as B fragments: each 8x8 block [keys][heads] transposed in registers
      const uint32_t pb0 = movmatrix_t(pack_bf16(p0, p1)), pb1 = movmatrix_t(pack_bf16(p2, p3));
      pv_t(smem_u32(st) + SP_SUB_K, lane, pb0, pb1, O);
      // this warp is done with the place: hand it back; its generic writes
      // there (zeroed rows) come before the next TMA writes into it
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(empty_bar(gr, pl));
    }
    // done with the item's slot (record, block ids, query and table rows)
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(qempty_bar(gr, sl));
    base += win.nsub;

#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    if (g == 0) {
      mml[(gw * 8 + 2 * t) * 2] = m0;
      mml[(gw * 8 + 2 * t) * 2 + 1] = l0;
      mml[(gw * 8 + 2 * t + 1) * 2] = m1;
      mml[(gw * 8 + 2 * t + 1) * 2 + 1] = l1;
    }
    float *mw = mo + gw * 8 * SP_OSTRIDE;
#pragma unroll
    for (int mm = 0; mm < 8; ++mm) {
      mw[(2 * t) * SP_OSTRIDE + 16 * mm + g] = O[mm][0];
      mw[(2 * t + 1) * SP_OSTRIDE + 16 * mm + g] = O[mm][1];
      mw[(2 * t) * SP_OSTRIDE + 16 * mm + g + 8] = O[mm][2];
      mw[(2 * t + 1) * SP_OSTRIDE + 16 * mm + g + 8] = O[mm][3];
    }
    tc::named_bar_sync(bar0 + 2, SP_GTHREADS);
    // per head (threads 0..G-1): maximum over the warps and the sink, each
    // warp's factor with the normalisation folded in (the sink joins the
    // denominator only)
    if (ltid < G) {
      const int hh = ltid;
      const float sl2 = sinks[kv * G + hh] * LOG2E;
      float M = sl2;
#pragma unroll
      for (int ww = 0; ww < SP_GWARPS; ++ww) M = fmaxf(M, mml[(ww * 8 + hh) * 2]);
      float f[SP_GWARPS], L = ex2(sl2 - M);
#pragma unroll
      for (int ww = 0; ww < SP_GWARPS; ++ww) {
        const float mv = mml[(ww * 8 + hh) * 2];
        f[ww] = mv == NEG_INF ? 0.f : ex2(mv - M);
        L += mml[(ww * 8 + hh) * 2 + 1] * f[ww];
      }
      const float inv = 1.f / L;
#pragma unroll
      for (int ww = 0; ww < SP_GWARPS; ++ww) fac[ww * 8 + hh] = f[ww] * inv;
    }
    tc::named_bar_sync(bar0 + 3, SP_GTHREADS);
    for (int idx = ltid; idx < G * (DV / 4); idx += SP_GTHREADS) {
      const int hh = idx / (DV / 4), d4 = 4 * (idx % (DV / 4));
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int ww = 0; ww < SP_GWARPS; ++ww) {
        const float f = fac[ww * 8 + hh];
        const float4 x = *reinterpret_cast<const float4 *>(mo + (ww * 8 + hh) * SP_OSTRIDE + d4);
        acc.x += x.x * f;
        acc.y += x.y * f;
        acc.z += x.z * f;
        acc.w += x.w * f;
      }
      uint16_t *o = out + ((long long)b * hq + (long long)kv * G + hh) * DV + d4;
      *reinterpret_cast<uint2 *>(o) = make_uint2(pack_bf16(acc.x, acc.y), pack_bf16(acc.z, acc.w));
    }
  }
  if (*abort_flag && ltid == 0) flag(status, SP_ST_TIMEOUT);
}

}  // namespace

// Windowed decode over pages for G <= 8 q heads per KV head (see above).
cudaError_t launch_swa_paged(const uint16_t *q, const int64_t *pos, const int32_t *seq, int B, int hq,
                             const KvView &pool, const float *sinks, const float *table, int64_t max_pos,
                             float softmax_scale, uint16_t *out, unsigned *status, cudaStream_t st) {
  const int hkv = pool.hkv, G = hq / hkv;
  if (G < 1 || G > 8) return cudaErrorInvalidValue;
  // positions past the pool are flagged as bad positions
  const long long cap = (long long)pool.max_blocks * pool.block_size;
  const long long max_ctx = cap < max_pos ? cap : max_pos;
  // the pool as rows of 64-element parts; boxes of all parts x 16 rows
  const long long rows = (long long)pool.num_blocks * hkv * pool.block_size;
  CUtensorMap km, vm;
  if (rows > 0x7fffffffLL || !make_tma_map_rows3d(&km, pool.k, rows, DQK, 16) ||
      !make_tma_map_rows3d(&vm, pool.v, rows, DV, 16))
    return cudaErrorInvalidValue;
  const long long items = (long long)B * hkv;
  // Two CTAs of one group per SM (a CTA of two groups, one per SM, measured
  // slower at every batch: 12.4 against 12.05 us at batch 64, 38.0 against
  // 35.7 us at batch 256; the next launch's CTAs also start beside this
  // one's last).
  using L = SpL<1>;
  cudaError_t e = ensure_smem_limit(13, (const void *)swa_paged_kernel<1>, L::SMEM, true);
  if (e != cudaSuccess) return e;
  long long grid = 2LL * num_sms();
  if (grid > items) grid = items;
  return launch_pdl(swa_paged_kernel<1>, dim3((unsigned)grid), dim3(L::THREADS), (size_t)L::SMEM, st, km, vm, q, pos,
                    seq, B, hq, G, pool, table, max_pos, softmax_scale * LOG2E, max_ctx, status, sinks, out,
                    take_stall());
}

}  // namespace kvr
