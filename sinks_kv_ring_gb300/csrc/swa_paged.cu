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
// Layout of the work: one item per (sequence, KV head); one persistent CTA
// per SM takes items round-robin.  An item's window is at most nine 16-key
// subtiles (the window starts on any key; subtiles start on 16-key
// boundaries, so a 16-multiple block size never splits one).  Four producer
// warps stream the CTA's items through two stage sets, each holding a whole
// window: per item the G query rows and the RoPE table row (bulk copies) on
// one mbarrier, each subtile's K and V (one TMA box of all parts x 16 rows
// each) on a mbarrier of its own; the producers share the subtiles, as one
// warp alone issues the boxes too slowly.  Two groups of four consumer warps
// take alternate items (group g uses set g), so one group's chain of
// dependent steps runs while the other's does and while the producers fill
// the sets; in a group, warp w takes subtiles w, w + 4, w + 8.  A set goes
// back to the producers when its group's warps are done reading it.
//
// The products run transposed, keys as the MMA rows: S^T[16 keys x 8 heads] =
// K Q^T (m16n8k16, the group's heads as the 8 columns) and O^T[128 x 8] +=
// V^T P^T, P^T moved into the B-fragment layout by movmatrix.  A group of 8
// heads fills the 8 columns; the query-rows formulation would leave half of
// 16 MMA rows empty, so this takes half the tensor-core work per key.  A
// group's warps then merge their (m, l, O) per head in a shared-memory area
// of the group's own (not over the stages, which already hold the next item).
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
constexpr int SP_CWARPS = 8;                     // consumer warps
constexpr int SP_CTHREADS = SP_CWARPS * 32;
constexpr int SP_PWARPS = 4;                     // producer warps
constexpr int SP_THREADS = SP_CTHREADS + SP_PWARPS * 32;
constexpr int SP_SUBS = WIN / 16 + 1;            // 9 subtiles cover any window
constexpr int SP_SUB_K = 16 * DQK * 2;           // 6144 B: [16][3 parts][128 B]
constexpr int SP_SUB_V = 16 * DV * 2;            // 4096 B: [16][2 parts][128 B]
constexpr int SP_STAGE = SP_SUB_K + SP_SUB_V;
constexpr int SP_SET = SP_SUBS * SP_STAGE;
constexpr int SP_NB = 16;  // block ids of one window (blocks of >= 16 keys)
static_assert((WIN + 15 + 15) / 16 + 1 <= SP_NB, "block ids of one window");
constexpr int SP_OSTRIDE = DV + 4;  // merge rows: the 8 x 4 lanes of a stash store hit 32 banks
// shared memory from a 1024-byte aligned base (the TMA boxes' 128-byte
// swizzle wants it): two stage sets, the merge area (per warp and head: (m,
// l), O row, factor), two query tiles [8][192] (plain rows), two table rows,
// two sets of block ids, two item records, the barriers, the abort flag
constexpr int SP_OFF_MERGE = 2 * SP_SET;
constexpr int SP_GWARPS = SP_CWARPS / 2;  // consumer warps per group
constexpr int SP_GTHREADS = SP_GWARPS * 32;
constexpr int SP_MERGE_G = (SP_GWARPS * 8 * 2 + SP_GWARPS * 8 * SP_OSTRIDE + SP_GWARPS * 8) * 4;  // per group
constexpr int SP_MERGE = 2 * SP_MERGE_G;
constexpr int SP_OFF_Q = SP_OFF_MERGE + SP_MERGE;
constexpr int SP_QTILE = 8 * DQK * 2;
constexpr int SP_OFF_CS = SP_OFF_Q + 2 * SP_QTILE;
constexpr int SP_OFF_NB = SP_OFF_CS + 2 * 256;
constexpr int SP_OFF_REC = SP_OFF_NB + 2 * SP_NB * 4;
constexpr int SP_OFF_BAR = SP_OFF_REC + 2 * 16;
// barriers: full[set][j] (one per subtile), qbar[set], empty[set], and one
// nothing arrives on (the test hook's stall)
constexpr int SP_NBAR = 2 * SP_SUBS + 5;
constexpr int SP_OFF_ABORT = SP_OFF_BAR + 8 * SP_NBAR;
constexpr int SP_SMEM = SP_OFF_ABORT + 16 + 1024;
static_assert(SP_SMEM <= 232448, "one CTA per SM");
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
// the plain [8][192] query tile: lane l gets head l/4, dims 2(l%4)..
__device__ __forceinline__ void load_qt_frags(const uint8_t *sQ, int lane, uint32_t (&qf)[12][2]) {
  const uint32_t base = smem_u32(sQ) + (lane & 7) * (DQK * 2);
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


__global__ void __launch_bounds__(SP_THREADS, 1)
    swa_paged_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                     const uint16_t *__restrict__ q, const int64_t *__restrict__ pos,
                     const int32_t *__restrict__ seq, int B, int hq, int G, KvView pool,
                     const float *__restrict__ table, int64_t max_pos, float scale_log2, long long max_ctx,
                     unsigned *status, const float *__restrict__ sinks, uint16_t *__restrict__ out,
                     unsigned long long stall_ns) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + (((smem_u32(smem_raw) + 1023u) & ~1023u) - smem_u32(smem_raw));
  const uint32_t sBar = smem_u32(smem + SP_OFF_BAR);
  const uint32_t qbar0 = sBar + 8 * (2 * SP_SUBS), empty0 = qbar0 + 16;  // qbar[set], empty[set]: + 8 * set
  const uint32_t stallBar = empty0 + 16;
  SpRec *rec = reinterpret_cast<SpRec *>(smem + SP_OFF_REC);
  int32_t *sNB = reinterpret_cast<int32_t *>(smem + SP_OFF_NB);
  volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + SP_OFF_ABORT);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hkv = pool.hkv, bsz = pool.block_size;
  const long long nitems = (long long)B * hkv;
  auto full_bar = [&](int set, int j) -> uint32_t { return sBar + 8 * (set * SP_SUBS + j); };

  if (tid == 0) {
    for (int j = 0; j < 2 * SP_SUBS; ++j) tc::mbar_init(sBar + 8 * j, 1);
    for (int set = 0; set < 2; ++set) {
      tc::mbar_init(qbar0 + 8 * set, 1);
      tc::mbar_init(empty0 + 8 * set, SP_GWARPS);
    }
    tc::mbar_init(stallBar, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  // rows G..7 of both query tiles stay zero (the copies write rows 0..G-1)
  for (int e = tid; e < 2 * SP_QTILE / 16; e += SP_THREADS)
    *reinterpret_cast<uint4 *>(smem + SP_OFF_Q + 16 * e) = make_uint4(0, 0, 0, 0);
  tc::fence_proxy_async_smem();  // the zeroing before the bulk copies into the same tiles
  // launched as a programmatic dependent (launch_pdl): the set-up above
  // overlaps the end of the kernel before it; nothing global before pdl_wait
  pdl_wait();
  __syncthreads();
  pdl_trigger();

  if (warp >= SP_CWARPS) {
    // ---------------------------------------------------------- producers
    // producer warp pw issues subtiles j = pw, pw + 4, ... of every item;
    // warp 0 of them also the item record, block ids and query copies
    const int pw = warp - SP_CWARPS;
    if (pw == 0 && lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(&kmap) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(&vmap) : "memory");
    }
    // an item's metadata is loaded one item ahead: its position and sequence
    // id at the top of the previous iteration, its block ids (lane i: the
    // window's i-th block) at that iteration's end, so both are in when the
    // set frees up
    long long p_n = 0;
    int s_n = 0, blk_n = -1;
    auto load_ps = [&](long long wn) {
      if (wn < nitems) {
        p_n = pos[wn / hkv];
        s_n = seq[wn / hkv];
      }
    };
    auto load_ids = [&]() {
      blk_n = -1;
      if (p_n >= 0 && p_n < max_pos && p_n + 1 <= max_ctx && s_n >= 0 && s_n < pool.num_seqs) {
        const long long b0n = (max(0LL, p_n - WIN + 1) & ~15LL) / bsz;
        if (lane < p_n / bsz - b0n + 1) blk_n = pool.block_table[(long long)s_n * pool.max_blocks + b0n + lane];
      }
    };
    load_ps(blockIdx.x);
    load_ids();
    int k = 0;  // items issued
    for (long long w = blockIdx.x; w < nitems; w += gridDim.x, ++k) {
      const int set = k & 1;
      const long long p = p_n;
      const int s = s_n, blk_l = blk_n;
      load_ps(w + gridDim.x);
      // The set is free once every consumer warp is done with item k - 2.
      // The producer warps then agree to go on (or all stop); the barrier
      // also puts every producer's arrivals for earlier items before warp
      // 0's query-barrier arrival for this one, so a consumer that has seen
      // the latter never meets a subtile barrier still in an older phase.
      bool ok = true;
      if (k >= 2) ok = __all_sync(0xffffffffu, tc::mbar_wait(empty0 + 8 * set, ((k >> 1) - 1) & 1u, abort_flag));
      if (!tc::named_bar_and(9, SP_PWARPS * 32, ok)) break;
      const int b = (int)(w / hkv), kv = (int)(w % hkv);
      const unsigned bad = (p < 0 || p >= max_pos || p + 1 > max_ctx ? ST_BAD_POS : 0u) |
                           (s < 0 || s >= pool.num_seqs ? ST_BAD_SEQ : 0u);
      int nsub = 0;
      long long key_lo = 0, b0 = 0;
      if (!bad) {
        key_lo = max(0LL, p - WIN + 1) & ~15LL;
        nsub = (int)((p + 1 - key_lo + 15) / 16);
        b0 = key_lo / bsz;
        if (pw == 0 && lane < p / bsz - b0 + 1) sNB[set * SP_NB + lane] = blk_l;
      }
      if (pw == 0) {
        if (lane == 0) {
          rec[set].p = p;
          rec[set].s = s;
          rec[set].pad = (int)bad;
        }
        __syncwarp();  // the record and block ids before the barrier's arrival
        const uint32_t qb = qbar0 + 8 * set;
        if (bad) {
          if (lane == 0) tc::mbar_arrive(qb);
        } else {
          tc::mbar_expect_tx_elect(qb, G * DQK * 2 + 256);
          tc::bulk_load_elect(smem_u32(smem + SP_OFF_Q + set * SP_QTILE),
                              q + ((long long)b * hq + (long long)kv * G) * DQK, G * DQK * 2, qb);
          tc::bulk_load_elect(smem_u32(smem + SP_OFF_CS + set * 256), table + p * 64, 256, qb);
        }
      }
      // every subtile barrier of the set completes once per item (no load:
      // a plain arrival), so its phase count is the set's item count
      for (int j = pw; j < SP_SUBS; j += SP_PWARPS) {
        const uint32_t fb = full_bar(set, j);
        const long long key0 = key_lo + 16LL * j;
        bool load = false;
        int hrow = 0;
        if (j < nsub) {
          const int blk = __shfl_sync(0xffffffffu, blk_l, (int)(key0 / bsz - b0));
          if (blk >= 0 && blk < pool.num_blocks) {
            load = true;
            hrow = (int)(((long long)blk * hkv + kv) * bsz + key0 % bsz);
          } else if (lane == 0) {
            flag(status, ST_BAD_BLOCK);
          }
        }
        const uint32_t dst = smem_u32(smem + set * SP_SET + j * SP_STAGE);
        if (load) {
          tc::mbar_expect_tx_elect(fb, SP_STAGE);
          tc::tma_load_3d_elect(dst, &kmap, 0, 0, hrow, fb);
          tc::tma_load_3d_elect(dst + SP_SUB_K, &vmap, 0, 0, hrow, fb);
        } else if (lane == 0) {
          tc::mbar_arrive(fb);
        }
      }
      load_ids();
    }
    // before leaving, wait (bounded, whatever the abort flag says) for the
    // loads of the last item issued into each set
    uint32_t never = 0;
    for (int set = 0; set < 2; ++set) {
      const int n = (k + 1 - set) / 2;  // items issued into this set
      if (n == 0) continue;
      const uint32_t par = (uint32_t)(n - 1) & 1u;
      if (pw == 0) tc::mbar_wait(qbar0 + 8 * set, par, &never);
      for (int j = pw; j < SP_SUBS; j += SP_PWARPS) tc::mbar_wait(full_bar(set, j), par, &never);
    }
    if (*abort_flag && lane == 0) flag(status, SP_ST_TIMEOUT);
    return;
  }
  // ------------------------------------------------------------ consumers
  // group gr (warps 4gr..4gr+3) takes items k = gr, gr + 2, ... from set gr
  const int g = lane >> 2, t = lane & 3;
  const int gr = warp / SP_GWARPS, gw = warp % SP_GWARPS, ltid = tid % SP_GTHREADS, set = gr;
  const int bar0 = 1 + 4 * gr;  // the group's named barriers bar0 .. bar0 + 3
  float *mml = reinterpret_cast<float *>(smem + SP_OFF_MERGE + gr * SP_MERGE_G);  // [4 warps][8 heads][2]
  float *mo = mml + SP_GWARPS * 16;                                               // [4][8][SP_OSTRIDE]
  float *fac = mo + SP_GWARPS * 8 * SP_OSTRIDE;                                   // [4][8]
  for (long long w = blockIdx.x + (long long)gr * gridDim.x, k = gr; w < nitems; w += 2LL * gridDim.x, k += 2) {
    const uint32_t par = (uint32_t)(k >> 1) & 1u;
    const bool got_q = __all_sync(0xffffffffu, tc::mbar_wait(qbar0 + 8 * set, par, abort_flag));
    // the group's warps: the item's record is in and the previous item's
    // merge area is free; a wait that gave up stops them here
    if (!tc::named_bar_and(bar0, SP_GTHREADS, got_q && *abort_flag == 0)) break;
    // test hook (stall_ns != 0): group 0 waits on a barrier nothing completes,
    // with the item's loads in flight; its limit sets the abort flag
    if (stall_ns && k == 0) tc::mbar_wait(stallBar, 0, abort_flag, stall_ns);
    const int b = (int)(w / hkv), kv = (int)(w % hkv);
    const long long p = rec[set].p;
    const unsigned bad = (unsigned)rec[set].pad;
    if (bad) {  // a bad position or sequence id: zero rows, flagged once per sequence
      if (kv == 0 && ltid == 0) flag(status, bad);
      uint16_t *o = out + ((long long)b * hq + (long long)kv * G) * DV;
      for (int e = ltid; e < G * DV; e += SP_GTHREADS) o[e] = 0;
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(empty0 + 8 * set);
      continue;
    }
    // keys key_min..p; subtiles from key_lo (16-aligned), rows outside masked
    const long long key_min = max(0LL, p - WIN + 1);
    const long long key_lo = key_min & ~15LL, key_hi = p + 1, b0 = key_lo / bsz;
    const int nsub = (int)((key_hi - key_lo + 15) / 16);
    uint32_t qf[12][2];
    load_qt_frags(smem + SP_OFF_Q + set * SP_QTILE, lane, qf);
    rope_qt_frags(qf, reinterpret_cast<const float *>(smem + SP_OFF_CS + set * 256), lane);
    const int32_t *nb = sNB + set * SP_NB;

    // per thread: O^T[dims 16m + g (+8)][heads 2t, 2t+1]; (m, l) of heads 2t, 2t+1
    float O[8][4];
#pragma unroll
    for (int m = 0; m < 8; ++m) O[m][0] = O[m][1] = O[m][2] = O[m][3] = 0.f;
    float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;
    for (int j = gw; j < nsub; j += SP_GWARPS) {
      const long long key0 = key_lo + 16LL * j;
      const int blk = nb[key0 / bsz - b0];
      const bool blk_ok = blk >= 0 && blk < pool.num_blocks;
      const bool got = __all_sync(0xffffffffu, tc::mbar_wait(full_bar(set, j), par, abort_flag));
      if (!got) continue;  // gave up: the subtile counts as masked, and the CTA stops at the next item
      uint8_t *st = smem + set * SP_SET + j * SP_STAGE;
      // rows outside the window (or of a bad block) hold other keys' values:
      // zero them, as their zero weights must not meet a non-finite value
      if (!blk_ok || key0 < key_min || key0 + 16 > key_hi) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int c = lane + 32 * u, r = c >> 4, ch = c & 15;
          const long long key = key0 + r;
          if (!(blk_ok && key < key_hi && key >= key_min))
            *reinterpret_cast<uint4 *>(st + SP_SUB_K + swrow<2>(r, ch)) = make_uint4(0, 0, 0, 0);
        }
      }
      __syncwarp();
      float sc[4];  // S^T: keys g, g + 8 (rows) x heads 2t, 2t + 1 (columns)
      qk_t(qf, smem_u32(st), lane, sc);
      const long long ka = key0 + g, kb = key0 + g + 8;
      const bool va = blk_ok && ka >= key_min && ka < key_hi, vb = blk_ok && kb >= key_min && kb < key_hi;
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
      for (int m = 0; m < 8; ++m) {
        O[m][0] *= c0;
        O[m][1] *= c1;
        O[m][2] *= c0;
        O[m][3] *= c1;
      }
      // P^T as B fragments: each 8x8 block [keys][heads] transposed in registers
      const uint32_t pb0 = movmatrix_t(pack_bf16(p0, p1)), pb1 = movmatrix_t(pack_bf16(p2, p3));
      pv_t(smem_u32(st) + SP_SUB_K, lane, pb0, pb1, O);
      __syncwarp();
    }
    // this warp is done with the set (stages, query tile): hand it back; its
    // generic writes there (zeroed rows) come before the next TMA writes
    // into it
    tc::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(empty0 + 8 * set);

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
    for (int m = 0; m < 8; ++m) {
      mw[(2 * t) * SP_OSTRIDE + 16 * m + g] = O[m][0];
      mw[(2 * t + 1) * SP_OSTRIDE + 16 * m + g] = O[m][1];
      mw[(2 * t) * SP_OSTRIDE + 16 * m + g + 8] = O[m][2];
      mw[(2 * t + 1) * SP_OSTRIDE + 16 * m + g + 8] = O[m][3];
    }
    tc::named_bar_sync(bar0 + 2, SP_GTHREADS);
    // per head (threads 0..G-1): maximum over the warps and the sink, each
    // warp's factor with the normalisation folded in (the sink joins the
    // denominator only)
    if (ltid < G) {
      const int hh = ltid;
      const float sl = sinks[kv * G + hh] * LOG2E;
      float M = sl;
#pragma unroll
      for (int ww = 0; ww < SP_GWARPS; ++ww) M = fmaxf(M, mml[(ww * 8 + hh) * 2]);
      float f[SP_GWARPS], L = ex2(sl - M);
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
  cudaError_t e = ensure_smem_limit(13, (const void *)swa_paged_kernel, SP_SMEM);
  if (e != cudaSuccess) return e;
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
  long long grid = (long long)num_sms();
  if (grid > items) grid = items;
  return launch_pdl(swa_paged_kernel, dim3((unsigned)grid), dim3(SP_THREADS), (size_t)SP_SMEM, st, km, vm, q, pos, seq, B,
                    hq, G, pool, table, max_pos, softmax_scale * LOG2E, max_ctx, status, sinks, out, take_stall());
}

}  // namespace kvr
