// swa_band.cu -- chunked prefill of a windowed layer on the tensor cores, one
// 144-key band per tile of query rows, persistent CTAs.
//
// colibri "MiMo-V2.6 (Xiaomi)", "What the engine implements": the sink joins
// the softmax denominator and nothing else; gaudi-cookbook "MiMo-V2.6-Flash on
// Gaudi 2", "What was built": the window is exactly the last 128 positions, so
// row i of a chunk at P0 (position P0 + i) attends positions P0+i-127..P0+i;
// colibri "System One mode and prompt reuse": a position before the chunk
// sits in ring slot p mod 128, whose tag records the position it holds.
//
// A work item is 128 query rows of one KV head's GQA group: np = 128 / G
// consecutive chunk rows r0 .. r0+np-1 (np <= 16) times the G heads, row
// d * G + g.  Every key such a row can attend lies in chunk rows r0-128 ..
// r0+15, one band of 144 keys, so an item is one S = Q K^T (N = 144) and one
// O = P V, and its softmax is a single pass with no rescaling: the window
// and the sink are all there.  In band column t (chunk row r0-128+t) row d
// attends columns d+1 .. d+128.  The RoPE warps fill a band's rows before
// the chunk: the ring row where its slot holds the position, zeros otherwise
// (for one chunk the box brought zeros there already, a negative coordinate;
// in a batch those rows of the box belong to the previous chunk).
//
// A batch of chunks (VARLEN): the long chunks' items come from the device
// plan (tiles of 128 query rows).  The query producer writes each item's
// record (chunk rows, length, position, ring, KV head, tile, ring-slot bits)
// into one of eight shared-memory slots before loading its query tile, and
// every other role reads it from there.  A chunk's partial last tile is
// stored row by row, as its box would reach into the next chunk's rows.
//
// One CTA per SM, 480 threads:
//   warps 0-7   softmax of item i, then the epilogue of item i-1; warp w
//               takes TMEM lanes 32 (w % 4) .. (one tile row each) and half
//               w / 4 of the band's columns and of O's columns
//   warps 8-11  RoPE of each query tile in shared memory; the ring rows of
//               the items that reach before the chunk
//   warp  12    TMEM owner and MMA issuer (converged; elect.sync issues)
//   warp  13    TMA producer of the bands, warp 14 of the query tiles
//               (converged; elect.sync issues)
// Shared memory: two query tiles (3 x 16 KB each, 128-byte swizzled,
// K-major), the band's K (3 x 18 KB, K-major) and V (2 x 18 KB, MN-major),
// one output tile (2 x 16 KB) that leaves as two TMA boxes.  The producers
// issue each load as soon as its buffer is free: the query tile of item
// i+2 once S(i) is done, the band's K of item i+1 once S(i) is done, its V
// once P V(i) is done; the band producer also tells the RoPE warps when a
// band that reaches before its chunk has landed.
// TMEM (512 columns): S0 at 0, S1 at 160 (144 fp32 columns each; the bf16
// probabilities P overwrite the first 72 and feed P V from TMEM), O at 320.
#include <cuda.h>

#include "launch.h"
#include "tc_ptx.cuh"

namespace kvr {
namespace {

using namespace tc;

constexpr int SB_THREADS = 480;
constexpr int SB_WARP_ROPE = 8, SB_WARP_MMA = 12, SB_WARP_TMA = 13, SB_WARP_TMAQ = 14;
constexpr int SB_N = 144;                          // keys of a band
constexpr int SB_QPART = 128 * 128;                // 128 rows x 64 dims
constexpr int SB_QTILE = 3 * SB_QPART;
constexpr int SB_KPART = SB_N * 128;               // 144 keys x 64 dims
constexpr int SB_OFF_K = 2 * SB_QTILE;
constexpr int SB_OFF_V = SB_OFF_K + 3 * SB_KPART;
constexpr int SB_OFF_O = SB_OFF_V + 2 * SB_KPART;
constexpr int SB_OFF_BAR = SB_OFF_O + 2 * SB_QPART;
constexpr int SB_OFF_RED = SB_OFF_BAR + 256;       // half-row maxima [2][128], sums [2][2][128] (fp32)
constexpr int SB_OFF_INFO = SB_OFF_RED + 768 * 4;  // records of the work items in flight [8] (SbInfo)
constexpr int SB_NINFO = 8;
constexpr int SB_SMEM = SB_OFF_INFO + SB_NINFO * 64 + 1024;  // + alignment slack
static_assert(SB_OFF_K % 1024 == 0 && SB_KPART % 1024 == 0 && SB_OFF_V % 1024 == 0 && SB_OFF_O % 1024 == 0,
              "swizzled tiles start on 1024-byte boundaries");
static_assert(SB_SMEM <= 227 * 1024, "one CTA per SM");
constexpr uint32_t SB_COL_S1 = 160, SB_COL_O = 320;
constexpr unsigned ST_TIMEOUT = 8u;

// barrier area (byte offsets): [2] = one per query tile / S buffer
constexpr int SBB_QFULL = 0;    // [2] query tile landed (TMA bytes)
constexpr int SBB_QROPE = 16;   // [2] query tile rotated (128 arrivals)
constexpr int SBB_QFREE = 32;   // [2] S = Q K^T of the tile done
constexpr int SBB_SFULL = 48;   // [2] S in TMEM
constexpr int SBB_PREADY = 64;  // [2] P in TMEM (256 arrivals: the eight softmax warps)
constexpr int SBB_KFULL = 80;   // band K landed
constexpr int SBB_VFULL = 88;   // band V landed
constexpr int SBB_KFREE = 96;   // band K read by S = Q K^T
constexpr int SBB_VFREE = 104;  // band V read by P V
constexpr int SBB_KPATCH = 112; // ring rows copied into K (128 arrivals)
constexpr int SBB_VPATCH = 120; // ring rows copied into V (128 arrivals)
constexpr int SBB_OFULL = 128;  // O in TMEM
constexpr int SBB_OFREE = 136;  // O read out of TMEM (256 arrivals)
constexpr int SBB_DRAIN = 144;  // every MMA of the CTA done
constexpr int SBB_TMEM = 152;   // u32: TMEM base
constexpr int SBB_ABORT = 156;  // u32: a wait timed out
constexpr int SBB_KLAND = 160;  // a band reaching before the chunk landed (K): fill its rows before the chunk
constexpr int SBB_VLAND = 168;  // the same for V
constexpr int SBB_INFO = 192;   // [8] the record of work item i is in slot i % 8

struct SbArgs {
  long long P0;              // one chunk: its first position, rows, ring row
  int C, hq, G, hkv, np, nitems;
  int ring_seq;
  VarlenPlan plan;           // a batch of chunks: the plan (items of 128 query rows)
  uint16_t *out;             // [rows][hq][128] (row-by-row stores)
  const int32_t *slot_pos;  // [ring sequences][128]
  const uint16_t *ring_k;   // [ring sequences][hkv][128][192]
  const uint16_t *ring_v;   // [ring sequences][hkv][128][128]
  const float *sinks;
  const float *table;
  float scale_log2;
  unsigned *status;
};

__device__ __forceinline__ bool sb_wait(uint32_t bar, uint32_t parity, volatile uint32_t *abort) {
  const bool ok = mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, ok);
}

// The record of a work item: 128 query rows (rows r0 .. r0 + 128/G - 1 of a
// chunk, times the G heads of KV head kv) and the chunk they belong to.
struct SbInfo {
  int c0;            // the chunk's first row in q, out and the staged rows
  int C;             // its rows
  int P0;            // position of its first row
  int seq;           // its ring
  int kv, r0;
  int mode;          // > 0: attend; 0: a bad position or sequence (rows written as zeros)
  int pad;
  uint32_t held[4];  // bit c: ring slot c holds position P0 - 128 + ((c - P0) mod 128)
  uint32_t pad2[4];
};
static_assert(sizeof(SbInfo) == 64, "64-byte records");
// Bits lo .. hi (clamped to 0 .. 31) of a word.
__device__ __forceinline__ uint32_t span_bits(int lo, int hi) {
  lo = lo < 0 ? 0 : lo;
  hi = hi > 31 ? 31 : hi;
  return lo > hi ? 0u : (0xffffffffu >> (31 - hi)) & (0xffffffffu << lo);
}
// An item whose rows reach before the chunk: those band columns are
// attended only where the position exists and its ring slot holds it.
__device__ __forceinline__ bool sb_boundary(const SbInfo &t) { return t.mode > 0 && t.r0 < WIN - 1; }

// VARLEN: the items of the long chunks of a batch (plan); else one chunk.
template <bool VARLEN>
__global__ void __launch_bounds__(SB_THREADS, 1)
    swa_band_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmo,
                    const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                    const SbArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *gbase = smem_raw + (base - raw);
  const uint32_t sK = base + SB_OFF_K, sV = base + SB_OFF_V, sO = base + SB_OFF_O, sBar = base + SB_OFF_BAR;
  volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(gbase + SB_OFF_BAR + SBB_ABORT);
  SbInfo *infos = reinterpret_cast<SbInfo *>(gbase + SB_OFF_INFO);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nitems = VARLEN ? a.plan.item_prefix[a.plan.n] : a.nitems;
  const int n_my = (int)blockIdx.x < nitems ? (nitems - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  // record of item i (written by the query producer, two items ahead)
  auto info = [&](int i) -> const SbInfo & { return infos[i % SB_NINFO]; };
  auto info_ready = [&](int i) {  // one thread
    return mbar_wait(sBar + SBB_INFO + 8 * (i % SB_NINFO), (uint32_t)(i / SB_NINFO) & 1u, abort_flag);
  };
  if (n_my == 0) return;  // (a batch of short chunks only: nothing set up yet, nothing to do)

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(sBar + SBB_QFULL + 8 * i, 1);
      mbar_init(sBar + SBB_QROPE + 8 * i, 128);
      mbar_init(sBar + SBB_QFREE + 8 * i, 1);
      mbar_init(sBar + SBB_SFULL + 8 * i, 1);
      mbar_init(sBar + SBB_PREADY + 8 * i, 256);
    }
    mbar_init(sBar + SBB_KFULL, 1);
    mbar_init(sBar + SBB_VFULL, 1);
    mbar_init(sBar + SBB_KFREE, 1);
    mbar_init(sBar + SBB_VFREE, 1);
    mbar_init(sBar + SBB_KPATCH, 128);
    mbar_init(sBar + SBB_VPATCH, 128);
    mbar_init(sBar + SBB_OFULL, 1);
    mbar_init(sBar + SBB_OFREE, 256);
    mbar_init(sBar + SBB_DRAIN, 1);
    mbar_init(sBar + SBB_KLAND, 1);
    mbar_init(sBar + SBB_VLAND, 1);
    for (int k = 0; k < SB_NINFO; ++k) mbar_init(sBar + SBB_INFO + 8 * k, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == SB_WARP_MMA) {
    tmem_alloc(sBar + SBB_TMEM, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(gbase + SB_OFF_BAR + SBB_TMEM);

  if (warp == SB_WARP_TMA || warp == SB_WARP_TMAQ) {
    // ------------------------------------------------------------ TMA producers
    // Warp 13 loads the bands, warp 14 the query tiles (a load from HBM
    // that waits for the TMA unit does not hold up the other stream).  Each
    // load goes out as soon as its buffer is free: K(k) after S(k-1), V(v)
    // after P V(v-1), Q(q) after S(q-2).  Lane 0's view of a barrier decides
    // for the warp.
    const bool qw = warp == SB_WARP_TMAQ;
    int last_a = -1, last_b = -1;  // last loads issued: K, V (warp 13); even, odd query tile (warp 14)
    // Warp 14 writes the record of item i (slot i % 8) before loading its
    // query tile; the slot last served item i-8, whose epilogue is done once
    // S(i-2) is (the query tile waits for that).  A batch's items come in
    // chunk order, so the chunk search starts at the previous item's chunk.
    int s_cur = 0;
    auto make_info = [&](int i) {
      const int w = (int)blockIdx.x + i * (int)gridDim.x;
      SbInfo t{};
      if (VARLEN) {
        int lo = s_cur, hi = a.plan.n;  // item_prefix[lo] <= w < item_prefix[hi]
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (a.plan.item_prefix[mid] <= w) lo = mid; else hi = mid;
        }
        s_cur = lo;
        const int local = w - a.plan.item_prefix[lo];
        t.kv = local % a.hkv;
        t.r0 = (local / a.hkv) * a.np;
        t.c0 = a.plan.cu_rows[lo];
        t.C = a.plan.cu_rows[lo + 1] - t.c0;
        t.P0 = (int)a.plan.P0[lo];
        t.seq = a.plan.seq[lo];
        t.mode = a.plan.mode[lo];
      } else {
        t.kv = w % a.hkv;
        t.r0 = (w / a.hkv) * a.np;
        t.c0 = 0;
        t.C = a.C;
        t.P0 = (int)a.P0;
        t.seq = a.ring_seq;
        t.mode = 1;
      }
      for (int k = 0; k < 4; ++k) {  // ring slot c = 32k + lane: holds its pre-chunk position?
        bool h = false;
        if (sb_boundary(t)) {
          const int c = 32 * k + lane;
          const long long pos = (long long)t.P0 - WIN + ((c - (t.P0 & (WIN - 1))) & (WIN - 1));
          h = pos >= 0 && a.slot_pos[(long long)t.seq * WIN + c] == (int32_t)pos;
        }
        t.held[k] = __ballot_sync(0xffffffffu, h);
      }
      if (lane == 0) {
        infos[i % SB_NINFO] = t;
        mbar_arrive(sBar + SBB_INFO + 8 * (i % SB_NINFO));
      }
      __syncwarp();
    };
    auto load_q = [&](int i) {
      make_info(i);
      const SbInfo &t = info(i);
      const uint32_t bar = sBar + SBB_QFULL + 8 * (i & 1);
      mbar_expect_tx_elect(bar, SB_QTILE);
      for (int part = 0; part < 3; ++part)
        tma_load_3d_elect(base + (i & 1) * SB_QTILE + part * SB_QPART, &tmq, 64 * part, t.kv * a.G, t.c0 + t.r0, bar);
      (i & 1 ? last_b : last_a) = i;
    };
    // (warp 13) false when the record did not come (abort)
    auto load_band = [&](int i, bool v) -> bool {
      if (!sb_wait(sBar + SBB_INFO + 8 * (i % SB_NINFO), (uint32_t)(i / SB_NINFO) & 1u, abort_flag)) return false;
      const SbInfo &t = info(i);
      const uint32_t bar = sBar + (v ? SBB_VFULL : SBB_KFULL);
      const int parts = v ? 2 : 3;
      mbar_expect_tx_elect(bar, parts * SB_KPART);
      for (int part = 0; part < parts; ++part)
        tma_load_4d_elect((v ? sV : sK) + part * SB_KPART, v ? (const void *)&tmv : (const void *)&tmk, 0, part, t.kv,
                          t.c0 + t.r0 - 128, bar);
      (v ? last_b : last_a) = i;
      return true;
    };
    auto ready = [&](uint32_t bar, uint32_t parity) {
      return __shfl_sync(0xffffffffu, (int)mbar_test(bar, parity), 0) != 0;
    };
    int n1 = 1, n2 = 1;  // next K and V (warp 13); next query tile: n1 (warp 14)
    if (n_my > 0) {
      if (qw) {
        load_q(0);
        if (n_my > 1) load_q(1);
        n1 = 2;
      } else if (!load_band(0, false) || !load_band(0, true)) {
        n1 = n2 = n_my;  // aborted: nothing more to load
      }
    }
    // Warp 13 also watches each band's K and V land, in item order, and
    // tells the RoPE warps when a band that reaches before the chunk is in
    // (they then fill its rows before the chunk).  A waiter on a barrier that
    // may be two phases behind would mistake an old phase for the one it
    // wants, so the next load of a stream goes out only once the previous
    // one was seen to land, and the RoPE warps wait on barriers that move
    // once per such band.
    int lk = 0, lv = 0;  // next items whose K / V landing is still to be seen
    uint64_t t_last = global_ns();
    while (qw ? n1 < n_my : (n1 < n_my || n2 < n_my || lk < n_my || lv < n_my)) {
      bool prog = false;
      if (qw) {
        if (ready(sBar + SBB_QFREE + 8 * (n1 & 1), (uint32_t)((n1 - 2) >> 1) & 1u)) {
          load_q(n1++);
          prog = true;
        }
      } else {
        if (lk < n1 && ready(sBar + SBB_KFULL, (uint32_t)lk & 1u)) {
          if (lane == 0 && sb_boundary(info(lk))) mbar_arrive(sBar + SBB_KLAND);
          ++lk;
          prog = true;
        }
        if (lv < n2 && ready(sBar + SBB_VFULL, (uint32_t)lv & 1u)) {
          if (lane == 0 && sb_boundary(info(lv))) mbar_arrive(sBar + SBB_VLAND);
          ++lv;
          prog = true;
        }
        if (n1 < n_my && lk == n1 && ready(sBar + SBB_KFREE, (uint32_t)(n1 - 1) & 1u)) {
          if (!load_band(n1++, false)) break;
          prog = true;
        }
        if (n2 < n_my && lv == n2 && ready(sBar + SBB_VFREE, (uint32_t)(n2 - 1) & 1u)) {
          if (!load_band(n2++, true)) break;
          prog = true;
        }
      }
      if (prog) {
        t_last = global_ns();
      } else {
        // warp-uniform: lane 0 decides whether to give up (aborted elsewhere,
        // or no buffer came free for 2 s)
        const bool stop =
            __shfl_sync(0xffffffffu, (int)(*abort_flag != 0 || global_ns() - t_last > 2000000000ull), 0) != 0;
        if (stop) {
          if (lane == 0) *abort_flag = 1;
          break;
        }
        __nanosleep(32);
      }
    }
    // On an abort, the loads already issued land before the CTA leaves
    // (bounded by time only: the abort flag is already set).
    if (*abort_flag && lane == 0) {
      volatile uint32_t local = 0;
      for (int s = 0; s < 2; ++s) {
        const int li = s ? last_b : last_a;
        if (li < 0) continue;
        local = 0;
        const uint32_t bar = qw ? sBar + SBB_QFULL + 8 * s : sBar + (s ? SBB_VFULL : SBB_KFULL);
        mbar_wait(bar, qw ? (uint32_t)(li >> 1) & 1u : (uint32_t)li & 1u, &local, 1000000000ull);
      }
    }
    __syncwarp();
  } else if (warp == SB_WARP_MMA) {
    // ------------------------------------------------------------ MMA issuer
    // Order: S(0), then S(i), P V(i-1) for i = 1.. (the tensor core computes
    // the next tile's scores while the softmax warps work on the last ones),
    // then P V of the last item.
    const uint32_t id_s = idesc_bf16(128, SB_N, 0, 0);
    const uint32_t id_pv = idesc_bf16(128, 128, 0, 1);
    const uint64_t dk = sdesc_sw128(sK, 16, 1024);
    const uint64_t dv = sdesc_sw128(sV, SB_KPART, 1024);  // LBO = the other 64-dim half of V
    int nbk = 0, nbv = 0;  // boundary items met (their patch barriers' phases)
    auto issue_S = [&](int i) -> bool {
      const int q = i & 1;
      if (!sb_wait(sBar + SBB_INFO + 8 * (i % SB_NINFO), (uint32_t)(i / SB_NINFO) & 1u, abort_flag)) return false;
      const bool bnd = sb_boundary(info(i));
      if (!sb_wait(sBar + SBB_QROPE + 8 * q, (uint32_t)(i >> 1) & 1u, abort_flag)) return false;
      if (!sb_wait(sBar + SBB_KFULL, (uint32_t)i & 1u, abort_flag)) return false;
      if (bnd) {
        if (!sb_wait(sBar + SBB_KPATCH, (uint32_t)nbk & 1u, abort_flag)) return false;
        ++nbk;
      }
      tc_fence_after();
      const uint64_t dq = sdesc_sw128(base + q * SB_QTILE, 16, 1024);
      const uint32_t d = tmem + (q ? SB_COL_S1 : 0u);
      for (int kb = 0; kb < 3; ++kb) {
        const uint64_t a0 = dq + (uint64_t)((kb * SB_QPART) >> 4);
        const uint64_t b0 = dk + (uint64_t)((kb * SB_KPART) >> 4);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_ss_elect(d, a0 + 2 * kk, b0 + 2 * kk, id_s, (kb | kk) != 0);
      }
      mma_commit_elect(sBar + SBB_SFULL + 8 * q);
      mma_commit_elect(sBar + SBB_KFREE);
      mma_commit_elect(sBar + SBB_QFREE + 8 * q);
      return true;
    };
    auto issue_PV = [&](int i) -> bool {  // (S(i) came first: the record of item i is in)
      const bool bnd = sb_boundary(info(i));
      const int s = i & 1;
      if (!sb_wait(sBar + SBB_PREADY + 8 * s, (uint32_t)(i >> 1) & 1u, abort_flag)) return false;
      if (!sb_wait(sBar + SBB_VFULL, (uint32_t)i & 1u, abort_flag)) return false;
      if (bnd) {
        if (!sb_wait(sBar + SBB_VPATCH, (uint32_t)nbv & 1u, abort_flag)) return false;
        ++nbv;
      }
      if (i > 0 && !sb_wait(sBar + SBB_OFREE, (uint32_t)(i - 1) & 1u, abort_flag)) return false;
      tc_fence_after();
      const uint32_t ap = tmem + (s ? SB_COL_S1 : 0u);
      const uint32_t d = tmem + SB_COL_O;
#pragma unroll
      for (int kk = 0; kk < SB_N / 16; ++kk) mma_ts_elect(d, ap + 8 * kk, dv + 128 * kk, id_pv, kk > 0 ? 1u : 0u);
      mma_commit_elect(sBar + SBB_OFULL);
      mma_commit_elect(sBar + SBB_VFREE);
      return true;
    };
    bool ok = true;
    for (int i = 0; i < n_my && ok; ++i) {
      ok = issue_S(i);
      if (ok && i > 0) ok = issue_PV(i - 1);
    }
    if (ok && n_my > 0) issue_PV(n_my - 1);
    // Every MMA issued must be finished before TMEM is released (bounded by
    // time only, even after an abort).
    mma_commit_elect(sBar + SBB_DRAIN);
    if (lane == 0) {
      volatile uint32_t local = 0;
      mbar_wait(sBar + SBB_DRAIN, 0, &local, 1000000000ull);
    }
    __syncwarp();
  }
  else if (warp >= SB_WARP_ROPE) {
    // ------------------------------------------------------------ RoPE + ring rows (warps 8-11)
    const int t = tid - 32 * SB_WARP_ROPE;
    int nb = 0;  // boundary items met (phases of the land / fill barriers)
    for (int i = 0; i < n_my; ++i) {
      if (!info_ready(i)) break;
      const SbInfo &it0 = info(i);
      const int kv = it0.kv, r0 = it0.r0;
      const int q = i & 1;
      // (row, chunk pair) tasks: row r = it / 4 (chunk row r0 + r / G), dims
      // 8c..8c+7 with 32+8c..; table rows fetched before the wait.  Rows past
      // the chunk, and every row of an item of a bad chunk, are not rotated.
      float4 tv[4][4];
      bool liv[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int it = t + 128 * k, r = it >> 2, c = it & 3;
        const int ii = r0 + r / a.G;
        liv[k] = it0.mode > 0 && ii < it0.C;
        if (liv[k]) {
          const float4 *tr = reinterpret_cast<const float4 *>(a.table + ((long long)it0.P0 + ii) * 64 + 16 * c);
#pragma unroll
          for (int u = 0; u < 4; ++u) tv[k][u] = tr[u];
        }
      }
      if (!mbar_wait(sBar + SBB_QFULL + 8 * q, (uint32_t)(i >> 1) & 1u, abort_flag)) break;
      uint8_t *qt = gbase + q * SB_QTILE;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (!liv[k]) continue;
        const int it = t + 128 * k, r = it >> 2, c = it & 3;
        float cs[16];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          cs[4 * u] = tv[k][u].x; cs[4 * u + 1] = tv[k][u].y; cs[4 * u + 2] = tv[k][u].z; cs[4 * u + 3] = tv[k][u].w;
        }
        uint4 *p1 = reinterpret_cast<uint4 *>(qt + r * 128 + ((c ^ (r & 7)) << 4));
        uint4 *p2 = reinterpret_cast<uint4 *>(qt + r * 128 + (((c + 4) ^ (r & 7)) << 4));
        uint4 o1, o2;
        rope_pair8(*p1, *p2, cs, o1, o2);
        *p1 = o1;
        *p2 = o2;
      }
      fence_proxy_async_smem();
      mbar_arrive(sBar + SBB_QROPE + 8 * q);
      if (!sb_boundary(it0)) continue;
      // Band rows 0 .. 127-r0 are chunk rows r0-128 .. -1, positions
      // P0+r0-128 .. P0-1: the ring row where the slot holds the position,
      // else zeros (in a batch these rows of the box belong to the previous
      // chunk; before row 0 of the batch the box brought zeros).
      const int t_hi = WIN - r0;
      const uint16_t *rk = a.ring_k + ((long long)it0.seq * a.hkv + kv) * WIN * DQK;
      const uint16_t *rv = a.ring_v + ((long long)it0.seq * a.hkv + kv) * WIN * DV;
      for (int h = 0; h < 2; ++h) {
        const bool v = h == 1;
        if (!mbar_wait(sBar + (v ? SBB_VLAND : SBB_KLAND), (uint32_t)nb & 1u, abort_flag)) break;
        const int nch = v ? DV / 8 : DQK / 8;  // 16-byte chunks of a row
        // asynchronous 16-byte copies, all in flight before the one wait
        for (int e = t; e < t_hi * nch; e += 128) {
          const int tr = e / nch, cc = e % nch;
          const long long p = (long long)it0.P0 + r0 - 128 + tr;
          const int slot = (int)(p & (WIN - 1));
          const uint32_t dst =
              (v ? SB_OFF_V : SB_OFF_K) + (cc >> 3) * SB_KPART + tr * 128 + (((cc & 7) ^ (tr & 7)) << 4);
          if (p >= 0 && ((it0.held[slot >> 5] >> (slot & 31)) & 1u)) {
            const uint16_t *src = v ? rv + (long long)slot * DV + 8 * cc : rk + (long long)slot * DQK + 8 * cc;
            cp_async16(base + dst, src);
          } else {
            *reinterpret_cast<uint4 *>(gbase + dst) = make_uint4(0, 0, 0, 0);
          }
        }
        cp_async_commit();
        cp_async_wait<0>();
        fence_proxy_async_smem();
        mbar_arrive(sBar + (v ? SBB_VPATCH : SBB_KPATCH));
      }
      ++nb;
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue (warps 0-7)
    // Warp w reads TMEM lanes 32 (w % 4) .. (tile rows d * G + g) and half
    // h = w / 4 of the columns: band columns 72h .. 72h+71, O columns
    // 64h .. 64h+63.  The halves of a row exchange their maxima and partial
    // sums through shared memory.  Named barriers 1 and 2 span the eight
    // warps; before each, the warps agree on their outcome, so all of them
    // always reach it.
    const int row = tid & 127, h = tid >> 7;
    const int d = row / a.G, g = row - d * a.G;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const float sl2 = a.scale_log2;
    float *red_m = reinterpret_cast<float *>(gbase + SB_OFF_RED);  // [2 halves][128] maxima
    float *red_l = red_m + 256;                                      // [2 items][2 halves][128] sums
    // The output of item j: O / l as bf16 into the staging tile, then two
    // TMA boxes; the last block of a chunk in a batch, whose box would reach
    // into the next chunk's rows, is stored row by row instead.
    auto epilogue = [&](int j, bool good) -> bool {
      const SbInfo &t = info(j);  // (its softmax waited for the record)
      const int kv = t.kv;
      const bool by_rows = VARLEN && t.r0 + a.np > t.C;
      if (good) good = sb_wait(sBar + SBB_OFULL, (uint32_t)j & 1u, abort_flag);
      if (tid == 0) bulk_wait_read_all();  // the last store has read the staging tile
      good = named_bar_and(1, 256, good);
      if (!good) return false;
      tc_fence_after();
      const float inv = 1.f / (red_l[(j & 1) * 256 + row] + red_l[(j & 1) * 256 + 128 + row]);  // l >= e^(sink-m) > 0
      const uint64_t invv = f32x2(inv, inv), zero2 = f32x2(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_base + SB_COL_O + 64 * h + 32 * c, o);
        tmem_wait_ld();
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {  // O / l, one packed multiply per pair
          float y0, y1;
          f32x2_split(fma_f32x2(f32x2(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), invv, zero2), y0, y1);
          w[e >> 1] = pack_bf16(y0, y1);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t w0 = w[4 * u], w1 = w[4 * u + 1], w2 = w[4 * u + 2], w3 = w[4 * u + 3];
          const int ch = 4 * c + u;  // 16-byte chunk of dims 64h + 8 ch .. within part h
          if (by_rows) {
            if (t.r0 + d < t.C)
              reinterpret_cast<uint4 *>(a.out + ((long long)(t.c0 + t.r0 + d) * a.hq + kv * a.G + g) * DV + 64 * h)[ch] =
                  make_uint4(w0, w1, w2, w3);
          } else {
            *reinterpret_cast<uint4 *>(gbase + SB_OFF_O + h * SB_QPART + row * 128 + ((ch ^ (row & 7)) << 4)) =
                make_uint4(w0, w1, w2, w3);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(sBar + SBB_OFREE);
      fence_proxy_async_smem();
      named_bar_sync(1, 256);
      if (tid == 0 && !by_rows) {  // rows past the last one of the output are clipped by the store
        tma_store_3d(&tmo, 0, kv * a.G, t.c0 + t.r0, sO);
        tma_store_3d(&tmo, 64, kv * a.G, t.c0 + t.r0, sO + SB_QPART);
        bulk_commit();
      }
      return true;
    };
    bool ok = true;
    for (int i = 0; i <= n_my; ++i) {
      if (i < n_my && ok) {
        const int s = i & 1;
        ok = sb_wait(sBar + SBB_INFO + 8 * (i % SB_NINFO), (uint32_t)(i / SB_NINFO) & 1u, abort_flag);
        const SbInfo &t = info(i);
        const float sink2 = ok ? a.sinks[t.kv * a.G + g] * LOG2E : 0.f;
        const int r0 = t.r0;
        if (ok) ok = sb_wait(sBar + SBB_SFULL + 8 * s, (uint32_t)(i >> 1) & 1u, abort_flag);
        ok = named_bar_and(2, 256, ok);
        if (ok) {
          tc_fence_after();
          const uint32_t tS = tmem + lane_base + (s ? SB_COL_S1 : 0u);
          const int cb = 72 * h;  // first band column of this half
          uint32_t v[72];
          tmem_ld32(tS + cb, *reinterpret_cast<uint32_t(*)[32]>(v));
          tmem_ld32(tS + cb + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
          tmem_ld8(tS + cb + 64, *reinterpret_cast<uint32_t(*)[8]>(v + 64));
          // Attended columns (bit e of word k = column cb + 32k + e): d+1 <=
          // t <= d+128 and, before the chunk, the position exists and its ring
          // slot holds it.
          uint32_t msk[3];
#pragma unroll
          for (int k = 0; k < 3; ++k) msk[k] = span_bits(d + 1 - cb - 32 * k, d + WIN - cb - 32 * k);
          if (t.mode <= 0) {  // a bad chunk: nothing attended, its rows come out as zeros
#pragma unroll
            for (int k = 0; k < 3; ++k) msk[k] = 0u;
          } else if (sb_boundary(t)) {
            const long long pfirst = (long long)t.P0 + r0 - 128;  // position of column 0
            const int tneg = WIN - r0;                     // columns before the chunk
            const int t0 = pfirst < 0 ? (int)-pfirst : 0;  // first column with a position
            const int off = (int)(pfirst & (WIN - 1));     // ring slot of column 0
#pragma unroll
            for (int k = 0; k < 3; ++k) {
              const int ck = cb + 32 * k;
              const int sb = ck + off, w0 = (sb >> 5) & 3, sh = sb & 31;
              const uint32_t hk = __funnelshift_r(t.held[w0], t.held[(w0 + 1) & 3], sh);  // bit e: slot (sb + e) % 128
              const uint32_t before = span_bits(-ck, tneg - 1 - ck);
              const uint32_t exists = span_bits(t0 - ck, 31);
              msk[k] &= ~before | (hk & exists);
            }
          }
          tmem_wait_ld();
          // Masked raw scores: outside the first items only columns 0 .. 15
          // (before a row's window) and 128 .. 143 (after it) can be masked,
          // i.e. the first 16 and the last 16 of either half.
          const uint32_t NINF = __float_as_uint(-INFINITY);
          if (sb_boundary(t) || t.mode <= 0) {
#pragma unroll
            for (int e = 0; e < 72; ++e) v[e] = (msk[e >> 5] >> (e & 31)) & 1u ? v[e] : NINF;
          } else {
#pragma unroll
            for (int e = 0; e < 72; ++e)
              if (e < 16 || e >= 56) v[e] = (msk[e >> 5] >> (e & 31)) & 1u ? v[e] : NINF;
          }
          float mx = -INFINITY;
#pragma unroll
          for (int e = 0; e < 72; e += 2) mx = fmax3(mx, __uint_as_float(v[e]), __uint_as_float(v[e + 1]));
          red_m[h * 128 + row] = mx;
          named_bar_sync(2, 256);  // both maxima; both halves' S loads done before any P store
          // row maximum in log2 units (the scale is positive), with the sink
          mx = fmaxf(fmaxf(red_m[row], red_m[128 + row]) * sl2, sink2);
          // p = 2^(s * scale - m) (one packed FMA per pair) as bf16 pairs,
          // packed into the registers already read; sums in packed pairs
          const uint64_t sl2v = f32x2(sl2, sl2), nmv = f32x2(-mx, -mx);
          uint64_t sumv[4] = {f32x2(h == 0 ? ex2(sink2 - mx) : 0.f, 0.f), 0, 0, 0};
#pragma unroll
          for (int e = 0; e < 72; e += 2) {
            float a0, a1;
            f32x2_split(fma_f32x2(f32x2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), sl2v, nmv), a0, a1);
            const float p0 = ex2(a0), p1 = ex2(a1);
            sumv[(e >> 1) & 3] = add_f32x2(sumv[(e >> 1) & 3], f32x2(p0, p1));
            v[e >> 1] = pack_bf16(p0, p1);
          }
          float su[8];
#pragma unroll
          for (int u = 0; u < 4; ++u) f32x2_split(sumv[u], su[2 * u], su[2 * u + 1]);
          red_l[(i & 1) * 256 + h * 128 + row] = ((su[0] + su[1]) + (su[2] + su[3])) + ((su[4] + su[5]) + (su[6] + su[7]));
          tmem_st32(tS + 36 * h, *reinterpret_cast<const uint32_t(*)[32]>(v));
          tmem_st4(tS + 36 * h + 32, *reinterpret_cast<const uint32_t(*)[4]>(v + 32));
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(sBar + SBB_PREADY + 8 * s);
        }
      }
      if (i > 0) {
        ok = epilogue(i - 1, ok);
        if (!ok) break;
      }
    }
    if (tid == 0) bulk_wait_all();  // the stores are done before the CTA leaves
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag && tid == 0) flag(a.status, ST_TIMEOUT);
  if (warp == SB_WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

namespace {

// Tensor maps (q and out as 128-row tiles of (position, head) rows; the
// staged rows as 144-token boxes of one KV head) and the common arguments.
bool band_setup(const uint16_t *q, long long T, int hq, const KvView &chunk, const KvView &ring, const float *sinks,
                const float *table, float softmax_scale, uint16_t *out, unsigned *status, CUtensorMap *m,
                SbArgs *a) {
  const int hkv = ring.hkv, G = hq / hkv;
  if (G < 8 || 128 % G || T <= 0 || T >= (1LL << 31)) return false;
  if (!make_tma_map_heads3d(&m[0], q, T, hq, DQK, G) || !make_tma_map_heads3d(&m[1], out, T, hq, DV, G) ||
      !make_tma_map_tokens4d(&m[2], chunk.k, T, hkv, DQK, SB_N, true) ||
      !make_tma_map_tokens4d(&m[3], chunk.v, T, hkv, DV, SB_N, true))
    return false;
  *a = SbArgs{};
  a->hq = hq;
  a->G = G;
  a->hkv = hkv;
  a->np = 128 / G;
  a->slot_pos = ring.slot_pos;
  a->ring_k = ring.k;
  a->ring_v = ring.v;
  a->sinks = sinks;
  a->table = table;
  a->scale_log2 = softmax_scale * LOG2E;
  a->out = out;
  a->status = status;
  return true;
}

}  // namespace

cudaError_t launch_swa_band(const uint16_t *q, int64_t P0, int C, int seq, int hq, const KvView &chunk,
                            const KvView &ring, const float *sinks, const float *table, float softmax_scale,
                            uint16_t *out, unsigned *status, cudaStream_t st, bool *taken) {
  *taken = false;
  CUtensorMap m[4];
  SbArgs a;
  if (!band_setup(q, C, hq, chunk, ring, sinks, table, softmax_scale, out, status, m, &a)) return cudaSuccess;
  const long long nitems = ((long long)C + a.np - 1) / a.np * a.hkv;
  if (nitems >= (1LL << 31)) return cudaSuccess;
  cudaError_t e = ensure_smem_limit(10, (const void *)swa_band_kernel<false>, SB_SMEM);
  if (e != cudaSuccess) return e;
  a.P0 = P0;
  a.C = C;
  a.nitems = (int)nitems;
  a.ring_seq = seq;
  const long long grid = nitems < num_sms() ? nitems : num_sms();
  swa_band_kernel<false><<<(unsigned)grid, SB_THREADS, SB_SMEM, st>>>(m[0], m[1], m[2], m[3], a);
  *taken = true;
  return cudaGetLastError();
}

cudaError_t launch_swa_band_varlen(const uint16_t *q, const int32_t *cu_rows, const int64_t *P0, const int32_t *seq,
                                   int n, long long T, int hq, const KvView &chunk, const KvView &ring,
                                   const float *sinks, const float *table, int64_t max_pos, float softmax_scale,
                                   void *ws, uint16_t *out, unsigned *status, cudaStream_t st, bool *taken) {
  *taken = false;
  CUtensorMap m[4];
  SbArgs a;
  if (!band_setup(q, T, hq, chunk, ring, sinks, table, softmax_scale, out, status, m, &a)) return cudaSuccess;
  // the plan in items of 128 query rows; chunks of at most 32 query rows and
  // 16 tokens go to the short-chunk kernel
  const VarlenSizes z = varlen_sizes(n, T, hq, a.hkv, max_pos, 128, false);
  if (z.items_max >= (1LL << 31)) return cudaSuccess;
  cudaError_t e = ensure_smem_limit(11, (const void *)swa_band_kernel<true>, SB_SMEM);
  if (e != cudaSuccess) return e;
  a.plan = varlen_plan_view(z, ws, cu_rows, P0, seq, n);
  e = launch_varlen_plan(a.plan, T, hq, a.hkv, 128, max_pos, ring.num_seqs, SWA_SHORT_ROWS, SWA_SHORT_MAX_C, status,
                         st);
  if (e != cudaSuccess) return e;
  const long long grid = z.items_max < num_sms() ? z.items_max : num_sms();
  if (grid > 0) swa_band_kernel<true><<<(unsigned)grid, SB_THREADS, SB_SMEM, st>>>(m[0], m[1], m[2], m[3], a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  *taken = true;
  return launch_swa_short(q, a.plan, n, T, hq, chunk, ring, sinks, table, softmax_scale, out, status, st);
}

}  // namespace kvr
