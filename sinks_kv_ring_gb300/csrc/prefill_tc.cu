// prefill_tc.cu -- chunked prefill on the Blackwell tensor cores: TMA tile
// loads, tcgen05.mma with accumulators in TMEM, fp32 online softmax in
// registers.  One kernel serves full-attention layers (paged pool) and, in
// window mode, windowed layers (ring + staged chunk rows, sink); one chunk
// or a batch of chunks of different lengths (varlen plan, with key splits
// for short chunks).
//
// gaudi-cookbook "MiMo-V2.6-Flash on Gaudi 2", "Tiled global-attention
// prefill": softmax is per query row, so independent tiles of query rows
// need no merge; row i of the chunk (position P0 + i) attends positions
// 0..P0 + i.  Xiaomi "Full-Pipeline Inference Optimization", section 1.1:
// chunked prefill is compute-bound, so this is the one contraction of the
// path that is sized for the tensor cores.
//
// One CTA = two query tiles of 128 rows (the rows are consecutive
// (position, head) pairs of one KV head's GQA group), one SM, 320 threads:
//   warps 0-3  softmax of tile 0 (thread = row = TMEM lane)
//   warps 4-7  softmax of tile 1
//   warp  8    TMEM owner and MMA issuer (converged; elect.sync issues)
//   warp  9    TMA producer (converged; elect.sync issues)
// TMEM (512 columns): S0 | S1 | O0 | O1, 128 fp32 columns each.  The bf16
// probabilities P of a tile are written over the first 64 columns of its S
// and feed the P.V product straight from TMEM.
// Shared memory: Q0, Q1 (3 x 16 KB each, 128-byte swizzled K-major) and a
// ring of eight 16 KB slots.  A query tile is three TMA boxes of q (128 / G
// positions x G heads x 64 dims) when G divides 128, its dims 0-63 then
// rotated in place; a single chunk's output tile leaves through its query
// region as two TMA boxes.  Every K/V tile of 128 keys is five slot loads:
// K dims 0-63, 64-127, 128-191 (K-major, for S = Q K^T) and V dims 0-63,
// 64-127 (MN-major, for O += P V).  The three K loads and the two V loads of
// a key tile each complete on one transaction barrier (double-buffered);
// query tile 1 relies on tile 0's waits.
// MMA order per key tile j (the two tiles ping-pong, so one tile's softmax
// overlaps the other tile's products):
//   O0 += P0(j-1) V(j-1);  S0 = Q0 K(j)^T;  O1 += P1(j-1) V(j-1);  S1 = Q1 K(j)^T
// Softmax keeps a per-row reference max and rescales O in TMEM only when the
// row max grows by more than 2^8, so most tiles never touch O.
#include <cuda.h>

#include "launch.h"
#include "tc_ptx.cuh"

namespace kvr {
namespace {

using namespace tc;

constexpr int TC_THREADS = 320;
constexpr int TC_SLOT = 16384;                 // 128 rows x 128 bytes
constexpr int TC_NSLOT = 8;
constexpr int TC_QTILE = 3 * TC_SLOT;          // 128 rows x 192 dims
constexpr int TC_OFF_RING = 2 * TC_QTILE;      // 96 KB
constexpr int TC_OFF_BAR = TC_OFF_RING + TC_NSLOT * TC_SLOT;  // 224 KB
constexpr int TC_OFF_TAG = TC_OFF_BAR + 256;                  // windowed: 128 bits, slot c holds its window position
constexpr int TC_SMEM = TC_OFF_TAG + 512 + 1024;              // + alignment slack
constexpr unsigned ST_TIMEOUT = 8u;
constexpr float NEG_INF = -INFINITY;
constexpr float RESCALE_THRESHOLD = 8.0f;      // log2 units

// barrier area layout (byte offsets)
constexpr int B_FULL = 0;       // [4]: K loads (0, 1) / V loads (2, 3) of key tile t landed, t % 2
constexpr int B_EMPTY = 64;     // [8]
constexpr int B_SFULL = 128;    // [2]
constexpr int B_PREADY = 144;   // [2]
constexpr int B_OFINAL = 160;   // [2]
constexpr int B_TMEM = 176;     // u32: TMEM base address
constexpr int B_ABORT = 180;    // u32: set when a wait timed out
constexpr int B_DRAIN = 192;    // all MMAs of the CTA done (before TMEM is freed)
constexpr int B_QFULL = 200;    // the query tiles' TMA boxes landed
constexpr int B_STALL = 208;    // test hook: a barrier nothing arrives on

// Every lane waits on the barrier; the warp agrees on the outcome so that it
// stays converged for the warp-collective (.sync.aligned / elect.sync)
// instructions that follow.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile uint32_t *abort,
                                          uint64_t limit_ns = 2000000000ull) {
  const bool ok = mbar_wait(bar, parity, abort, limit_ns);
  return __all_sync(0xffffffffu, ok);
}

struct TcArgs {
  const uint16_t *q;
  long long P0;
  int C, hq, G, hkv;
  const int32_t *bt;  // block-table row of the sequence (one chunk) or the whole table (varlen)
  int bsz, num_blocks, max_blocks;
  long long total_rows;  // rows of the pool tensors (num_blocks * hkv * bsz)
  const float *table;
  float scale_log2;
  uint16_t *out;
  unsigned *status;
  VarlenPlan plan;       // varlen only
  // windowed layers: ring tags, sinks, the ring row (sequence) of a single chunk
  const int32_t *slot_pos;
  const float *sinks;
  int ring_seq;
  int q_tma;  // query tiles come in as TMA boxes (tmq); else 16-byte copies
  int o_tma;  // one chunk: output tiles leave as TMA boxes (tmo); else per-row stores
  unsigned long long stall_ns;  // test hook: the MMA warp stalls before its first product (0 = never)
};

// Rows f0 .. f0+255 (those below nrows) of KV head kv's group, written as zeros.
__device__ void zero_rows(uint16_t *oc, long long f0, long long nrows, int kv, int G, int hq) {
  for (int it = threadIdx.x; it < 256 * 16; it += blockDim.x) {
    const long long f = f0 + it / 16;
    if (f < nrows)
      reinterpret_cast<uint4 *>(oc + ((f / G) * hq + (long long)kv * G + f % G) * DV)[it % 16] = make_uint4(0, 0, 0, 0);
  }
}

// 10 warps share 4 schedulers (3 warps on some), which caps registers at 168.
// VARLEN: the CTA's work item comes from the plan (chunk, row tile, KV head,
// key split); otherwise from blockIdx over one chunk.
// WINDOW: a windowed layer.  Row i attends positions (P0 + i - 128, P0 + i]
// with the sink in the denominator (its softmax state starts at (m, l) =
// (sink, 1)).  Key tiles are aligned at P0: tile u >= 0 holds the chunk's
// own rows P0 + 128u .. (tmk2 / tmv2: 4-D boxes of 128 staged tokens of one
// KV head); tile u = -1 is the sequence's whole ring in slot order (tmk / tmv:
// 128 ring rows), slot c holding position P0 - 128 + ((c - P0) mod 128) when
// its tag says so.  Otherwise tmk / tmv are the paged pool and tmk2 / tmv2
// are unused.
template <bool VARLEN, bool WINDOW>
__global__ void __launch_bounds__(TC_THREADS, 1)
    full_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                           const __grid_constant__ CUtensorMap tmk2, const __grid_constant__ CUtensorMap tmv2,
                           const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmo,
                           const TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *gbase = smem_raw + (base - raw);
  const uint32_t sQ0 = base, sQ1 = base + TC_QTILE, sRing = base + TC_OFF_RING, sBar = base + TC_OFF_BAR;
  volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(gbase + TC_OFF_BAR + B_ABORT);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- the work item: flat rows f0 .. f0+255 of KV head kv's group (row f is
  // position P0 + f / G, head f % G), keys k_lo .. k_hi-1
  int kv, split = 0, nsp = 1, plan_chunk = 0, rseq = a.ring_seq;
  long long f0, nrows, P0, prow = 0, crow0 = 0;
  const uint16_t *qc = a.q;  // row 0 of the chunk
  uint16_t *oc = a.out;
  const int32_t *bt = a.bt;
  if constexpr (VARLEN) {
    const long long b = blockIdx.x;
    if (b >= a.plan.item_prefix[a.plan.n]) return;
    const int s = plan_find(a.plan.item_prefix, a.plan.n, b);
    plan_chunk = s;
    const int local = (int)(b - a.plan.item_prefix[s]);
    const int mode = a.plan.mode[s];
    const long long c0 = a.plan.cu_rows[s];
    nrows = (a.plan.cu_rows[s + 1] - c0) * a.G;
    qc += c0 * a.hq * DQK;
    oc += c0 * a.hq * DV;
    kv = local % a.hkv;
    if (mode <= 0) {  // a position or the sequence id is out of range
      zero_rows(oc, (long long)(local / a.hkv) * 256, nrows, kv, a.G, a.hq);
      return;
    }
    nsp = mode;
    split = (local / a.hkv) % nsp;
    f0 = (long long)(local / a.hkv / nsp) * 256;
    P0 = a.plan.P0[s];
    crow0 = c0;
    rseq = a.plan.seq[s];
    if (!WINDOW) bt += (long long)rseq * a.max_blocks;
    prow = a.plan.prow_prefix[s];
  } else {
    // KV-head-major: the CTAs that run together read the same KV head's
    // K/V (at 122880 cached tokens one head's is 79 MB, all four together
    // more than L2), so it comes from DRAM about once.
    nrows = (long long)a.C * a.G;
    const int tiles = (int)((nrows + 255) / 256);
    kv = blockIdx.x / tiles;
    f0 = (long long)(blockIdx.x % tiles) * 256;
    P0 = a.P0;
  }
  const long long i_last = min(nrows - 1, f0 + 255) / a.G;
  long long k_lo = 0, k_hi = P0 + i_last + 1;
  if constexpr (VARLEN) {
    if (nsp > 1) {
      const long long L = a.plan.slen[plan_chunk];
      k_lo = split * L;
      k_hi = min(k_hi, k_lo + L);
    }
  }
  const long long pmin = P0 + f0 / a.G;  // smallest row position in the CTA
  // Windowed: key tiles u_lo .. u_hi, aligned at P0 (u = -1: the ring).
  int u_lo = 0;
  if constexpr (WINDOW) {
    u_lo = pmin - P0 >= WIN - 1 ? (int)((pmin - P0 - (WIN - 1)) / 128) : (P0 > 0 ? -1 : 0);
    k_lo = P0 + 128LL * u_lo;  // first key of tile 0 (for the ring tile: nominal)
  }
  const int ntiles = WINDOW ? (int)(i_last / 128) - u_lo + 1 : (int)((k_hi - k_lo + 127) / 128);
  // query tiles with live rows (a single chunk always runs both)
  const int nq = (!VARLEN || f0 + 128 < nrows) ? 2 : 1;

  // ---- set-up: barriers, TMEM, rotated Q tiles
  if constexpr (WINDOW) {
    // Slot c of the ring tile stands for position P0 - 128 + ((c - P0) mod
    // 128); one bit per slot says whether its tag agrees (warps 0-3).
    if (tid < WIN) {
      const long long pos = P0 - WIN + ((tid - (int)(P0 & (WIN - 1))) & (WIN - 1));
      const bool held = pos >= 0 && a.slot_pos[(long long)rseq * WIN + tid] == (int32_t)pos;
      const unsigned bits = __ballot_sync(0xffffffffu, held);
      if (lane == 0) reinterpret_cast<uint32_t *>(gbase + TC_OFF_TAG)[warp] = bits;
    }
  }
  if (tid == 0) {
    for (int i = 0; i < TC_NSLOT; ++i) mbar_init(sBar + B_EMPTY + 8 * i, 1);
    for (int i = 0; i < 4; ++i) mbar_init(sBar + B_FULL + 8 * i, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(sBar + B_SFULL + 8 * i, 1);
      mbar_init(sBar + B_PREADY + 8 * i, 128);
      mbar_init(sBar + B_OFINAL + 8 * i, 1);
    }
    mbar_init(sBar + B_DRAIN, 1);
    mbar_init(sBar + B_QFULL, 1);
    mbar_init(sBar + B_STALL, 1);
    *abort_flag = 0;
    fence_mbar_init();
    if (a.q_tma) {
      // Query tile r is rows f0 + 128r .. of the group: 128 / G positions
      // starting at chunk position (f0 + 128r) / G, G heads, three 64-dim parts.
      mbar_expect_tx(sBar + B_QFULL, nq * 3 * TC_SLOT);
      for (int r = 0; r < nq; ++r)
        for (int part = 0; part < 3; ++part)
          tma_load_3d(base + r * TC_QTILE + part * TC_SLOT, &tmq, 64 * part, kv * a.G,
                      (int)(crow0 + ((int)f0 + 128 * r) / a.G), sBar + B_QFULL);
    }
  }
  if (warp == 8) {
    tmem_alloc(sBar + B_TMEM, 512);
    tmem_relinquish();
  }
  // Q rows: CTA row r -> tile r / 128, TMEM lane r % 128; flat row f0 + r is
  // position (f0 + r) / G, head (f0 + r) % G of this KV head's group.
  // Byte offset of 16-byte chunk ch (0..23) of CTA row r (128-byte swizzle).
  auto q_chunk = [&](int r, int ch) {
    const int t = r & 127;
    return (uint32_t)((r >> 7) * TC_QTILE + (ch >> 3) * TC_SLOT + t * 128 + (((ch & 7) ^ (t & 7)) << 4));
  };
  // (f0 + r < nrows < 2^31: 32-bit index math)
  auto q_row = [&](int r, bool &live) {
    const int f = (int)f0 + r;
    live = f < (int)nrows;
    const int i = live ? f / a.G : 0;
    const int g = live ? f - i * a.G : 0;
    return qc + ((long long)i * a.hq + kv * a.G + g) * DQK;
  };
  constexpr int NB = (256 * 4 + TC_THREADS - 1) / TC_THREADS;  // (row, chunk pair) items per thread
  if (a.q_tma) {
    // The boxes bring every dim; dims 0..63 are then rotated in place, the
    // table rows fetched while the boxes land.  Rows past the chunk keep what
    // the boxes brought (finite values; their outputs are never stored).
    float4 tv[NB][4];
    bool liv[NB];
#pragma unroll
    for (int k = 0; k < NB; ++k) {
      const int it = tid + k * TC_THREADS;
      const int r = it >> 2, c = it & 3;
      liv[k] = it < nq * 128 * 4 && (int)f0 + r < (int)nrows;
      if (liv[k]) {
        const float4 *tr = reinterpret_cast<const float4 *>(a.table + (P0 + ((int)f0 + r) / a.G) * 64 + 16 * c);
#pragma unroll
        for (int u = 0; u < 4; ++u) tv[k][u] = tr[u];
      }
    }
    __syncthreads();  // the barrier's initialisation is visible
    if (mbar_wait(sBar + B_QFULL, 0, abort_flag)) {
#pragma unroll
      for (int k = 0; k < NB; ++k) {
        if (!liv[k]) continue;
        const int it = tid + k * TC_THREADS;
        const int r = it >> 2, c = it & 3;
        float cs[16];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          cs[4 * u] = tv[k][u].x; cs[4 * u + 1] = tv[k][u].y; cs[4 * u + 2] = tv[k][u].z; cs[4 * u + 3] = tv[k][u].w;
        }
        uint4 *p1 = reinterpret_cast<uint4 *>(gbase + q_chunk(r, c));
        uint4 *p2 = reinterpret_cast<uint4 *>(gbase + q_chunk(r, c + 4));
        uint4 o1, o2;
        rope_pair8(*p1, *p2, cs, o1, o2);
        *p1 = o1;
        *p2 = o2;
      }
    }
  } else {
    // Dims 64..191 pass through: asynchronous 16-byte copies (zero-filled
    // past the chunk), all in flight at once.
    for (int it = tid; it < nq * 128 * 16; it += TC_THREADS) {
      const int r = it >> 4, ch = 8 + (it & 15);
      bool live;
      const uint16_t *qh = q_row(r, live);
      cp_async16(base + q_chunk(r, ch), live ? qh + ch * 8 : qc, live ? 16 : 0);
    }
    cp_async_commit();
    // Dims 0..63: rotate-half with the table row of the position, four
    // (row, chunk pair) items per thread, loads issued before any use.
    uint4 x1[NB], x2[NB];
    float4 tv[NB][4];
#pragma unroll
    for (int k = 0; k < NB; ++k) {
      const int it = tid + k * TC_THREADS;
      const int r = it >> 2, c = it & 3;
      bool live = false;
      const uint16_t *qh = q_row(r < nq * 128 ? r : 0, live);
      live = live && it < nq * 128 * 4;
      x1[k] = x2[k] = make_uint4(0, 0, 0, 0);
      tv[k][0] = tv[k][1] = tv[k][2] = tv[k][3] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (live) {
        const uint4 *s4 = reinterpret_cast<const uint4 *>(qh);
        x1[k] = s4[c];
        x2[k] = s4[c + 4];
        const float4 *tr = reinterpret_cast<const float4 *>(a.table + (P0 + ((int)f0 + r) / a.G) * 64 + 16 * c);
#pragma unroll
        for (int u = 0; u < 4; ++u) tv[k][u] = tr[u];
      }
    }
#pragma unroll
    for (int k = 0; k < NB; ++k) {
      const int it = tid + k * TC_THREADS;
      if (it < nq * 128 * 4) {
        const int r = it >> 2, c = it & 3;
        float cs[16];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          cs[4 * u] = tv[k][u].x; cs[4 * u + 1] = tv[k][u].y; cs[4 * u + 2] = tv[k][u].z; cs[4 * u + 3] = tv[k][u].w;
        }
        uint4 o1, o2;
        rope_pair8(x1[k], x2[k], cs, o1, o2);  // zero in, zero out for rows past the chunk
        *reinterpret_cast<uint4 *>(gbase + q_chunk(r, c)) = o1;
        *reinterpret_cast<uint4 *>(gbase + q_chunk(r, c + 4)) = o2;
      }
    }
  }
  cp_async_wait<0>();
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  bool all_held = false;  // windowed: every ring slot holds its window position
  if constexpr (WINDOW) {
    const uint32_t *held = reinterpret_cast<const uint32_t *>(gbase + TC_OFF_TAG);
    all_held = (held[0] & held[1] & held[2] & held[3]) == 0xffffffffu;
  }
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(gbase + TC_OFF_BAR + B_TMEM);

  if (warp == 9) {
    // ------------------------------------------------------------ TMA producer
    // The whole warp runs the loop (converged); elect.sync issues.  Lane b
    // holds the tensor-map row of box b of a key tile; the next tile's rows
    // are fetched (block table) while the current tile's loads go out.
    const int low = a.bsz & -a.bsz;
    const int rb = low < 128 ? low : 128;      // rows per box: divides the page size and 128
    const int nb = 128 / rb;
    const int total = (int)a.total_rows;       // < 2^31, checked by the launcher
    const int khi = (int)k_hi, klo = (int)k_lo;
    auto box_row = [&](int t) {
      int y = total;                           // past the end: the TMA unit fills zeros
      if (lane < nb) {
        const int key = klo + 128 * t + lane * rb;
        if (key < khi) {
          const int blk = bt[key / a.bsz];
          if (blk >= 0 && blk < a.num_blocks)
            y = (blk * a.hkv + kv) * a.bsz + key % a.bsz;
          else
            flag(a.status, ST_BAD_BLOCK);
        }
      }
      return y;
    };
    int y_next = WINDOW ? 0 : box_row(0);
    long long L = 0;
    bool ok = true;
    const int ring_row = (rseq * a.hkv + kv) * WIN;  // windowed: the (sequence, KV head) ring
    for (int t = 0; t < ntiles && ok; ++t) {
      const int y_cur = y_next;
      if (!WINDOW && t + 1 < ntiles) y_next = box_row(t + 1);
      const int u = u_lo + t;
      // Two transaction barriers per key tile (each double-buffered): its
      // three K loads and its two V loads.  A barrier's arrive + byte count
      // goes out once the first slot of its part is free; that slot was freed
      // by products issued after the wait on the same barrier for tile t-2,
      // so that phase is over.
      for (int part = 0; part < 5; ++part, ++L) {
        const int slot = (int)(L % TC_NSLOT);
        const uint32_t round = (uint32_t)(L / TC_NSLOT);
        if (!warp_wait(sBar + B_EMPTY + 8 * slot, (round & 1u) ^ 1u, abort_flag)) { ok = false; break; }
        const uint32_t full = sBar + B_FULL + 8 * ((part < 3 ? 0 : 2) + (t & 1));
        if (part == 0) mbar_expect_tx_elect(full, 3 * TC_SLOT);
        if (part == 3) mbar_expect_tx_elect(full, 2 * TC_SLOT);
        const int pi = part < 3 ? part : part - 3;
        if (WINDOW && u >= 0) {
          const void *map = part < 3 ? (const void *)&tmk2 : (const void *)&tmv2;
          tma_load_4d_elect(sRing + slot * TC_SLOT, map, 0, pi, kv, (int)(crow0 + 128LL * u), full);
        } else if (WINDOW) {
          const void *map = part < 3 ? (const void *)&tmk : (const void *)&tmv;
          tma_load_2d_elect(sRing + slot * TC_SLOT, map, 64 * pi, ring_row, full);
        } else {
          const void *map = part < 3 ? (const void *)&tmk : (const void *)&tmv;
          for (int b = 0; b < nb; ++b)
            tma_load_2d_elect(sRing + slot * TC_SLOT + b * rb * 128, map, 64 * pi, __shfl_sync(0xffffffffu, y_cur, b),
                              full);
        }
      }
    }
    // On an abort, let the loads already issued land before the CTA exits
    // (bounded by time only: the abort flag is already set).
    if (lane == 0 && L > 0) {
      volatile uint32_t local = 0;
      const long long tl = (L - 1) / 5;  // the last tile with a load issued, and the one before
      for (long long t = tl; t >= 0 && t >= tl - 1; --t) {
        for (int h = 0; h < 2; ++h) {
          if (h == 1 && 5 * t + 3 >= L) continue;  // its V loads were never issued
          local = 0;
          mbar_wait(sBar + B_FULL + 8 * (2 * h + (t & 1)), (uint32_t)(t >> 1) & 1u, &local, 1000000000ull);
        }
      }
    }
    __syncwarp();
  } else if (warp == 8) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop (converged, operands warp-uniform) and
    // elect.sync issues each MMA and commit.  Descriptors are precomputed and
    // advanced by adding address offsets >> 4.
    const uint32_t id_qk = idesc_bf16(128, 128, 0, 0);
    const uint32_t id_pv64 = idesc_bf16(128, 64, 0, 1);
    const uint32_t id_pv128 = idesc_bf16(128, 128, 0, 1);
    const uint64_t dq0 = sdesc_sw128(sQ0, 16, 1024), dq1 = sdesc_sw128(sQ1, 16, 1024);
    const uint64_t dring_k = sdesc_sw128(sRing, 16, 1024);
    const uint64_t dring_v = sdesc_sw128(sRing, TC_SLOT, 1024);  // LBO = next slot (the other value half)
    bool ok = true;
    auto slot_of = [](long long L) { return (uint32_t)(L % TC_NSLOT); };
    auto wait_k = [&](int t) {  // the three K loads of key tile t
      return warp_wait(sBar + B_FULL + 8 * (t & 1), (uint32_t)(t >> 1) & 1u, abort_flag);
    };
    auto wait_v = [&](int t) {  // the two V loads of key tile t
      return warp_wait(sBar + B_FULL + 8 * (2 + (t & 1)), (uint32_t)(t >> 1) & 1u, abort_flag);
    };
    // S_i = Q_i K(t)^T : 12 MMAs of K = 16 over three 64-dim slots.
    auto issue_S = [&](int i, int t, bool release) {
      const uint64_t dq = i ? dq1 : dq0;
      const uint32_t d = tmem + 128 * i;
      if (i == 0) {  // query tile 1 reads the same slots right after tile 0
        if (!wait_k(t)) { ok = false; return; }
        tc_fence_after();
      }
      for (int kb = 0; kb < 3; ++kb) {
        const long long L = 5LL * t + kb;
        const uint64_t a0 = dq + (uint64_t)((kb * TC_SLOT) >> 4);
        const uint64_t b0 = dring_k + (uint64_t)((slot_of(L) * TC_SLOT) >> 4);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_ss_elect(d, a0 + 2 * kk, b0 + 2 * kk, id_qk, (kb | kk) != 0);
        if (release) mma_commit_elect(sBar + B_EMPTY + 8 * slot_of(L));
      }
      mma_commit_elect(sBar + B_SFULL + 8 * i);
    };
    // O_i += P_i(t) V(t): 8 MMAs of K = 16 keys, N = 128 value dims when the
    // two value halves sit in adjacent slots, else two N = 64 passes.
    auto issue_PV = [&](int i, int t, bool release) {
      if (!warp_wait(sBar + B_PREADY + 8 * i, (uint32_t)t & 1u, abort_flag)) { ok = false; return; }
      const long long L0 = 5LL * t + 3;
      if (i == 0 && !wait_v(t)) { ok = false; return; }  // tile 1 reads them right after tile 0
      for (int db = 0; db < 2 && i == 0; ++db) {
        if (WINDOW && i == 0 && u_lo + t < 0 && !all_held) {
          // The ring tile: V rows of slots that hold no position of the
          // window may be stale or never written; zero them before the product.
          const uint32_t *held = reinterpret_cast<const uint32_t *>(gbase + TC_OFF_TAG);
          uint4 *g = reinterpret_cast<uint4 *>(gbase + TC_OFF_RING + slot_of(L0 + db) * TC_SLOT);
#pragma unroll 4
          for (int e = lane; e < 128 * 8; e += 32)
            if (!((held[e >> 8] >> ((e >> 3) & 31)) & 1u)) g[e] = make_uint4(0, 0, 0, 0);
          fence_proxy_async_smem();
          __syncwarp();
        }
        if (i == 0 && t == ntiles - 1 && k_lo + 128LL * t + 128 > k_hi) {
          // Rows past the last key may hold stale bytes of the page; P is 0
          // there, but 0 * NaN is not, so zero them before the product.
          const int first = (int)(k_hi - k_lo - 128LL * t);
          uint4 *g = reinterpret_cast<uint4 *>(gbase + TC_OFF_RING + slot_of(L0 + db) * TC_SLOT);
          for (int e = first * 8 + lane; e < 128 * 8; e += 32) g[e] = make_uint4(0, 0, 0, 0);
          fence_proxy_async_smem();
          __syncwarp();
        }
      }
      tc_fence_after();
      const uint32_t ap = tmem + 128 * i;
      const uint32_t d = tmem + 256 + 128 * i;
      const uint32_t s0 = slot_of(L0), s1 = slot_of(L0 + 1);
      const uint32_t acc0 = t > 0 ? 1u : 0u;
      if (s1 == s0 + 1) {
        const uint64_t b0 = dring_v + (uint64_t)((s0 * TC_SLOT) >> 4);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ts_elect(d, ap + 8 * kk, b0 + 128 * kk, id_pv128, kk > 0 ? 1u : acc0);
      } else {
#pragma unroll
        for (int db = 0; db < 2; ++db) {
          const uint64_t b0 = dring_v + (uint64_t)(((db ? s1 : s0) * TC_SLOT) >> 4);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts_elect(d + 64 * db, ap + 8 * kk, b0 + 128 * kk, id_pv64, kk > 0 ? 1u : acc0);
        }
      }
      if (release) {
        mma_commit_elect(sBar + B_EMPTY + 8 * s0);
        mma_commit_elect(sBar + B_EMPTY + 8 * s1);
      }
    };
    // With one live query tile, tile 0's products release the ring slots.
    const bool one = nq == 1;
    if (a.stall_ns && !warp_wait(sBar + B_STALL, 0, abort_flag, a.stall_ns)) ok = false;
    if (ok) issue_S(0, 0, one);
    if (ok && !one) issue_S(1, 0, true);
    for (int t = 1; t < ntiles && ok; ++t) {
      issue_PV(0, t - 1, one);
      if (ok) issue_S(0, t, one);
      if (ok && !one) issue_PV(1, t - 1, true);
      if (ok && !one) issue_S(1, t, true);
    }
    if (ok) issue_PV(0, ntiles - 1, one);
    if (ok) mma_commit_elect(sBar + B_OFINAL);
    if (ok && !one) issue_PV(1, ntiles - 1, true);
    if (ok && !one) mma_commit_elect(sBar + B_OFINAL + 8);
    // Every MMA issued must be finished before TMEM is released (bounded by
    // time only, even after an abort).
    mma_commit_elect(sBar + B_DRAIN);
    if (lane == 0) {
      volatile uint32_t local = 0;
      mbar_wait(sBar + B_DRAIN, 0, &local, 1000000000ull);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax (warps 0-7)
    const int wg = warp >> 2;
    const int row = tid & 127;                       // TMEM lane = row of the tile
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t tS = tmem + lane_base + 128 * wg;
    const uint32_t tO = tmem + lane_base + 256 + 128 * wg;
    const long long f = f0 + 128 * wg + row;
    const bool live = f < nrows;
    const long long fc = live ? f : nrows - 1;
    const long long pr = P0 + fc / a.G;
    const int g = (int)(fc % a.G);
    const float sl2 = a.scale_log2;
    float m_ref = NEG_INF, l = 0.f;
    if constexpr (WINDOW) {  // the sink starts the softmax: e^{sink - m} = 1 in the denominator
      m_ref = a.sinks[kv * a.G + g] * LOG2E;
      l = 1.f;
    }
    bool ok = wg < nq;
    for (int t = 0; t < ntiles && ok; ++t) {
      if (!warp_wait(sBar + B_SFULL + 8 * wg, (uint32_t)t & 1u, abort_flag)) { ok = false; break; }
      tc_fence_after();
      uint32_t s[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, s[c]);
      tmem_wait_ld();
      const long long j0 = k_lo + 128LL * t;
      if constexpr (WINDOW) {
        const int ii = (int)(pr - P0);  // this row's offset in the chunk
        if (u_lo + t < 0) {
          // The ring: slot c is position P0 - 128 + k, k = (c - P0) mod 128,
          // inside this row's window iff k > ii, and present iff its bit is set.
          const uint32_t *held = reinterpret_cast<const uint32_t *>(gbase + TC_OFF_TAG);
          const int pm = (int)(P0 & (WIN - 1));
          if (all_held) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (((32 * c + e - pm) & (WIN - 1)) <= ii) s[c][e] = __float_as_uint(NEG_INF);
          } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint32_t hb = held[c];
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (!((hb >> e) & 1u) || ((32 * c + e - pm) & (WIN - 1)) <= ii) s[c][e] = __float_as_uint(NEG_INF);
            }
          }
        } else {
          // Chunk rows 128u + col: inside the window iff ii - 128 < 128u + col <= ii.
          const int d = ii - 128 * (u_lo + t);
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (32 * c + e > d || 32 * c + e <= d - WIN) s[c][e] = __float_as_uint(NEG_INF);
        }
      } else if (j0 + 127 > pmin) {  // the diagonal (and the end of the keys) is in this tile
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (j0 + 32 * c + e > pr) s[c][e] = __float_as_uint(NEG_INF);
      }
      // Row max with eight independent chains.
      float mxv[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) mxv[u] = NEG_INF;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          mxv[(e >> 1) & 7] = fmax3(mxv[(e >> 1) & 7], __uint_as_float(s[c][e]), __uint_as_float(s[c][e + 1]));
      const float mx = fmaxf(fmaxf(fmaxf(mxv[0], mxv[1]), fmaxf(mxv[2], mxv[3])),
                             fmaxf(fmaxf(mxv[4], mxv[5]), fmaxf(mxv[6], mxv[7])));
      const float m_new = fmaxf(m_ref, mx * sl2);
      float factor = 1.f;
      bool resc = false;
      if (m_ref == NEG_INF) {
        m_ref = m_new;  // nothing accumulated yet (all earlier P were 0)
      } else if (m_new > m_ref + RESCALE_THRESHOLD) {
        factor = ex2(m_ref - m_new);
        m_ref = m_new;
        resc = true;
      }
      const float b = m_ref == NEG_INF ? 0.f : m_ref;
      // p = 2^(s * scale - b), two elements per packed FMA; row sums in
      // four packed accumulators
      uint64_t sumv[4] = {0, 0, 0, 0};  // (+0.0f, +0.0f) pairs
      uint32_t pk[2][32];
      const uint64_t sl2v = f32x2(sl2, sl2), nbv = f32x2(-b, -b);
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float a0, a1;
          f32x2_split(fma_f32x2(f32x2(__uint_as_float(s[c][e]), __uint_as_float(s[c][e + 1])), sl2v, nbv), a0, a1);
          const float p0 = ex2(a0), p1 = ex2(a1);
          sumv[(e >> 1) & 3] = add_f32x2(sumv[(e >> 1) & 3], f32x2(p0, p1));
          pk[c >> 1][(c & 1) * 16 + e / 2] = pack_bf16(p0, p1);
        }
      float su[8];
#pragma unroll
      for (int u = 0; u < 4; ++u) f32x2_split(sumv[u], su[2 * u], su[2 * u + 1]);
      l = l * factor + (((su[0] + su[1]) + (su[2] + su[3])) + ((su[4] + su[5]) + (su[6] + su[7])));
      tmem_st32(tS, pk[0]);
      tmem_st32(tS + 32, pk[1]);
      if (__any_sync(0xffffffffu, resc)) {
        // O is quiescent: its last product finished before S(t) did, and the
        // next one waits for this tile's P.
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + 32 * c, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * factor);
          tmem_st32(tO + 32 * c, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(sBar + B_PREADY + 8 * wg);
    }
    if (ok) ok = warp_wait(sBar + B_OFINAL + 8 * wg, 0, abort_flag);
    // The TMA epilogue needs all four warps of the group: they agree first
    // (every warp reaches this barrier, whatever its own outcome).
    bool box_store = false;
    if constexpr (!VARLEN) {
      if (a.o_tma) box_store = named_bar_and(1 + wg, 128, ok);
    }
    if (ok && nsp > 1) {
      // One split of the keys: the unnormalised numerator, the max (log2
      // units) and the sum, merged later by varlen_combine_kernel.
      tc_fence_after();
      const long long rec = (prow + (pr - P0) * a.hq + (long long)kv * a.G + g) * a.plan.nsp_max + split;
      if (live) a.plan.pml[rec] = make_float2(m_ref, l);
      float4 *dst = reinterpret_cast<float4 *>(a.plan.po + rec * DV);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + 32 * c, o);
        tmem_wait_ld();
        if (live) {
#pragma unroll
          for (int u = 0; u < 8; ++u)
            dst[8 * c + u] = make_float4(__uint_as_float(o[4 * u]), __uint_as_float(o[4 * u + 1]),
                                         __uint_as_float(o[4 * u + 2]), __uint_as_float(o[4 * u + 3]));
        }
      }
    } else if (box_store) {
      // One chunk: every row of the tile inside the output tensor is live, so
      // the tile goes out as two TMA boxes (dims 0-63, 64-127) staged in its
      // query region, which no product reads once O is final.
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const uint32_t stage = base + wg * TC_QTILE;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + 32 * c, o);
        tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t w0 = pack_bf16(__uint_as_float(o[8 * u + 0]) * inv, __uint_as_float(o[8 * u + 1]) * inv);
          const uint32_t w1 = pack_bf16(__uint_as_float(o[8 * u + 2]) * inv, __uint_as_float(o[8 * u + 3]) * inv);
          const uint32_t w2 = pack_bf16(__uint_as_float(o[8 * u + 4]) * inv, __uint_as_float(o[8 * u + 5]) * inv);
          const uint32_t w3 = pack_bf16(__uint_as_float(o[8 * u + 6]) * inv, __uint_as_float(o[8 * u + 7]) * inv);
          const int ch = 4 * (c & 1) + u;  // 16-byte chunk of dims 8 * ch .. within the part
          *reinterpret_cast<uint4 *>(gbase + wg * TC_QTILE + (c >> 1) * TC_SLOT + row * 128 +
                                     ((ch ^ (row & 7)) << 4)) = make_uint4(w0, w1, w2, w3);
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(1 + wg, 128);
      if (row == 0) {
        const int pos0 = (int)(crow0 + ((int)f0 + 128 * wg) / a.G);
        tma_store_3d(&tmo, 0, kv * a.G, pos0, stage);
        tma_store_3d(&tmo, 64, kv * a.G, pos0, stage + TC_SLOT);
        bulk_commit();
        bulk_wait_read_all();  // the staging area stays valid until read
      }
    } else if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint16_t *orow = oc + ((pr - P0) * a.hq + (long long)kv * a.G + g) * DV;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + 32 * c, o);
        tmem_wait_ld();
        if (live) {
          uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * c);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(o[8 * u + 0]) * inv, __uint_as_float(o[8 * u + 1]) * inv);
            w.y = pack_bf16(__uint_as_float(o[8 * u + 2]) * inv, __uint_as_float(o[8 * u + 3]) * inv);
            w.z = pack_bf16(__uint_as_float(o[8 * u + 4]) * inv, __uint_as_float(o[8 * u + 5]) * inv);
            w.w = pack_bf16(__uint_as_float(o[8 * u + 6]) * inv, __uint_as_float(o[8 * u + 7]) * inv);
            dst[u] = w;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag && tid == 0) {
    flag(a.status, ST_TIMEOUT);
    if (a.q_tma) {  // the query boxes must have landed before the CTA leaves (time bound only)
      volatile uint32_t local = 0;
      mbar_wait(sBar + B_QFULL, 0, &local, 1000000000ull);
    }
  }
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

namespace {

// Tensor maps of the pool and the common kernel arguments.
cudaError_t tc_setup(const KvView &pool, int hq, const float *table, float softmax_scale, uint16_t *out,
                     unsigned *status, CUtensorMap *mk, CUtensorMap *mv, TcArgs *a) {
  const int hkv = pool.hkv;
  const long long rows = (long long)pool.num_blocks * hkv * pool.block_size;
  if (rows >= (1LL << 31)) return cudaErrorInvalidValue;
  const int low = pool.block_size & -pool.block_size;
  const int box_rows = low < 128 ? low : 128;
  if (!make_tma_map_2d(mk, pool.k, rows, DQK, box_rows) || !make_tma_map_2d(mv, pool.v, rows, DV, box_rows))
    return cudaErrorInvalidValue;
  *a = TcArgs{};
  a->hq = hq;
  a->G = hq / hkv;
  a->hkv = hkv;
  a->bt = pool.block_table;
  a->bsz = pool.block_size;
  a->num_blocks = pool.num_blocks;
  a->max_blocks = pool.max_blocks;
  a->total_rows = rows;
  a->table = table;
  a->scale_log2 = softmax_scale * LOG2E;
  a->stall_ns = 0;
  a->out = out;
  a->status = status;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_full_prefill(const uint16_t *q, int64_t P0, int C, int seq, int hq, const KvView &pool,
                                const float *table, int64_t max_pos, float softmax_scale, uint16_t *out,
                                unsigned *status, cudaStream_t st) {
  (void)max_pos;
  CUtensorMap mk, mv;
  TcArgs a;
  cudaError_t e = tc_setup(pool, hq, table, softmax_scale, out, status, &mk, &mv, &a);
  if (e != cudaSuccess) return e;
  e = ensure_smem_limit(2, (const void *)full_prefill_tc_kernel<false, false>, TC_SMEM);
  if (e != cudaSuccess) return e;
  a.q = q;
  a.P0 = P0;
  a.C = C;
  a.bt = pool.block_table + (long long)seq * pool.max_blocks;
  a.stall_ns = take_stall();
  CUtensorMap mq, mo;
  a.q_tma = make_tma_map_heads3d(&mq, q, C, hq, DQK, a.G) ? 1 : 0;
  a.o_tma = make_tma_map_heads3d(&mo, out, C, hq, DV, a.G) ? 1 : 0;
  const long long ctas = ((long long)C * a.G + 255) / 256 * a.hkv;
  full_prefill_tc_kernel<false, false><<<(unsigned)ctas, TC_THREADS, TC_SMEM, st>>>(
      mk, mv, mk, mv, a.q_tma ? mq : mk, a.o_tma ? mo : mk, a);
  return cudaGetLastError();
}

cudaError_t launch_full_varlen(const uint16_t *q, const int32_t *cu_rows, const int64_t *P0, const int32_t *seq,
                               int n, long long T, int hq, const KvView &pool, const float *table,
                               float softmax_scale, long long max_ctx, void *ws, uint16_t *out, unsigned *status,
                               cudaStream_t st) {
  CUtensorMap mk, mv;
  TcArgs a;
  cudaError_t e = tc_setup(pool, hq, table, softmax_scale, out, status, &mk, &mv, &a);
  if (e != cudaSuccess) return e;
  e = ensure_smem_limit(4, (const void *)full_prefill_tc_kernel<true, false>, TC_SMEM);
  if (e != cudaSuccess) return e;
  const VarlenSizes z = varlen_sizes(n, T, hq, pool.hkv, max_ctx, 256, true);
  a.q = q;
  a.plan = varlen_plan_view(z, ws, cu_rows, P0, seq, n);
  CUtensorMap mq;
  a.q_tma = make_tma_map_heads3d(&mq, q, T, hq, DQK, a.G) ? 1 : 0;
  e = launch_varlen_plan(a.plan, T, hq, pool.hkv, 256, max_ctx, pool.num_seqs, 0, 0, status, st);
  if (e != cudaSuccess) return e;
  full_prefill_tc_kernel<true, false><<<(unsigned)z.items_max, TC_THREADS, TC_SMEM, st>>>(
      mk, mv, mk, mv, a.q_tma ? mq : mk, mk, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_varlen_combine(a.plan, z.prows_max, hq, out, st);
}

namespace {

// Tensor maps of a windowed layer: the ring (128-row boxes of one 64-dim
// part) and the staged chunk rows (4-D boxes of 128 tokens of one KV head,
// one part), and the common arguments.
cudaError_t tc_window_setup(const KvView &chunk, long long T, const KvView &ring, int hq, const float *sinks,
                            const float *table, float softmax_scale, uint16_t *out, unsigned *status, CUtensorMap *m,
                            TcArgs *a) {
  const int hkv = ring.hkv;
  const long long rows = (long long)ring.num_seqs * hkv * WIN;
  if (rows >= (1LL << 31) || T >= (1LL << 31)) return cudaErrorInvalidValue;
  if (!make_tma_map_2d(&m[0], ring.k, rows, DQK, 128) || !make_tma_map_2d(&m[1], ring.v, rows, DV, 128) ||
      !make_tma_map_tokens4d(&m[2], chunk.k, T, hkv, DQK, 128, true) ||
      !make_tma_map_tokens4d(&m[3], chunk.v, T, hkv, DV, 128, true))
    return cudaErrorInvalidValue;
  *a = TcArgs{};
  a->hq = hq;
  a->G = hq / hkv;
  a->hkv = hkv;
  a->table = table;
  a->scale_log2 = softmax_scale * LOG2E;
  a->out = out;
  a->status = status;
  a->slot_pos = ring.slot_pos;
  a->sinks = sinks;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_swa_prefill_tc(const uint16_t *q, int64_t P0, int C, int seq, int hq, const KvView &chunk,
                                  const KvView &ring, const float *sinks, const float *table, float softmax_scale,
                                  uint16_t *out, unsigned *status, cudaStream_t st) {
  bool taken = false;
  cudaError_t e = launch_swa_band(q, P0, C, seq, hq, chunk, ring, sinks, table, softmax_scale, out, status, st,
                                  &taken);
  if (e != cudaSuccess || taken) return e;
  CUtensorMap m[4];
  TcArgs a;
  e = tc_window_setup(chunk, C, ring, hq, sinks, table, softmax_scale, out, status, m, &a);
  if (e != cudaSuccess) return e;
  e = ensure_smem_limit(7, (const void *)full_prefill_tc_kernel<false, true>, TC_SMEM);
  if (e != cudaSuccess) return e;
  a.q = q;
  a.P0 = P0;
  a.C = C;
  a.ring_seq = seq;
  CUtensorMap mq, mo;
  a.q_tma = make_tma_map_heads3d(&mq, q, C, hq, DQK, a.G) ? 1 : 0;
  a.o_tma = make_tma_map_heads3d(&mo, out, C, hq, DV, a.G) ? 1 : 0;
  const long long ctas = ((long long)C * a.G + 255) / 256 * a.hkv;
  full_prefill_tc_kernel<false, true><<<(unsigned)ctas, TC_THREADS, TC_SMEM, st>>>(
      m[0], m[1], m[2], m[3], a.q_tma ? mq : m[0], a.o_tma ? mo : m[0], a);
  return cudaGetLastError();
}

cudaError_t launch_swa_varlen(const uint16_t *q, const int32_t *cu_rows, const int64_t *P0, const int32_t *seq,
                              int n, long long T, int hq, const KvView &chunk, const KvView &ring,
                              const float *sinks, const float *table, int64_t max_pos, float softmax_scale,
                              void *ws, uint16_t *out, unsigned *status, cudaStream_t st) {
  const int hkv = ring.hkv;
  bool taken = false;
  cudaError_t e = launch_swa_band_varlen(q, cu_rows, P0, seq, n, T, hq, chunk, ring, sinks, table, max_pos,
                                         softmax_scale, ws, out, status, st, &taken);
  if (e != cudaSuccess || taken) return e;
  CUtensorMap m[4];
  TcArgs a;
  e = tc_window_setup(chunk, T, ring, hq, sinks, table, softmax_scale, out, status, m, &a);
  if (e != cudaSuccess) return e;
  e = ensure_smem_limit(8, (const void *)full_prefill_tc_kernel<true, true>, TC_SMEM);
  if (e != cudaSuccess) return e;
  const VarlenSizes z = varlen_sizes(n, T, hq, hkv, max_pos, 256, false);
  a.q = q;
  a.plan = varlen_plan_view(z, ws, cu_rows, P0, seq, n);
  CUtensorMap mq;
  a.q_tma = make_tma_map_heads3d(&mq, q, T, hq, DQK, a.G) ? 1 : 0;
  e = launch_varlen_plan(a.plan, T, hq, hkv, 256, max_pos, ring.num_seqs, SWA_SHORT_ROWS, SWA_SHORT_MAX_C, status,
                         st);
  if (e != cudaSuccess) return e;
  // Chunks of more than 32 query rows are tiled here; the short ones go to
  // the short-chunk kernel.
  full_prefill_tc_kernel<true, true><<<(unsigned)z.items_max, TC_THREADS, TC_SMEM, st>>>(
      m[0], m[1], m[2], m[3], a.q_tma ? mq : m[0], m[0], a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_swa_short(q, a.plan, n, T, hq, chunk, ring, sinks, table, softmax_scale, out, status, st);
}

}  // namespace kvr
