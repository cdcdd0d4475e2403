// decode.cu -- one-token decode over a full-attention layer: paged pool,
// split-K with a log-sum-exp combine.
//
// Math (colibri "MiMo-V2.6", "What the engine implements"): q is rotated on
// dims 0..63 with the table row of its position and rounded to bf16; s = q.k'
// scaled; softmax in the base-2 domain with fp32 state (m, l, o); no sink on
// full-attention layers.
// Decode is memory-bound (Xiaomi "Full-Pipeline Inference Optimization",
// section 1.2): every K/V byte is read once, through 16-byte cp.async copies
// into swizzled shared memory, and the two small products per key tile run
// on the bf16 tensor cores (mma.sync m16n8k16, fp32 accumulate) with the G
// query heads of one KV head as the 16 rows of the MMA.
//
// The same split kernel serves a windowed layer kept in pages (the paged SWA
// pool of Xiaomi section 2.1; gaudi-cookbook "Windowed KV groups"): the key
// range starts at p - 127 (rounded down to a 16-key subtile, the extra keys
// masked), one split covers it, and the kernel normalises directly with the
// sink in the denominator (colibri "What the engine implements").
#include <cuda.h>

#include "launch.h"
#include "tc_ptx.cuh"
#include "warp_attn.cuh"

namespace kvr {
namespace {

// ---------------------------------------------------------------------------
// Full layer, phase 1: persistent CTAs walk the plan's items (sequence,
// split, KV head) round-robin; each streams its key range through per-warp
// cp.async pipelines of 16-key subtiles and writes fp32 partials.

constexpr unsigned ST_TIMEOUT = 8u;  // KVR_DEV_TIMEOUT
constexpr int FD_WARPS = 4;
constexpr int FD_STAGES = 2;
constexpr int FD_SUB_K = 16 * DQK * 2;                 // 6144 B
constexpr int FD_SUB_V = 16 * DV * 2;                  // 4096 B
constexpr int FD_STAGE = FD_SUB_K + FD_SUB_V;          // 10240 B
// Windowed layer in pages: a window of WIN keys starting anywhere covers at
// most FDW_SUBS 16-key subtiles, each with a stage of its own, so the whole
// window is requested at once (at most FDW_AHEAD subtiles per warp), by TMA.
constexpr int FDW_SUBS = WIN / 16 + 1;
constexpr int FDW_AHEAD = (FDW_SUBS + FD_WARPS - 1) / FD_WARPS;
constexpr int FDW_NB = 16;
// head of the shared memory: the query tile, the table row, then (windowed
// layer) the next item's block ids, one mbarrier per stage and the abort flag
constexpr int FD_OFF_CS = 16 * DQK * 2;
constexpr int FD_OFF_NB = FD_OFF_CS + 256;
constexpr int FD_OFF_BAR = FD_OFF_NB + FDW_NB * 4;
constexpr int FD_OFF_ABORT = FD_OFF_BAR + 8 * FDW_SUBS;
constexpr int FD_HEAD = (FD_OFF_ABORT + 4 + 127) / 128 * 128;
constexpr int FD_SMEM = FD_HEAD + FD_WARPS * FD_STAGES * FD_STAGE;
// (the TMA stages start on the next 1024-byte boundary, as the 128-byte swizzle wants)
constexpr int FDW_SMEM = FD_HEAD + 1024 + FDW_SUBS * FD_STAGE;
// a window's keys (at most WIN + 15 from its 16-key aligned start) over
// blocks of at least 16 keys
static_assert((WIN + 15 + 15) / 16 + 1 <= FDW_NB, "block ids of one window");
// split plan (see full_decode_plan_kernel): the fixed cost of an item in keys,
// the longest split, and where the per-sequence item prefix starts in the
// plan (after L and the item count, 256-byte aligned)
constexpr long long FD_ITEM_KEYS = 300;
constexpr long long FD_MAX_LEN = 8192 + 256;
constexpr int DPLAN_PREFIX = 64;

// Full layer, phase 0: the split plan, from the batch's own contexts (one
// CTA).  The split kernel is persistent with R = 2 CTAs per SM taking items
// round-robin, so a CTA does ceil(items / R) items of up to L keys, each with
// a fixed cost (query tile, pipeline fill, partial-state store) worth about
// FD_ITEM_KEYS keys.  Candidate split lengths: those giving about k items per
// resident CTA (k = 1..8) for the longest context alone, and for the batch's
// total keys; capped at FD_MAX_LEN keys, at least 64.  The plan takes the
// candidate minimising ceil(items / R) * (L + that cost) with the batch's
// real item count (ties: fewer items), then writes L, the item count and the
// per-sequence item prefix.  Sequences with a bad position or id get no items
// (flagged here; the merge zeroes their rows).
constexpr int DP_CANDS = 16;
constexpr int DP_INLINE_MAX = 4096;
constexpr int FD_EARLY_KEYS = 256;   // keys of a CTA's first item prefetched before the wait (B <= 32)  // batches the split kernel plans itself (prefix in shared memory)

// The plan by one CTA of NT threads: the split length (returned), the item
// count (*nitems) and the per-sequence item prefix (prefix[0..B]).  Flags bad
// entries when `status` is not null.
template <int NT>
__device__ int decode_plan_block(const int64_t *__restrict__ pos, const int32_t *__restrict__ seq, int B, int hkv,
                                 int num_seqs, int64_t max_pos, long long max_ctx, int R, int32_t *prefix,
                                 int *nitems, unsigned *status) {
  constexpr int NW = NT / 32;
  __shared__ long long s_tot[NW], s_mx[NW];
  __shared__ int s_cnt[NW][DP_CANDS];
  __shared__ int s_scan[NW];
  __shared__ int s_L;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  auto ctx_of = [&](int b) -> long long {
    const long long p = pos[b];
    const int s = seq[b];
    return (p >= 0 && p < max_pos && p + 1 <= max_ctx && s >= 0 && s < num_seqs) ? p + 1 : 0;
  };
  // 1. total keys, longest context, bad entries
  long long tot = 0, mx = 0;
  unsigned bad = 0;
  for (int b = tid; b < B; b += NT) {
    const long long p = pos[b];
    const int s = seq[b];
    const bool bp = p < 0 || p >= max_pos || p + 1 > max_ctx, bs = s < 0 || s >= num_seqs;
    if (bp || bs) {
      bad |= (bp ? ST_BAD_POS : 0u) | (bs ? ST_BAD_SEQ : 0u);
    } else {
      tot += p + 1;
      mx = p + 1 > mx ? p + 1 : mx;
    }
  }
  if (bad && status) flag(status, bad);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    tot += __shfl_xor_sync(0xffffffffu, tot, o);
    const long long y = __shfl_xor_sync(0xffffffffu, mx, o);
    mx = y > mx ? y : mx;
  }
  if (lane == 0) {
    s_tot[warp] = tot;
    s_mx[warp] = mx;
  }
  __syncthreads();
  tot = 0;
  mx = 0;
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    tot += s_tot[i];
    mx = s_mx[i] > mx ? s_mx[i] : mx;
  }
  // 2. candidate split lengths: lane c of every warp derives candidate c and
  // the warp shares them by shuffles (GB300's FP64 rate is a small fraction of
  // its integer rate, so no double arithmetic here; one 64-bit division per
  // lane, the rest in 32 bits as contexts and split lengths fit)
  unsigned mine_L;
  {
    const unsigned k = lane % 8 + 1;
    unsigned L;
    if (lane < 8) {  // about k items per resident CTA for the longest context
      unsigned n = k * (unsigned)R / ((unsigned)B * (unsigned)hkv);
      if (n < 1) n = 1;
      L = ((unsigned)mx + n - 1) / n;
    } else {         // ... for the batch's total keys
      const unsigned long long d = (unsigned long long)k * (unsigned)R;
      const unsigned long long l = ((unsigned long long)tot * (unsigned)hkv + d - 1) / d;
      L = l > (unsigned long long)FD_MAX_LEN ? (unsigned)FD_MAX_LEN : (unsigned)l;
    }
    L = (L + 63) / 64 * 64;
    mine_L = L < 64 ? 64u : (L > (unsigned)FD_MAX_LEN ? (unsigned)FD_MAX_LEN : L);
  }
  unsigned cand[DP_CANDS];
#pragma unroll
  for (int c = 0; c < DP_CANDS; ++c) cand[c] = __shfl_sync(0xffffffffu, mine_L, c);
  // 3. items of every candidate, one combined reduction
  int cnt[DP_CANDS];
#pragma unroll
  for (int c = 0; c < DP_CANDS; ++c) cnt[c] = 0;
  for (int b = tid; b < B; b += NT) {
    const unsigned ctx = (unsigned)ctx_of(b);
#pragma unroll
    for (int c = 0; c < DP_CANDS; ++c) cnt[c] += (int)((ctx + cand[c] - 1) / cand[c]);
  }
#pragma unroll
  for (int c = 0; c < DP_CANDS; ++c) cnt[c] = __reduce_add_sync(0xffffffffu, cnt[c]);
  if (lane == 0) {
#pragma unroll
    for (int c = 0; c < DP_CANDS; ++c) s_cnt[warp][c] = cnt[c];
  }
  __syncthreads();
  // 4. choose: the least cost, ties to fewer items (one thread: measured
  // quicker here than a warp-wide argmin)
  if (tid == 0) {
    unsigned best_L = (unsigned)FD_MAX_LEN, best_items = 0;
    long long best_cost = -1;
    for (int c = 0; c < DP_CANDS; ++c) {
      unsigned items = 0;
      for (int i = 0; i < NW; ++i) items += (unsigned)s_cnt[i][c];
      items *= (unsigned)hkv;
      const long long cost = (long long)((items + (unsigned)R - 1) / (unsigned)R) * (cand[c] + FD_ITEM_KEYS);
      if (best_cost < 0 || cost < best_cost || (cost == best_cost && items < best_items)) {
        best_cost = cost;
        best_L = cand[c];
        best_items = items;
      }
    }
    s_L = (int)best_L;
  }
  __syncthreads();
  const unsigned L = (unsigned)s_L;
  // 5. per-sequence item prefix (exclusive scan, NT sequences at a time)
  int running = 0;
  for (int b0 = 0; b0 < B; b0 += NT) {
    const int b = b0 + tid;
    const int mine = b < B ? (int)(((unsigned)ctx_of(b) + L - 1) / L) * hkv : 0;
    int x = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_scan[warp] = x;
    __syncthreads();
    int before = 0, all = 0;
#pragma unroll
    for (int i = 0; i < NW; ++i) {
      before += i < warp ? s_scan[i] : 0;
      all += s_scan[i];
    }
    if (b < B) prefix[b] = running + before + x - mine;
    running += all;
    __syncthreads();  // s_scan is rewritten by the next round
  }
  if (tid == 0) prefix[B] = running;
  *nitems = running;
  return (int)L;
}

// The same plan made by one warp for a batch of at most 32 sequences (lane b
// is sequence b): warp reductions and shuffles only, no block barrier.  Ties
// between candidates of equal cost go to the lower candidate index.  The
// split length and the item count go to prefix[B + 1] and prefix[B + 2].
// Lane b < B passes sequence b's position p and id s (the other lanes
// anything).
__device__ void decode_plan_warp(long long p, int s, int B, int hkv,
                                 int num_seqs, int64_t max_pos, long long max_ctx, int R, int32_t *prefix,
                                 unsigned *status) {
  constexpr unsigned FULL = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  unsigned ctx = 0, bad = 0;
  if (lane < B) {
    const bool bp = p < 0 || p >= max_pos || p + 1 > max_ctx, bs = s < 0 || s >= num_seqs;
    if (bp || bs)
      bad = (bp ? ST_BAD_POS : 0u) | (bs ? ST_BAD_SEQ : 0u);
    else
      ctx = (unsigned)(p + 1);
  }
  if (bad && status) flag(status, bad);
  const unsigned mx = __reduce_max_sync(FULL, ctx);
  const unsigned long long tot = ((unsigned long long)__reduce_add_sync(FULL, ctx >> 16) << 16) +
                                 __reduce_add_sync(FULL, ctx & 0xffffu);
  // candidate `lane` (lanes 0 .. 15), as in decode_plan_block
  unsigned mine_L;
  {
    const unsigned k = lane % 8 + 1;
    unsigned L;
    if (lane < 8) {
      unsigned n = k * (unsigned)R / ((unsigned)B * (unsigned)hkv);
      if (n < 1) n = 1;
      L = (mx + n - 1) / n;
    } else {
      const unsigned long long d = (unsigned long long)k * (unsigned)R;
      const unsigned long long l = (tot * (unsigned)hkv + d - 1) / d;
      L = l > (unsigned long long)FD_MAX_LEN ? (unsigned)FD_MAX_LEN : (unsigned)l;
    }
    L = (L + 63) / 64 * 64;
    mine_L = L < 64 ? 64u : (L > (unsigned)FD_MAX_LEN ? (unsigned)FD_MAX_LEN : L);
  }
  unsigned items_mine = 0;  // items of candidate `lane`
#pragma unroll
  for (int c = 0; c < DP_CANDS; ++c) {
    const unsigned L = __shfl_sync(FULL, mine_L, c);
    const unsigned n = __reduce_add_sync(FULL, (ctx + L - 1) / L);
    if (lane == c) items_mine = n * (unsigned)hkv;
  }
  unsigned key = FULL;
  if (lane < DP_CANDS) {
    unsigned cost = (items_mine + (unsigned)R - 1) / (unsigned)R * (mine_L + FD_ITEM_KEYS);
    cost = cost > 0x7ffffffu ? 0x7ffffffu : cost;
    key = (cost << 4) | (unsigned)lane;
  }
  const unsigned L = __shfl_sync(FULL, mine_L, (int)(__reduce_min_sync(FULL, key) & 15u));
  // per-sequence item prefix
  const int mine = lane < B ? (int)((ctx + L - 1) / L) * hkv : 0;
  int x = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(FULL, x, o);
    if (lane >= o) x += y;
  }
  if (lane < B) prefix[lane] = x - mine;
  if (lane == 31) {
    prefix[B] = x;
    prefix[B + 1] = (int)L;
    prefix[B + 2] = x;
  }
}

static_assert(FD_WARPS * FD_STAGES * FD_STAGE >= (FD_WARPS * 16 * (MO_STRIDE + 2) + FD_WARPS * 16) * 4, "merge area");
static_assert(FDW_SUBS * FD_STAGE >= (FD_WARPS * 16 * (MO_STRIDE + 2) + FD_WARPS * 16) * 4, "merge area");

// WINDOW = false: a full layer (keys 0..p, split partials to the workspace);
// true: a windowed layer kept in pages (keys p-127..p, one split, direct
// normalised output with the sink).  Separate instantiations keep the full
// layer's issue path free of the window's per-row checks.
template <bool WINDOW>
__global__ void __launch_bounds__(FD_WARPS * 32, 2)
    full_decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                       const uint16_t *__restrict__ q, const int64_t *__restrict__ pos,
                       const int32_t *__restrict__ seq, int B, int hq, int G, KvView pool,
                       const float *__restrict__ table, int64_t max_pos, float scale_log2,
                       long long max_ctx, const int32_t *__restrict__ plan, int split_len,
                       float *__restrict__ part_ml, float *__restrict__ part_o, unsigned *status, int window,
                       const float *__restrict__ sinks, uint16_t *__restrict__ out_direct) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int32_t *prefix = plan + DPLAN_PREFIX;
  long long pe = 0;  // full layer, B <= 32, warp 0: lane b's early copy of pos[b] (and seq[b])
  int se = 0;
  if (!WINDOW && B <= 32 && threadIdx.x < 32) {
    // Ahead of the wait for the kernel before this one (which may still
    // run): the plan from positions and sequence ids read early (see
    // ld_early_s32), and the first keys of this CTA's first item requested
    // into L2, so the DRAM streams while the kernel ahead drains.  After the
    // wait the plan is kept only if every position and id reads the same.
    const int lane = threadIdx.x;
    int32_t *sPrefix = reinterpret_cast<int32_t *>(smem + FD_SMEM);
    if (lane < B) {
      pe = ld_early_s64(pos + lane);
      se = ld_early_s32(seq + lane);
    }
    decode_plan_warp(pe, se, B, pool.hkv, pool.num_seqs, max_pos, max_ctx, gridDim.x, sPrefix, nullptr);
    __syncwarp();
    const int L = sPrefix[B + 1];
    if ((int)blockIdx.x < sPrefix[B + 2]) {
      const int b = plan_find(sPrefix, B, blockIdx.x);
      const int local = (int)blockIdx.x - sPrefix[b], split = local / pool.hkv, kv = local % pool.hkv;
      const long long p = __shfl_sync(0xffffffffu, pe, b);  // (a sequence with items has a valid p and id)
      const int sq = __shfl_sync(0xffffffffu, se, b), bsz = pool.block_size;
      const long long k0 = (long long)split * L, k1 = min(k0 + min(L, FD_EARLY_KEYS), p + 1) - 1;
      const long long blk0 = k0 / bsz;
      if (lane <= k1 / bsz - blk0) {
        const int blk = ld_early_s32(pool.block_table + (long long)sq * pool.max_blocks + blk0 + lane);
        if (blk >= 0 && blk < pool.num_blocks) {
          const long long first = (blk0 + lane) * bsz;
          const long long r0 = max(k0, first), r1 = min(k1, first + bsz - 1);
          const long long hrow = ((long long)blk * pool.hkv + kv) * bsz + (r0 - first);
          prefetch_l2(pool.k + hrow * DQK, (uint32_t)(r1 - r0 + 1) * DQK * 2);
          prefetch_l2(pool.v + hrow * DV, (uint32_t)(r1 - r0 + 1) * DV * 2);
        }
      }
      if (lane == 31) prefetch_l2(q + ((long long)b * hq + (long long)kv * G) * DQK, G * DQK * 2);
    }
  }
  // launched as a programmatic dependent (launch_pdl); the merge kernel after
  // it may be scheduled as its CTAs leave and reads nothing of this kernel's
  // before this kernel has completed
  pdl_wait();
  pdl_trigger();
  uint8_t *sQ = smem;
  uint8_t *sCS = smem + FD_OFF_CS;
  int32_t *sNB = reinterpret_cast<int32_t *>(smem + FD_OFF_NB);
  const uint32_t sBar = smem_u32(smem + FD_OFF_BAR);
  volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + FD_OFF_ABORT);
  uint8_t *sStage = WINDOW ? smem + (((smem_u32(smem) + FD_HEAD + 1023u) & ~1023u) - smem_u32(smem))
                           : smem + FD_HEAD;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hkv = pool.hkv;
  // Full layer: the items (sequence, split, KV head) of the device plan, in
  // sequence order, sequence b owning items prefix[b] .. prefix[b+1]-1.
  // Windowed layer: one item per (sequence, KV head).
  // A batch of up to DP_INLINE_MAX sequences is planned by every CTA itself
  // (the same inputs give every CTA the same plan; CTA 0 stores it for the
  // merge); a larger one by full_decode_plan_kernel before this kernel.
  long long nitems = (long long)B * hkv;
  // windowed layer: bit j of ph is the parity of stage j's next phase, bit j
  // of pend marks a load into stage j not yet seen complete (this warp's
  // stages j = warp + 4i only)
  uint32_t ph = 0, pend = 0;
  if (WINDOW) {
    if (tid == 0) {
      for (int j = 0; j < FDW_SUBS; ++j) tc::mbar_init(sBar + 8 * j, 1);
      *abort_flag = 0;
      tc::fence_mbar_init();
    }
    __syncthreads();
  }
  if (!WINDOW) {
    if (B <= DP_INLINE_MAX) {
      int32_t *sPrefix = reinterpret_cast<int32_t *>(smem + FD_SMEM);
      int n;
      if (B <= 32) {  // one warp plans, the others wait at the barrier
        if (warp == 0) {
          long long p = 0;
          int sq = 0;
          if (lane < B) {
            p = pos[lane];
            sq = seq[lane];
          }
          if (!__all_sync(0xffffffffu, p == pe && sq == se)) {
            decode_plan_warp(p, sq, B, hkv, pool.num_seqs, max_pos, max_ctx, gridDim.x, sPrefix,
                             blockIdx.x == 0 ? status : nullptr);
          } else if (blockIdx.x == 0 && lane < B) {  // the early plan stands; its bad entries flagged here
            const bool bp = p < 0 || p >= max_pos || p + 1 > max_ctx, bs = sq < 0 || sq >= pool.num_seqs;
            if (bp || bs) flag(status, (bp ? ST_BAD_POS : 0u) | (bs ? ST_BAD_SEQ : 0u));
          }
        }
        __syncthreads();
        split_len = sPrefix[B + 1];
        n = sPrefix[B + 2];
      } else {
        split_len = decode_plan_block<FD_WARPS * 32>(pos, seq, B, hkv, pool.num_seqs, max_pos, max_ctx, gridDim.x,
                                                     sPrefix, &n, blockIdx.x == 0 ? status : nullptr);
      }
      nitems = n;
      if (blockIdx.x == 0) {
        int32_t *gp = const_cast<int32_t *>(plan);
        for (int b = tid; b <= B; b += blockDim.x) gp[DPLAN_PREFIX + b] = sPrefix[b];
        if (tid == 0) {
          gp[0] = split_len;
          gp[1] = n;
        }
      }
      prefix = sPrefix;
    } else {
      split_len = plan[0];
      nitems = plan[1];
    }
  }

  // Windowed layer, across items: the next item's position and sequence id
  // are loaded during the current one (carried), its query rows, table row
  // and window rows prefetched into L2, and its block ids left in sNB
  // (nb_ok) by the last warp.
  bool carried = false, nb_ok = false;
  long long p_next = 0;
  int s_next = 0;
  const int bsz = pool.block_size;

  for (long long w = blockIdx.x; w < nitems; w += gridDim.x) {
    int b, split, kv;
    if (WINDOW) {
      b = (int)(w / hkv);
      kv = (int)(w % hkv);
      split = 0;
    } else {
      b = plan_find(prefix, B, w);
      const int local = (int)(w - prefix[b]);
      split = local / hkv;
      kv = local - split * hkv;
    }
    // The query rows' copies go out before anything is waited for; they join
    // the query group closed below (or are drained on the early exits).
    q_rows_issue<FD_WARPS * 32>(q + ((long long)b * hq + (long long)kv * G) * DQK, G, sQ, tid);
    long long p;
    int s;
    if (WINDOW && carried) {
      p = p_next;
      s = s_next;
    } else {
      p = pos[b];
      s = seq[b];
    }
    const long long wn = w + gridDim.x;
    const bool has_next = WINDOW && wn < nitems;
    int kv_next = 0;
    if (has_next) {
      const int bn = (int)(wn / hkv);
      kv_next = (int)(wn % hkv);
      p_next = pos[bn];
      s_next = seq[bn];
      if (tid == 0) prefetch_l2(q + ((long long)bn * hq + (long long)kv_next * G) * DQK, G * DQK * 2);
    }
    carried = has_next;
    const bool use_nb = WINDOW && nb_ok;  // sNB holds this item's block ids
    nb_ok = false;
    const bool bad_pos = p < 0 || p >= max_pos || p + 1 > max_ctx;
    const bool bad_seq = s < 0 || s >= pool.num_seqs;
    if (bad_pos || bad_seq) {  // (the plan gives such a sequence no items; flagged there)
      cp_async_wait_all();
      if (WINDOW) {
        if (kv == 0 && tid == 0) flag(status, (bad_pos ? ST_BAD_POS : 0u) | (bad_seq ? ST_BAD_SEQ : 0u));
        uint16_t *o = out_direct + ((long long)b * hq + (long long)kv * G) * DV;  // direct mode: zero rows
        for (int e = tid; e < G * DV; e += blockDim.x) o[e] = 0;
      }
      continue;  // otherwise the combine writes zeros for this sequence
    }
    // window: keys p-window+1..p; the range starts on a 16-key subtile boundary
    // (a subtile never straddles a block); rows below key_min are zero-filled
    // instead of read and their scores masked
    const long long key_min = WINDOW ? max(0LL, p - window + 1) : 0;
    const long long key_lo = (key_min & ~15LL) + (long long)split * split_len;
    const long long key_hi = min(key_lo + split_len, p + 1);
    if (key_lo > p) {
      cp_async_wait_all();
      continue;
    }

    // the previous item's merge area (over the stages) is free again; a
    // windowed layer whose wait gave up stops here
    if (WINDOW) {
      if (__syncthreads_or(*abort_flag != 0)) {
        cp_async_wait_all();
        break;
      }
      tc::fence_proxy_async_smem();  // generic accesses to the stages before the TMA writes
    } else {
      __syncthreads();
    }
    // The query group closes before the first key subtiles go out; the query
    // tile is rotated once it has landed.  The subtiles do not depend on it,
    // and the query's copies do not queue behind theirs.
    q_table_issue(table + p * 64, sCS, tid);
    const int nsub = (int)((key_hi - key_lo + 15) / 16);
    const int my_n = nsub > warp ? (nsub - warp + FD_WARPS - 1) / FD_WARPS : 0;
    // the warp's i-th subtile (subtile warp + 4i of the item): a ring of
    // FD_STAGES stages per warp, or (window) the subtile's own stage
    auto stage = [&](int i) -> uint8_t * {
      return sStage + (WINDOW ? warp + i * FD_WARPS : warp * FD_STAGES + i % FD_STAGES) * FD_STAGE;
    };
    const int32_t *bt = pool.block_table + (long long)s * pool.max_blocks;

    auto issue = [&](int i) {
      const long long key0 = key_lo + 16LL * (warp + i * FD_WARPS);
      const int blk = use_nb ? sNB[key0 / bsz - key_lo / bsz] : bt[key0 / bsz];
      const bool blk_ok = blk >= 0 && blk < pool.num_blocks;
      if (!blk_ok && lane == 0) flag(status, ST_BAD_BLOCK);
      const long long hrow = ((long long)(blk_ok ? blk : 0) * hkv + kv) * bsz + (key0 % bsz);
      const uint16_t *kg = pool.k + hrow * DQK;
      const uint16_t *vg = pool.v + hrow * DV;
      const uint32_t kb = smem_u32(stage(i));
      const uint32_t vb = kb + FD_SUB_K;
#pragma unroll
      for (int u = 0; u < 12; ++u) {
        const int c = lane + 32 * u, r = c / 24, ch = c % 24;
        const int nb = (blk_ok && key0 + r < key_hi && (!WINDOW || key0 + r >= key_min)) ? 16 : 0;
        cp_async16(kb + swz<DQK>(r, ch), kg + r * DQK + ch * 8, nb);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = lane + 32 * u, r = c >> 4, ch = c & 15;
        const int nb = (blk_ok && key0 + r < key_hi && (!WINDOW || key0 + r >= key_min)) ? 16 : 0;
        cp_async16(vb + swz<DV>(r, ch), vg + r * DV + ch * 8, nb);
      }
    };

    // Windowed layer: the warp's subtiles by TMA, one box of 16 rows each for K and V
    // (a 16-key subtile never straddles a block), each completing on its
    // stage's barrier; rows outside the window arrive too (zeroed or masked
    // below).  A bad block id: no load, the barrier completes at once and the
    // subtile counts as masked.
    auto issue_tma = [&](int i) {
      const int j = warp + i * FD_WARPS;
      const long long key0 = key_lo + 16LL * j;
      const int blk = use_nb ? sNB[key0 / bsz - key_lo / bsz] : bt[key0 / bsz];
      const uint32_t bar = sBar + 8 * j, dst = smem_u32(stage(i));
      if (blk >= 0 && blk < pool.num_blocks) {
        const int hrow = (int)(((long long)blk * hkv + kv) * bsz + key0 % bsz);
        tc::mbar_expect_tx_elect(bar, FD_STAGE);
        tc::tma_load_3d_elect(dst, &kmap, 0, 0, hrow, bar);
        tc::tma_load_3d_elect(dst + FD_SUB_K, &vmap, 0, 0, hrow, bar);
      } else if (lane == 0) {
        flag(status, ST_BAD_BLOCK);
        tc::mbar_arrive(bar);
      }
      pend |= 1u << j;
    };

    constexpr int AHEAD = WINDOW ? 0 : FD_STAGES - 1;
    if (WINDOW) {
#pragma unroll
      for (int i = 0; i < FDW_AHEAD; ++i)
        if (i < my_n) issue_tma(i);
    }
#pragma unroll
    for (int i = 0; i < AHEAD; ++i) {
      if (i < my_n) issue(i);
      cp_async_commit();
    }
    cp_async_wait<AHEAD>();  // the query group (the oldest)
    __syncthreads();
    q_tile_rotate(G, sQ, sCS, tid);
    __syncthreads();
    uint32_t qf[12][4];
    load_q_frags(sQ, lane, qf);
    if (WINDOW && has_next) {
      // the next item: its window rows and table row into L2, its block ids
      // into sNB (every issue of this item has read sNB before the barrier
      // above); the warp's wait for the ids overlaps its first subtile's
      const bool ok_next = p_next >= 0 && p_next < max_pos && p_next + 1 <= max_ctx && s_next >= 0 &&
                           s_next < pool.num_seqs;
      if (ok_next) {
        const long long kmin = max(0LL, p_next - window + 1), klo = kmin & ~15LL;
        const long long b0 = klo / bsz, nblk = p_next / bsz - b0 + 1;
        if (warp == FD_WARPS - 1) {
          const int32_t *btn = pool.block_table + (long long)s_next * pool.max_blocks;
          if (lane < nblk) {
            const int blk = btn[b0 + lane];
            sNB[lane] = blk;
            if (blk >= 0 && blk < pool.num_blocks) {
              const long long first = (b0 + lane) * bsz;
              const long long r0 = max(kmin, first) - first, r1 = min(p_next, first + bsz - 1) - first;
              const long long hrow = ((long long)blk * hkv + kv_next) * bsz + r0;
              prefetch_l2(pool.k + hrow * DQK, (uint32_t)(r1 - r0 + 1) * DQK * 2);
              prefetch_l2(pool.v + hrow * DV, (uint32_t)(r1 - r0 + 1) * DV * 2);
            }
          }
          if (lane == 0) prefetch_l2(table + p_next * 64, 256);
        }
        nb_ok = true;
      }
    }

    float O[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) O[nt][0] = O[nt][1] = O[nt][2] = O[nt][3] = 0.f;
    float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;
    for (int i = 0; i < my_n; ++i) {
      const uint32_t kb = smem_u32(stage(i));
      const long long key0 = key_lo + 16LL * (warp + i * FD_WARPS);
      const int blk = WINDOW && use_nb ? sNB[key0 / bsz - key_lo / bsz] : bt[key0 / bsz];
      const bool blk_ok = blk >= 0 && blk < pool.num_blocks;
      if (WINDOW) {
        const int j = warp + i * FD_WARPS;
        const bool got = __all_sync(0xffffffffu, tc::mbar_wait(sBar + 8 * j, (ph >> j) & 1u, abort_flag));
        if (!got) continue;  // gave up: the subtile counts as masked, and the kernel stops at the next item
        ph ^= 1u << j;
        pend &= ~(1u << j);
        // rows outside the window (or of a bad block) hold other keys' values:
        // zero them, as their zero weights must not meet a non-finite value
        if (!blk_ok || key0 < key_min || key0 + 16 > key_hi) {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int c = lane + 32 * u, r = c >> 4, ch = c & 15;
            const long long key = key0 + r;
            if (!(blk_ok && key < key_hi && key >= key_min))
              *reinterpret_cast<uint4 *>(stage(i) + FD_SUB_K + sub_off<DV, true>(r, ch)) = make_uint4(0, 0, 0, 0);
          }
        }
      } else {
        if (i + FD_STAGES - 1 < my_n) issue(i + FD_STAGES - 1);
        cp_async_commit();
        cp_async_wait<FD_STAGES - 1>();
      }
      __syncwarp();
      float S[2][4];
      qk_16keys<WINDOW>(qf, kb, 0, lane, S);
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const long long key = key0 + 8 * j + 2 * (lane & 3) + (e & 1);
          S[j][e] = (blk_ok && key < key_hi && (!WINDOW || key >= key_min)) ? S[j][e] * scale_log2 : NEG_INF;
        }
      softmax_update(S, m0, m1, l0, l1, O);
      pv_16keys<WINDOW>(S, kb + FD_SUB_K, 0, lane, O);
      __syncwarp();
    }
    cp_async_wait<0>();
    __syncthreads();  // all warps done with their stages: reuse them as the merge area

    float *mml = reinterpret_cast<float *>(sStage);   // [4][16][2]
    float *mo = mml + FD_WARPS * 16 * 2;              // [4][16][MO_STRIDE]
    stash_warp_state(mml + warp * 32, mo + warp * 16 * MO_STRIDE, lane, m0, m1, l0, l1, O);
    __syncthreads();

    // Per q head (threads 0..G-1): the head's maximum over the four warps
    // and each warp's scale factor; then every thread takes 4-dim pieces of
    // the G x 128 outputs.
    float *fac = mo + FD_WARPS * 16 * MO_STRIDE;  // [4 warps][16 heads]
    if (tid < G) {
      const int g = tid;
      const float sl = WINDOW ? sinks[kv * G + g] * LOG2E : NEG_INF;
      float M = sl;
#pragma unroll
      for (int ww = 0; ww < FD_WARPS; ++ww) M = fmaxf(M, mml[ww * 32 + g * 2]);
      const float base = M == NEG_INF ? 0.f : M;
      float f[FD_WARPS], L = WINDOW ? ex2(sl - base) : 0.f;
#pragma unroll
      for (int ww = 0; ww < FD_WARPS; ++ww) {
        const float mw = mml[ww * 32 + g * 2];
        f[ww] = mw == NEG_INF ? 0.f : ex2(mw - base);
        L += mml[ww * 32 + g * 2 + 1] * f[ww];
      }
      if (WINDOW) {
        // one split holds the whole window: normalise here, the sink joining
        // the denominator only (its numerator is zero)
        const float inv = 1.f / L;
#pragma unroll
        for (int ww = 0; ww < FD_WARPS; ++ww) fac[ww * 16 + g] = f[ww] * inv;
      } else {
#pragma unroll
        for (int ww = 0; ww < FD_WARPS; ++ww) fac[ww * 16 + g] = f[ww];
        float *pml = part_ml + w * G * 2;
        pml[g * 2] = M;
        pml[g * 2 + 1] = L;
      }
    }
    __syncthreads();
    for (int idx = tid; idx < G * (DV / 4); idx += blockDim.x) {
      const int g = idx / (DV / 4), d4 = 4 * (idx % (DV / 4));
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int ww = 0; ww < FD_WARPS; ++ww) {
        const float f = fac[ww * 16 + g];
        const float4 x = *reinterpret_cast<const float4 *>(mo + (ww * 16 + g) * MO_STRIDE + d4);
        acc.x += x.x * f;
        acc.y += x.y * f;
        acc.z += x.z * f;
        acc.w += x.w * f;
      }
      if (WINDOW) {
        uint16_t *o = out_direct + ((long long)b * hq + (long long)kv * G + g) * DV + d4;
        *reinterpret_cast<uint2 *>(o) = make_uint2(pack_bf16(acc.x, acc.y), pack_bf16(acc.z, acc.w));
      } else {
        *reinterpret_cast<float4 *>(part_o + (w * G + g) * DV + d4) = acc;
      }
    }
  }
  if (WINDOW && pend) {
    // a wait gave up: report it, and before leaving wait (bounded, whatever
    // the abort flag says) for this warp's loads still in flight
    if (lane == 0) flag(status, ST_TIMEOUT);
    uint32_t never = 0;
    for (int j = 0; j < FDW_SUBS; ++j)
      if ((pend >> j) & 1u) tc::mbar_wait(sBar + 8 * j, (ph >> j) & 1u, &never);
  }
}

// Batches past DP_INLINE_MAX sequences: the plan by a kernel of its own,
// written to the workspace for the split and merge kernels.
constexpr int DP_THREADS = 256;

__global__ void __launch_bounds__(DP_THREADS)
    full_decode_plan_kernel(const int64_t *__restrict__ pos, const int32_t *__restrict__ seq, int B, int hkv,
                            int num_seqs, int64_t max_pos, long long max_ctx, int R, int32_t *__restrict__ plan,
                            unsigned *status) {
  pdl_wait();
  pdl_trigger();
  int nitems;
  const int L = decode_plan_block<DP_THREADS>(pos, seq, B, hkv, num_seqs, max_pos, max_ctx, R,
                                              plan + DPLAN_PREFIX, &nitems, status);
  if (threadIdx.x == 0) {
    plan[0] = L;
    plan[1] = nitems;
  }
}

// Full layer, phase 2: merge the splits of each (sequence, KV head, q head)
// row by log-sum-exp and normalise.  NW warps per row (NW in {1, 2, 4, 8,
// 16}, from the expected split count) fold interleaved subsets of the splits
// -- lane l owns value dims 4l..4l+3 -- FC_K splits at a time, all of their
// loads in flight together, and the row's first warp merges their partial
// states from shared memory.  Sixteen warps per CTA, 16 / NW rows per CTA, so
// short contexts with many sequences and one long sequence with hundreds of
// splits both keep the GPU busy.
//
// The kernel is launched as a programmatic dependent of the split kernel: its
// CTAs may start while the split kernel's last CTAs run, read the inputs the
// split kernel does not write (positions, sequence ids), and wait at
// griddepcontrol.wait -- which returns once the split kernel has completed
// and its writes are visible -- before reading the plan and the partials.
constexpr int FC_WARPS = 16;
constexpr int FC_K = 8;

__global__ void __launch_bounds__(FC_WARPS * 32)
    full_combine_kernel(const int64_t *__restrict__ pos, const int32_t *__restrict__ seq, int B, int hq, int G,
                        int hkv, int num_seqs, int64_t max_pos, long long max_ctx, const int32_t *__restrict__ plan,
                        int nw, const float *__restrict__ part_ml, const float *__restrict__ part_o,
                        uint16_t *__restrict__ out) {
  __shared__ float s_ml[FC_WARPS][2];
  __shared__ float4 s_acc[FC_WARPS][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rows_per_cta = FC_WARPS / nw;
  const long long row = (long long)blockIdx.x * rows_per_cta + warp / nw;  // ((b * hkv) + kv) * G + g
  const int sub = warp % nw;
  const bool have = row < (long long)B * hkv * G;
  const int g = have ? (int)(row % G) : 0;
  const int kv = have ? (int)((row / G) % hkv) : 0;
  const int b = have ? (int)(row / ((long long)G * hkv)) : 0;
  bool ok = false;
  long long p = 0;
  if (have) {
    p = pos[b];
    const int s = seq[b];
    ok = p >= 0 && p < max_pos && p + 1 <= max_ctx && s >= 0 && s < num_seqs;
  }
  pdl_wait();
  pdl_trigger();
  const int split_len = plan[0];
  const int n = ok ? (int)(p / split_len) + 1 : 0;
  const long long base = have ? plan[DPLAN_PREFIX + b] : 0;
  float M = NEG_INF, L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i0 = sub; i0 < n; i0 += FC_K * nw) {
    float2 ml[FC_K];
    float4 o[FC_K];
#pragma unroll
    for (int k = 0; k < FC_K; ++k) {
      const int i = i0 + k * nw;
      ml[k] = make_float2(NEG_INF, 0.f);
      o[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i < n) {
        const long long w = base + (long long)i * hkv + kv;
        ml[k] = *reinterpret_cast<const float2 *>(part_ml + (w * G + g) * 2);
        o[k] = *reinterpret_cast<const float4 *>(part_o + (w * G + g) * DV + 4 * lane);
      }
    }
    float Mn = M;
#pragma unroll
    for (int k = 0; k < FC_K; ++k) Mn = fmaxf(Mn, ml[k].x);
    if (Mn == NEG_INF) continue;  // nothing yet (empty splits only)
    const float c = ex2(M - Mn);  // M = -inf gives 0
    L *= c;
    acc.x *= c;
    acc.y *= c;
    acc.z *= c;
    acc.w *= c;
#pragma unroll
    for (int k = 0; k < FC_K; ++k) {
      const float f = ex2(ml[k].x - Mn);  // an empty split (-inf) gives 0
      L += ml[k].y * f;
      acc.x += o[k].x * f;
      acc.y += o[k].y * f;
      acc.z += o[k].z * f;
      acc.w += o[k].w * f;
    }
    M = Mn;
  }
  if (nw > 1) {
    if (lane == 0) {
      s_ml[warp][0] = M;
      s_ml[warp][1] = L;
    }
    s_acc[warp][lane] = acc;
    __syncthreads();
    if (sub == 0) {
      float Mt = NEG_INF;
      for (int u = 0; u < nw; ++u) Mt = fmaxf(Mt, s_ml[warp + u][0]);
      L = 0.f;
      acc = make_float4(0.f, 0.f, 0.f, 0.f);
      if (Mt != NEG_INF) {
        for (int u = 0; u < nw; ++u) {
          const float mu = s_ml[warp + u][0];
          if (mu == NEG_INF) continue;
          const float f = ex2(mu - Mt);
          const float4 o = s_acc[warp + u][lane];
          L += s_ml[warp + u][1] * f;
          acc.x += o.x * f;
          acc.y += o.y * f;
          acc.z += o.z * f;
          acc.w += o.w * f;
        }
      }
    }
  }
  if (!have || sub != 0) return;
  const float inv = L > 0.f ? 1.f / L : 0.f;
  uint2 w2;
  w2.x = pack_bf16(acc.x * inv, acc.y * inv);
  w2.y = pack_bf16(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2 *>(out + ((long long)b * hq + (long long)kv * G + g) * DV + 4 * lane) = w2;
}

}  // namespace

// ---------------------------------------------------------------------------

// Uniform-batch estimate of the split plan (every sequence at max_ctx): the
// first eight candidates of full_decode_plan_kernel.  The merge kernel sizes
// its warps per row from it.  Measured with the plan taken this way: at batch
// 1 and 4 one item per CTA beats eight short ones by 1.5x; at batch 16, four
// per CTA beat an uneven 1.05; a cap of 8192 keys against 16K / 32K: the
// 128-sequence ragged step 73.9 ms against 80.3 / 83.8, uniform batch 16 at
// 524K 3.01 ms against 2.94 / 2.92.  The cap has 256 keys of headroom so that
// an 8K context (8193 keys, 8256 rounded) is still one split.
DecodePlan full_decode_plan(int B, int hkv, long long max_ctx) {
  const long long R = 2LL * num_sms();
  const long long units = (long long)B * hkv;  // (sequence, KV head) pairs
  long long best_cost = -1;
  DecodePlan best{1, 64};
  for (int k = 1; k <= 8; ++k) {
    long long n = k * R / units;
    if (n < 1) n = 1;
    long long len = ((max_ctx + n - 1) / n + 63) / 64 * 64;
    if (len > FD_MAX_LEN) len = FD_MAX_LEN;
    n = (max_ctx + len - 1) / len;
    const long long rounds = (units * n + R - 1) / R;
    const long long cost = rounds * (len + FD_ITEM_KEYS);
    if (best_cost < 0 || cost < best_cost || (cost == best_cost && n < best.splits)) {
      best_cost = cost;
      best.splits = (int)n;
      best.split_len = (int)len;
    }
  }
  return best;
}

static size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Most items a device plan can give: a candidate of about k items per
// resident CTA gives at most k * R plus one partial split per (sequence, KV
// head); a capped one at most ceil(max_ctx / FD_MAX_LEN) splits per sequence.
static long long decode_items_cap(int B, int hkv, long long max_ctx) {
  const long long R = 2LL * num_sms(), units = (long long)B * hkv;
  const long long a = 8 * R + units, c = units * ((max_ctx + FD_MAX_LEN - 1) / FD_MAX_LEN);
  return a > c ? a : c;
}

// Workspace: the plan (L, item count, item prefix), then fp32 (m, l) and
// numerators per (item, q head of the group).
static size_t plan_bytes(int B) { return align256(((size_t)DPLAN_PREFIX + B + 1) * 4); }

size_t full_decode_workspace(int B, int hq, int hkv, long long max_ctx) {
  const size_t items = (size_t)decode_items_cap(B, hkv, max_ctx);
  const size_t G = (size_t)(hq / hkv);
  return plan_bytes(B) + align256(items * G * 2 * sizeof(float)) + align256(items * G * DV * sizeof(float));
}

cudaError_t launch_full_decode(const uint16_t *q, const int64_t *pos, const int32_t *seq, int B, int hq,
                               const KvView &pool, const float *table, int64_t max_pos,
                               float softmax_scale, long long max_ctx, void *ws, uint16_t *out,
                               unsigned *status, cudaStream_t st) {
  // shared memory: the stages, plus the plan's item prefix when the kernel plans itself
  constexpr int FD_SMEM_MAX = FD_SMEM + (DP_INLINE_MAX + 3) * 4;
  cudaError_t e = ensure_smem_limit(0, (const void *)full_decode_kernel<false>, FD_SMEM_MAX);
  if (e != cudaSuccess) return e;
  const int hkv = pool.hkv, G = hq / hkv;
  const size_t items = (size_t)decode_items_cap(B, hkv, max_ctx);
  int32_t *plan = reinterpret_cast<int32_t *>(ws);
  uint8_t *w8 = reinterpret_cast<uint8_t *>(ws) + plan_bytes(B);
  float *part_ml = reinterpret_cast<float *>(w8);
  float *part_o = reinterpret_cast<float *>(w8 + align256(items * G * 2 * sizeof(float)));
  const int R = 2 * num_sms();
  int smem = FD_SMEM;
  if (B <= DP_INLINE_MAX) {
    smem += ((B + 3) * 4 + 15) / 16 * 16;  // prefix[B + 1] and a split length and item count
  } else {
    e = launch_pdl(full_decode_plan_kernel, dim3(1), dim3(DP_THREADS), 0, st, pos, seq, B, hkv, pool.num_seqs, max_pos,
                   max_ctx, R, plan, status);
    if (e != cudaSuccess) return e;
  }
  const CUtensorMap unused{};  // (the full layer's subtiles go by cp.async)
  e = launch_pdl(full_decode_kernel<false>, dim3((unsigned)R), dim3(FD_WARPS * 32), (size_t)smem, st, unused, unused, q,
                 pos, seq, B, hq, G, pool, table, max_pos, softmax_scale * LOG2E, max_ctx, (const int32_t *)plan, 0,
                 part_ml, part_o, status, 0, (const float *)nullptr, (uint16_t *)nullptr);
  if (e != cudaSuccess) return e;
  // warps per merged row: about four splits each, at most sixteen
  const DecodePlan est = full_decode_plan(B, hkv, max_ctx);
  int nw = 1;
  while (nw < FC_WARPS && nw * 4 < est.splits) nw *= 2;
  const long long rows = (long long)B * hkv * G;
  const long long ctas = (rows + FC_WARPS / nw - 1) / (FC_WARPS / nw);
  // a programmatic dependent of the split kernel (see full_combine_kernel)
  return launch_pdl(full_combine_kernel, dim3((unsigned)ctas), dim3(FC_WARPS * 32), 0, st, pos, seq, B, hq, G, hkv,
                    pool.num_seqs, max_pos, max_ctx, (const int32_t *)plan, nw, (const float *)part_ml,
                    (const float *)part_o, out);
}

cudaError_t launch_swa_decode_paged(const uint16_t *q, const int64_t *pos, const int32_t *seq, int B, int hq,
                                    const KvView &pool, const float *sinks, const float *table, int64_t max_pos,
                                    float softmax_scale, uint16_t *out, unsigned *status, cudaStream_t st) {
  if (hq / pool.hkv <= 8)  // groups of up to 8 q heads: the keys-as-rows kernel (swa_paged.cu)
    return launch_swa_paged(q, pos, seq, B, hq, pool, sinks, table, max_pos, softmax_scale, out, status, st);
  cudaError_t e = ensure_smem_limit(9, (const void *)full_decode_kernel<true>, FDW_SMEM);
  if (e != cudaSuccess) return e;
  const int hkv = pool.hkv, G = hq / hkv;
  // positions past the pool are flagged as bad positions, like full_attn_decode's max_ctx
  const long long cap = (long long)pool.max_blocks * pool.block_size;
  const long long max_ctx = cap < max_pos ? cap : max_pos;
  const long long items = (long long)B * hkv;
  long long grid = (long long)num_sms() * 2;
  if (grid > items) grid = items;
  // the pool as rows of 64-element parts, boxes of all parts x 16 rows
  const long long rows = (long long)pool.num_blocks * hkv * pool.block_size;
  CUtensorMap km, vm;
  if (rows > 0x7fffffffLL || !make_tma_map_rows3d(&km, pool.k, rows, DQK, 16) ||
      !make_tma_map_rows3d(&vm, pool.v, rows, DV, 16))
    return cudaErrorInvalidValue;
  static_assert((WIN + 16) / 16 == FDW_SUBS, "split length of the window below: at most FDW_SUBS subtiles");
  return launch_pdl(full_decode_kernel<true>, dim3((unsigned)grid), dim3(FD_WARPS * 32), (size_t)FDW_SMEM, st, km, vm, q,
                    pos, seq, B, hq, G, pool, table, max_pos, softmax_scale * LOG2E, max_ctx, (const int32_t *)nullptr,
                    WIN + 16, (float *)nullptr, (float *)nullptr, status, WIN, sinks, out);
}

}  // namespace kvr
