// decode.cu -- one-token decode over a windowed layer (ring + sink) and over
// a full-attention layer (paged pool, split-K with a log-sum-exp combine).
//
// Math (colibri "MiMo-V2.6", "What the engine implements"; gaudi-cookbook
// "MiMo-V2.6-Flash on Gaudi 2", "What was built"): q is rotated on dims 0..63
// with the table row of its position and rounded to bf16; s = q.k' scaled;
// softmax in the base-2 domain with fp32 state (m, l, o); the windowed layer
// adds e^{sink - m} to the denominator exactly once, at the final merge.
// Decode is memory-bound (Xiaomi "Full-Pipeline Inference Optimization",
// section 1.2): every K/V byte is read once, through 16-byte cp.async copies
// into swizzled shared memory, and the two small products per key tile run
// on the bf16 tensor cores (mma.sync m16n8k16, fp32 accumulate) with the G
// query heads of one KV head as the 16 rows of the MMA.
#include "launch.h"

#include <cfloat>

namespace kvr {
namespace {

constexpr float NEG_INF = -INFINITY;

// ---------------------------------------------------------------------------
// Shared pieces.

// Rotate the G query heads of one token (q_heads [G][192]) with the table
// row cs_row ([32][2] fp32), round to bf16 and store them as rows 0..G-1 of
// the swizzled [16][192] tile sQ; rows G..15 are zero.
__device__ __forceinline__ void load_q_tile(const uint16_t *__restrict__ q_heads, int G,
                                            const float *__restrict__ cs_row, uint8_t *sQ, int tid,
                                            int nthreads) {
  for (int it = tid; it < 16 * 20; it += nthreads) {
    const int r = it / 20, c = it % 20;
    const uint4 zero = make_uint4(0, 0, 0, 0);
    if (c < 4) {
      uint4 o1 = zero, o2 = zero;
      if (r < G) {
        const uint4 *src = reinterpret_cast<const uint4 *>(q_heads + r * DQK);
        const float4 *tr = reinterpret_cast<const float4 *>(cs_row + 16 * c);
        float cs[16];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float4 f = tr[u];
          cs[4 * u] = f.x; cs[4 * u + 1] = f.y; cs[4 * u + 2] = f.z; cs[4 * u + 3] = f.w;
        }
        rope_pair8(src[c], src[c + 4], cs, o1, o2);
      }
      *reinterpret_cast<uint4 *>(sQ + swz<DQK>(r, c)) = o1;
      *reinterpret_cast<uint4 *>(sQ + swz<DQK>(r, c + 4)) = o2;
    } else {
      const int ch = c + 4;  // chunks 8..23
      uint4 x = zero;
      if (r < G) x = reinterpret_cast<const uint4 *>(q_heads + r * DQK)[ch];
      *reinterpret_cast<uint4 *>(sQ + swz<DQK>(r, ch)) = x;
    }
  }
}

// A fragments of the [16][192] Q tile for the 12 k-steps.
__device__ __forceinline__ void load_q_frags(const uint8_t *sQ, int lane, uint32_t (&qf)[12][4]) {
  const uint32_t base = smem_u32(sQ);
#pragma unroll
  for (int kk = 0; kk < 12; ++kk) {
    const int row = lane & 15;
    const int ch = 2 * kk + (lane >> 4);
    ldsm_x4(base + swz<DQK>(row, ch), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
  }
}

// S[16 x 16 keys] = Q K^T for the 16 K rows starting at row r0 of a swizzled
// [*][192] tile.
__device__ __forceinline__ void qk_16keys(const uint32_t (&qf)[12][4], uint32_t kbase, int r0, int lane,
                                          float (&S)[2][4]) {
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) S[j][e] = 0.f;
  const int row = r0 + (lane & 7) + ((lane >> 4) << 3);
  const int csel = (lane >> 3) & 1;
#pragma unroll
  for (int kk = 0; kk < 12; ++kk) {
    uint32_t b0, b1, b2, b3;
    ldsm_x4(kbase + swz<DQK>(row, 2 * kk + csel), b0, b1, b2, b3);
    mma_bf16(S[0], qf[kk], b0, b1);
    mma_bf16(S[1], qf[kk], b2, b3);
  }
}

// O[16 x 128] += P[16 x 16 keys] V[16 keys x 128] for the V rows starting at
// row r0 of a swizzled [*][128] tile; P comes from the S accumulators.
__device__ __forceinline__ void pv_16keys(const float (&P)[2][4], uint32_t vbase, int r0, int lane,
                                          float (&O)[16][4]) {
  uint32_t a[4];
  a[0] = pack_bf16(P[0][0], P[0][1]);
  a[1] = pack_bf16(P[0][2], P[0][3]);
  a[2] = pack_bf16(P[1][0], P[1][1]);
  a[3] = pack_bf16(P[1][2], P[1][3]);
  const int row = r0 + (lane & 7) + (((lane >> 3) & 1) << 3);
  const int csel = lane >> 4;
#pragma unroll
  for (int dp = 0; dp < 8; ++dp) {
    uint32_t b0, b1, b2, b3;
    ldsm_x4_t(vbase + swz<DV>(row, 2 * dp + csel), b0, b1, b2, b3);
    mma_bf16(O[2 * dp], a, b0, b1);
    mma_bf16(O[2 * dp + 1], a, b2, b3);
  }
}

// Online-softmax update of one warp's state with a 16-key score tile already
// scaled to the base-2 domain (masked entries = -inf).  Rows lane/4 and
// lane/4 + 8; l is this thread's partial row sum (quad-reduced at the end).
__device__ __forceinline__ void softmax_update(float (&S)[2][4], float &m0, float &m1, float &l0, float &l1,
                                               float (&O)[16][4]) {
  float r0 = fmaxf(fmaxf(S[0][0], S[0][1]), fmaxf(S[1][0], S[1][1]));
  float r1 = fmaxf(fmaxf(S[0][2], S[0][3]), fmaxf(S[1][2], S[1][3]));
  r0 = fmaxf(r0, __shfl_xor_sync(0xffffffffu, r0, 1));
  r0 = fmaxf(r0, __shfl_xor_sync(0xffffffffu, r0, 2));
  r1 = fmaxf(r1, __shfl_xor_sync(0xffffffffu, r1, 1));
  r1 = fmaxf(r1, __shfl_xor_sync(0xffffffffu, r1, 2));
  const float n0 = fmaxf(m0, r0), n1 = fmaxf(m1, r1);
  const float b0 = n0 == NEG_INF ? 0.f : n0;
  const float b1 = n1 == NEG_INF ? 0.f : n1;
  const float c0 = ex2(m0 - b0), c1 = ex2(m1 - b1);
  m0 = n0;
  m1 = n1;
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    S[j][0] = ex2(S[j][0] - b0);
    S[j][1] = ex2(S[j][1] - b0);
    S[j][2] = ex2(S[j][2] - b1);
    S[j][3] = ex2(S[j][3] - b1);
    s0 += S[j][0] + S[j][1];
    s1 += S[j][2] + S[j][3];
  }
  l0 = l0 * c0 + s0;
  l1 = l1 * c1 + s1;
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
    O[nt][0] *= c0;
    O[nt][1] *= c0;
    O[nt][2] *= c1;
    O[nt][3] *= c1;
  }
}

// Write one warp's (m, l, O) into the merge area: ml [16][2], o [16][128].
__device__ __forceinline__ void stash_warp_state(float *ml, float *o, int lane, float m0, float m1, float l0,
                                                 float l1, const float (&O)[16][4]) {
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const int r = lane >> 2, cq = 2 * (lane & 3);
  if ((lane & 3) == 0) {
    ml[r * 2] = m0;
    ml[r * 2 + 1] = l0;
    ml[(r + 8) * 2] = m1;
    ml[(r + 8) * 2 + 1] = l1;
  }
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
    *reinterpret_cast<float2 *>(o + r * DV + 8 * nt + cq) = make_float2(O[nt][0], O[nt][1]);
    *reinterpret_cast<float2 *>(o + (r + 8) * DV + 8 * nt + cq) = make_float2(O[nt][2], O[nt][3]);
  }
}

// ---------------------------------------------------------------------------
// Windowed layer: one CTA per (sequence, KV head); 4 warps, 32 ring slots each.

constexpr int SWA_WARPS = 4;
constexpr int SWA_SMEM = 16 * DQK * 2 + WIN * DQK * 2 + WIN * DV * 2 + WIN * 4;

__global__ void __launch_bounds__(SWA_WARPS * 32, 2)
    swa_decode_kernel(const uint16_t *__restrict__ q, const int64_t *__restrict__ pos,
                      const int32_t *__restrict__ seq, int hq, int G, KvView ring,
                      const float *__restrict__ sinks, const float *__restrict__ table, int64_t max_pos,
                      float scale_log2, uint16_t *__restrict__ out, unsigned *status) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *sQ = smem;
  uint8_t *sK = sQ + 16 * DQK * 2;
  uint8_t *sV = sK + WIN * DQK * 2;
  int32_t *sPos = reinterpret_cast<int32_t *>(sV + WIN * DV * 2);

  const int hkv = ring.hkv;
  const int b = blockIdx.x / hkv, kv = blockIdx.x % hkv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long p = pos[b];
  const int s = seq[b];
  uint16_t *orow = out + ((long long)b * hq + (long long)kv * G) * DV;
  const bool bad_pos = p < 0 || p >= max_pos;
  const bool bad_seq = s < 0 || s >= ring.num_seqs;
  if (bad_pos || bad_seq) {
    for (int i = tid; i < G * DV; i += blockDim.x) orow[i] = 0;
    if (tid == 0) flag(status, (bad_pos ? ST_BAD_POS : 0u) | (bad_seq ? ST_BAD_SEQ : 0u));
    return;
  }

  // K/V of this warp's 32 slots: contiguous 12 KB + 8 KB in the ring.
  const long long head = (long long)s * hkv + kv;
  {
    const uint16_t *kg = ring.k + (head * WIN + 32 * warp) * DQK;
    const uint16_t *vg = ring.v + (head * WIN + 32 * warp) * DV;
    const uint32_t kb = smem_u32(sK), vb = smem_u32(sV);
#pragma unroll
    for (int i = 0; i < 24; ++i) {
      const int c = lane + 32 * i, r = c / 24, ch = c % 24;
      cp_async16(kb + swz<DQK>(32 * warp + r, ch), kg + r * DQK + ch * 8);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int c = lane + 32 * i, r = c >> 4, ch = c & 15;
      cp_async16(vb + swz<DV>(32 * warp + r, ch), vg + r * DV + ch * 8);
    }
    cp_async_commit();
  }
  sPos[tid] = ring.slot_pos[(long long)s * WIN + tid];  // 128 threads, 128 slots
  load_q_tile(q + ((long long)b * hq + (long long)kv * G) * DQK, G, table + p * 64, sQ, tid, blockDim.x);
  cp_async_wait<0>();
  __syncthreads();

  // A slot is in the window iff it holds a position in (p - 128, p].
  // Zero the V rows of slots outside it so that stale bytes cannot reach
  // the product (their P is 0, but 0 * NaN is not).
  const int myslot = 32 * warp + lane;
  const int sp = sPos[myslot];
  const bool valid = sp >= 0 && sp <= p && sp > p - WIN;
  unsigned bad = __ballot_sync(0xffffffffu, !valid);
  while (bad) {
    const int r = __ffs(bad) - 1;
    bad &= bad - 1;
    if (lane < 16) *reinterpret_cast<uint4 *>(sV + swz<DV>(32 * warp + r, lane)) = make_uint4(0, 0, 0, 0);
  }
  __syncwarp();

  uint32_t qf[12][4];
  load_q_frags(sQ, lane, qf);
  float O[16][4];
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) O[nt][0] = O[nt][1] = O[nt][2] = O[nt][3] = 0.f;
  float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;
  const uint32_t kb = smem_u32(sK), vb = smem_u32(sV);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r0 = 32 * warp + 16 * half;
    float S[2][4];
    qk_16keys(qf, kb, r0, lane, S);
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int slot = r0 + 8 * j + 2 * (lane & 3) + (e & 1);
        const int spos = sPos[slot];
        const bool ok = spos >= 0 && spos <= p && spos > p - WIN;
        S[j][e] = ok ? S[j][e] * scale_log2 : NEG_INF;
      }
    softmax_update(S, m0, m1, l0, l1, O);
    pv_16keys(S, vb, r0, lane, O);
  }
  __syncthreads();  // K tile no longer needed: reuse it as the merge area

  float *mml = reinterpret_cast<float *>(sK);       // [4][16][2]
  float *mo = mml + SWA_WARPS * 16 * 2;            // [4][16][128]
  stash_warp_state(mml + warp * 32, mo + warp * 16 * DV, lane, m0, m1, l0, l1, O);
  __syncthreads();

  // Final merge of the 4 warps with the sink counted once.
  const int d = tid;  // 128 threads = 128 value dims
  for (int g = 0; g < G; ++g) {
    const float sk = sinks[kv * G + g] * LOG2E;
    float M = sk;
#pragma unroll
    for (int w = 0; w < SWA_WARPS; ++w) M = fmaxf(M, mml[w * 32 + g * 2]);
    float L = ex2(sk - M), acc = 0.f;
#pragma unroll
    for (int w = 0; w < SWA_WARPS; ++w) {
      const float mw = mml[w * 32 + g * 2];
      const float f = mw == NEG_INF ? 0.f : ex2(mw - M);
      L += mml[w * 32 + g * 2 + 1] * f;
      acc += mo[(w * 16 + g) * DV + d] * f;
    }
    orow[g * DV + d] = f2bf(acc / L);
  }
}

// ---------------------------------------------------------------------------
// Full layer, phase 1: persistent CTAs walk the virtual items
// (sequence, split, KV head); each real item streams its key range through
// per-warp cp.async pipelines of 16-key subtiles and writes fp32 partials.

constexpr int FD_WARPS = 4;
constexpr int FD_STAGES = 2;
constexpr int FD_SUB_K = 16 * DQK * 2;                 // 6144 B
constexpr int FD_SUB_V = 16 * DV * 2;                  // 4096 B
constexpr int FD_STAGE = FD_SUB_K + FD_SUB_V;          // 10240 B
constexpr int FD_SMEM = 16 * DQK * 2 + FD_WARPS * FD_STAGES * FD_STAGE;
constexpr int FD_TARGET_ITEMS = 152 * 8;
static_assert(FD_WARPS * FD_STAGES * FD_STAGE >= FD_WARPS * 16 * (DV + 2) * 4, "merge area");

__global__ void __launch_bounds__(FD_WARPS * 32, 2)
    full_decode_kernel(const uint16_t *__restrict__ q, const int64_t *__restrict__ pos,
                       const int32_t *__restrict__ seq, int B, int hq, int G, KvView pool,
                       const float *__restrict__ table, int64_t max_pos, float scale_log2,
                       long long max_ctx, int splits, int split_len, float *__restrict__ part_ml,
                       float *__restrict__ part_o, unsigned *status) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *sQ = smem;
  uint8_t *sStage = smem + 16 * DQK * 2;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hkv = pool.hkv;
  const long long nvirt = (long long)B * splits * hkv;

  for (long long w = blockIdx.x; w < nvirt; w += gridDim.x) {
    const int kv = (int)(w % hkv);
    const int split = (int)((w / hkv) % splits);
    const int b = (int)(w / ((long long)hkv * splits));
    const long long p = pos[b];
    const int s = seq[b];
    const bool bad_pos = p < 0 || p >= max_pos || p + 1 > max_ctx;
    const bool bad_seq = s < 0 || s >= pool.num_seqs;
    if (bad_pos || bad_seq) {
      if (split == 0 && kv == 0 && tid == 0)
        flag(status, (bad_pos ? ST_BAD_POS : 0u) | (bad_seq ? ST_BAD_SEQ : 0u));
      continue;  // the combine writes zeros for this sequence
    }
    const long long key_lo = (long long)split * split_len;
    if (key_lo > p) continue;
    const long long key_hi = min(key_lo + split_len, p + 1);

    __syncthreads();  // the previous item's merge area is free again
    load_q_tile(q + ((long long)b * hq + (long long)kv * G) * DQK, G, table + p * 64, sQ, tid, blockDim.x);
    __syncthreads();
    uint32_t qf[12][4];
    load_q_frags(sQ, lane, qf);

    float O[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) O[nt][0] = O[nt][1] = O[nt][2] = O[nt][3] = 0.f;
    float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;

    const int nsub = (int)((key_hi - key_lo + 15) / 16);
    const int my_n = nsub > warp ? (nsub - warp + FD_WARPS - 1) / FD_WARPS : 0;
    uint8_t *wst = sStage + warp * FD_STAGES * FD_STAGE;
    const int32_t *bt = pool.block_table + (long long)s * pool.max_blocks;
    const int bsz = pool.block_size;

    auto issue = [&](int i) {
      const long long key0 = key_lo + 16LL * (warp + i * FD_WARPS);
      const int blk = bt[key0 / bsz];
      const bool blk_ok = blk >= 0 && blk < pool.num_blocks;
      if (!blk_ok && lane == 0) flag(status, ST_BAD_BLOCK);
      const long long hrow = ((long long)(blk_ok ? blk : 0) * hkv + kv) * bsz + (key0 % bsz);
      const uint16_t *kg = pool.k + hrow * DQK;
      const uint16_t *vg = pool.v + hrow * DV;
      const uint32_t kb = smem_u32(wst + (i % FD_STAGES) * FD_STAGE);
      const uint32_t vb = kb + FD_SUB_K;
#pragma unroll
      for (int u = 0; u < 12; ++u) {
        const int c = lane + 32 * u, r = c / 24, ch = c % 24;
        const int nb = (blk_ok && key0 + r < key_hi) ? 16 : 0;
        cp_async16(kb + swz<DQK>(r, ch), kg + r * DQK + ch * 8, nb);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = lane + 32 * u, r = c >> 4, ch = c & 15;
        const int nb = (blk_ok && key0 + r < key_hi) ? 16 : 0;
        cp_async16(vb + swz<DV>(r, ch), vg + r * DV + ch * 8, nb);
      }
    };

#pragma unroll
    for (int i = 0; i < FD_STAGES - 1; ++i) {
      if (i < my_n) issue(i);
      cp_async_commit();
    }
    for (int i = 0; i < my_n; ++i) {
      if (i + FD_STAGES - 1 < my_n) issue(i + FD_STAGES - 1);
      cp_async_commit();
      cp_async_wait<FD_STAGES - 1>();
      __syncwarp();
      const uint32_t kb = smem_u32(wst + (i % FD_STAGES) * FD_STAGE);
      const long long key0 = key_lo + 16LL * (warp + i * FD_WARPS);
      const int blk = bt[key0 / bsz];
      const bool blk_ok = blk >= 0 && blk < pool.num_blocks;
      float S[2][4];
      qk_16keys(qf, kb, 0, lane, S);
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const long long key = key0 + 8 * j + 2 * (lane & 3) + (e & 1);
          S[j][e] = (blk_ok && key < key_hi) ? S[j][e] * scale_log2 : NEG_INF;
        }
      softmax_update(S, m0, m1, l0, l1, O);
      pv_16keys(S, kb + FD_SUB_K, 0, lane, O);
      __syncwarp();
    }
    cp_async_wait<0>();
    __syncthreads();  // all warps done with their stages: reuse them as the merge area

    float *mml = reinterpret_cast<float *>(sStage);   // [4][16][2]
    float *mo = mml + FD_WARPS * 16 * 2;              // [4][16][128]
    stash_warp_state(mml + warp * 32, mo + warp * 16 * DV, lane, m0, m1, l0, l1, O);
    __syncthreads();

    float *pml = part_ml + w * G * 2;
    float *po = part_o + w * G * DV;
    for (int g = 0; g < G; ++g) {
      float M = NEG_INF;
#pragma unroll
      for (int ww = 0; ww < FD_WARPS; ++ww) M = fmaxf(M, mml[ww * 32 + g * 2]);
      const float base = M == NEG_INF ? 0.f : M;
      float L = 0.f;
      for (int d = tid; d < DV; d += blockDim.x) {
        float acc = 0.f;
#pragma unroll
        for (int ww = 0; ww < FD_WARPS; ++ww) {
          const float mw = mml[ww * 32 + g * 2];
          acc += mo[(ww * 16 + g) * DV + d] * (mw == NEG_INF ? 0.f : ex2(mw - base));
        }
        po[g * DV + d] = acc;
      }
      if (tid == 0) {
#pragma unroll
        for (int ww = 0; ww < FD_WARPS; ++ww) {
          const float mw = mml[ww * 32 + g * 2];
          L += mml[ww * 32 + g * 2 + 1] * (mw == NEG_INF ? 0.f : ex2(mw - base));
        }
        pml[g * 2] = M;
        pml[g * 2 + 1] = L;
      }
    }
  }
}

// Full layer, phase 2: merge the splits of each (sequence, KV head) by
// log-sum-exp and normalise.  One CTA per (sequence, KV head), 128 threads.
__global__ void __launch_bounds__(128)
    full_combine_kernel(const int64_t *__restrict__ pos, const int32_t *__restrict__ seq, int hq, int G,
                        int hkv, int num_seqs, int64_t max_pos, long long max_ctx, int splits, int split_len,
                        const float *__restrict__ part_ml, const float *__restrict__ part_o,
                        uint16_t *__restrict__ out) {
  const int b = blockIdx.x / hkv, kv = blockIdx.x % hkv;
  const int d = threadIdx.x;
  const long long p = pos[b];
  const int s = seq[b];
  const bool ok = p >= 0 && p < max_pos && p + 1 <= max_ctx && s >= 0 && s < num_seqs;
  const int n = ok ? (int)(p / split_len) + 1 : 0;
  uint16_t *orow = out + ((long long)b * hq + (long long)kv * G) * DV;
  for (int g = 0; g < G; ++g) {
    float M = NEG_INF;
    for (int i = 0; i < n; ++i) {
      const long long w = ((long long)b * splits + i) * hkv + kv;
      M = fmaxf(M, part_ml[(w * G + g) * 2]);
    }
    float L = 0.f, acc = 0.f;
    for (int i = 0; i < n; ++i) {
      const long long w = ((long long)b * splits + i) * hkv + kv;
      const float mi = part_ml[(w * G + g) * 2];
      const float f = mi == NEG_INF ? 0.f : ex2(mi - M);
      L += part_ml[(w * G + g) * 2 + 1] * f;
      acc += part_o[(w * G + g) * DV + d] * f;
    }
    orow[g * DV + d] = f2bf(L > 0.f ? acc / L : 0.f);
  }
}

}  // namespace

// ---------------------------------------------------------------------------

cudaError_t launch_swa_decode(const uint16_t *q, const int64_t *pos, const int32_t *seq, int B, int hq,
                              const KvView &ring, const float *sinks, const float *table,
                              int64_t max_pos, float softmax_scale, uint16_t *out, unsigned *status,
                              cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(swa_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SWA_SMEM);
  if (e != cudaSuccess) return e;
  const int G = hq / ring.hkv;
  swa_decode_kernel<<<B * ring.hkv, SWA_WARPS * 32, SWA_SMEM, st>>>(q, pos, seq, hq, G, ring, sinks, table,
                                                                  max_pos, softmax_scale * LOG2E, out, status);
  return cudaGetLastError();
}

DecodePlan full_decode_plan(int B, int hkv, long long max_ctx) {
  long long len0 = ((long long)B * hkv * max_ctx + FD_TARGET_ITEMS - 1) / FD_TARGET_ITEMS;
  if (len0 < 512) len0 = 512;
  if (len0 > 8192) len0 = 8192;
  long long n = (max_ctx + len0 - 1) / len0;
  long long len = ((max_ctx + n - 1) / n + 63) / 64 * 64;
  n = (max_ctx + len - 1) / len;
  DecodePlan pl;
  pl.splits = (int)n;
  pl.split_len = (int)len;
  return pl;
}

static size_t align256(size_t x) { return (x + 255) / 256 * 256; }

size_t full_decode_workspace(int B, int hq, int hkv, long long max_ctx) {
  const DecodePlan pl = full_decode_plan(B, hkv, max_ctx);
  const size_t items = (size_t)B * pl.splits * hkv;
  const size_t G = (size_t)(hq / hkv);
  return align256(items * G * 2 * sizeof(float)) + align256(items * G * DV * sizeof(float));
}

cudaError_t launch_full_decode(const uint16_t *q, const int64_t *pos, const int32_t *seq, int B, int hq,
                               const KvView &pool, const float *table, int64_t max_pos,
                               float softmax_scale, long long max_ctx, void *ws, uint16_t *out,
                               unsigned *status, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(full_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, FD_SMEM);
  if (e != cudaSuccess) return e;
  const int hkv = pool.hkv, G = hq / hkv;
  const DecodePlan pl = full_decode_plan(B, hkv, max_ctx);
  const size_t items = (size_t)B * pl.splits * hkv;
  float *part_ml = reinterpret_cast<float *>(ws);
  float *part_o = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(ws) +
                                            align256(items * G * 2 * sizeof(float)));
  long long grid = (long long)num_sms() * 2;
  if (grid > (long long)items) grid = (long long)items;
  full_decode_kernel<<<(unsigned)grid, FD_WARPS * 32, FD_SMEM, st>>>(
      q, pos, seq, B, hq, G, pool, table, max_pos, softmax_scale * LOG2E, max_ctx, pl.splits, pl.split_len,
      part_ml, part_o, status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  full_combine_kernel<<<B * hkv, 128, 0, st>>>(pos, seq, hq, G, hkv, pool.num_seqs, max_pos, max_ctx, pl.splits,
                                               pl.split_len, part_ml, part_o, out);
  return cudaGetLastError();
}

}  // namespace kvr
