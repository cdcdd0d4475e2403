// warp_attn.cuh -- warp-level pieces of the decode kernels: rotated query
// tile staging, m16n8k16 bf16 products over 16-key subtiles with the GQA
// group as the 16 MMA rows, online softmax in the base-2 domain, and the
// per-warp state hand-off used by the cross-warp merges.
#pragma once

#include "common.cuh"

namespace kvr {
namespace {

constexpr float NEG_INF = -INFINITY;

// Rotated query tile in steps.  q_rows_issue: cp.async copies of the G query
// heads of one token (q_heads [G][192]) into rows 0..G-1 of the swizzled
// [16][192] tile sQ (rows G..15 zero-filled); q_table_issue: of the table row
// cs_row ([32][2] fp32, 256 B) into sCS, closing the commit group.  Copies
// issued after that group (the first key subtiles) queue behind it, not in
// front of it.  q_tile_rotate, once the group has landed and the block has
// synchronised: rotate dims 0..63 of each row in place and round to bf16
// (threads 0..63, one (row, chunk pair c, c + 4) each).
template <int NTH>
__device__ __forceinline__ void q_rows_issue(const uint16_t *__restrict__ q_heads, int G, uint8_t *sQ, int tid) {
  const uint32_t qb = smem_u32(sQ);
  // opaque copy of tid: keeps the compiler from hoisting these per-thread
  // offsets out of a caller's item loop and holding them in registers
  asm volatile("" : "+r"(tid));
#pragma unroll
  for (int k = 0; k < (16 * 24 + NTH - 1) / NTH; ++k) {
    const int it = tid + k * NTH, r = it / 24, c = it % 24;
    if (it < 16 * 24) cp_async16(qb + swz<DQK>(r, c), q_heads + (r < G ? r : 0) * DQK + c * 8, r < G ? 16 : 0);
  }
}

__device__ __forceinline__ void q_table_issue(const float *__restrict__ cs_row, uint8_t *sCS, int tid) {
  if (tid < 16) cp_async16(smem_u32(sCS) + 16 * tid, cs_row + 4 * tid);
  cp_async_commit();
}

__device__ __forceinline__ void q_tile_rotate(int G, uint8_t *sQ, const uint8_t *sCS, int tid) {
  const int r = tid >> 2, c = tid & 3;
  if (tid >= 64 || r >= G) return;
  uint4 *p1 = reinterpret_cast<uint4 *>(sQ + swz<DQK>(r, c));
  uint4 *p2 = reinterpret_cast<uint4 *>(sQ + swz<DQK>(r, c + 4));
  const float *cs = reinterpret_cast<const float *>(sCS) + 16 * c;
  uint4 o1, o2;
  rope_pair8(*p1, *p2, cs, o1, o2);
  *p1 = o1;
  *p2 = o2;
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
// [*][192] tile (chunk swizzle of swz<DQK>).
// Byte offset of 16-byte chunk ch of row r of a 16-row subtile: the
// XOR-swizzled [16][ROW_ELEMS] tile of the cp.async path, or (PARTED) the
// [16][ROW_ELEMS / 64][128 B] tile that a TMA box of all parts x 16 rows
// writes with the 128-byte swizzle (conflict-free ldmatrix for 3 parts, 2-way
// for 2).
template <int ROW_ELEMS, bool PARTED>
__device__ __forceinline__ uint32_t sub_off(int r, int ch) {
  if (PARTED) return swrow<ROW_ELEMS / 64>(r, ch);
  return swz<ROW_ELEMS>(r, ch);
}

template <bool PARTED = false>
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
    ldsm_x4(kbase + sub_off<DQK, PARTED>(row, 2 * kk + csel), b0, b1, b2, b3);
    mma_bf16(S[0], qf[kk], b0, b1);
    mma_bf16(S[1], qf[kk], b2, b3);
  }
}

// O[16 x 128] += P[16 x 16 keys] V[16 keys x 128] for the V rows starting at
// row r0 of a swizzled [*][128] tile; P comes from the S accumulators.
template <bool PARTED = false>
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
    ldsm_x4_t(vbase + sub_off<DV, PARTED>(row, 2 * dp + csel), b0, b1, b2, b3);
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

// Row stride (floats) of the per-warp numerators in the merge areas: 128 + 8,
// so the 8 rows a quad-group writes at once fall on different banks.
constexpr int MO_STRIDE = DV + 8;

// Write one warp's (m, l, O) into the merge area: ml [16][2], o [16][MO_STRIDE].
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
    *reinterpret_cast<float2 *>(o + r * MO_STRIDE + 8 * nt + cq) = make_float2(O[nt][0], O[nt][1]);
    *reinterpret_cast<float2 *>(o + (r + 8) * MO_STRIDE + 8 * nt + cq) = make_float2(O[nt][2], O[nt][3]);
  }
}

}  // namespace
}  // namespace kvr
