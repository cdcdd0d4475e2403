// append.cu -- fused KV write: rotate-half RoPE of k (dims 0..63), value
// scale of v, bf16 store into a ring slot, a pool page or a staging row.
//
// Follows colibri "MiMo-V2.6", "What the engine implements" (partial RoPE on
// the first 64 of 192 dims, rotate-half; values multiplied by
// attention_value_scale) and "System One mode and prompt reuse" (position p
// lives in ring slot p mod 128, and the ring records which position each slot
// holds).
//
// One warp per (token, KV head).  A head is 40 chunks of 16 bytes (24 of k,
// 16 of v); lanes 0..3 rotate the chunk pairs (c, c+4) of dims 0..63, lanes
// 4..19 copy the 16 chunks of dims 64..191 untouched, lanes 20..31 and 0..3
// scale the 16 chunks of v.  All of it is pure bandwidth.
#include "launch.h"

namespace kvr {
namespace {

constexpr int APPEND_WARPS = 8;

__global__ void __launch_bounds__(APPEND_WARPS * 32)
    append_kernel(const uint16_t *__restrict__ k, const uint16_t *__restrict__ v,
                  const int64_t *__restrict__ pos, const int32_t *__restrict__ seq, int T, int hkv,
                  const float *__restrict__ table, int64_t max_pos, float vscale, KvView dst,
                  unsigned *status) {
  const int lane = threadIdx.x & 31;
  const long long item = (long long)blockIdx.x * APPEND_WARPS + (threadIdx.x >> 5);
  if (item >= (long long)T * hkv) return;
  const int t = (int)(item / hkv);
  const int h = (int)(item % hkv);

  const long long p = pos[t];
  if (p < 0 || p >= max_pos) {
    if (lane == 0) flag(status, ST_BAD_POS);
    return;
  }
  long long row;  // destination head-row index
  int s = 0;
  if (dst.kind == 3) {
    row = (long long)t * hkv + h;
  } else {
    s = seq[t];
    if (s < 0 || s >= dst.num_seqs) {
      if (lane == 0) flag(status, ST_BAD_SEQ);
      return;
    }
    if (dst.kind == 1) {
      row = ((long long)s * hkv + h) * WIN + (p & (WIN - 1));
    } else {
      const long long bi = p / dst.block_size;
      const int blk = bi < dst.max_blocks ? dst.block_table[(long long)s * dst.max_blocks + bi] : -1;
      if (blk < 0 || blk >= dst.num_blocks) {
        if (lane == 0) flag(status, ST_BAD_BLOCK);
        return;
      }
      row = ((long long)blk * hkv + h) * dst.block_size + (p % dst.block_size);
    }
  }

  const uint4 *ks = reinterpret_cast<const uint4 *>(k + item * DQK);
  const uint4 *vs = reinterpret_cast<const uint4 *>(v + item * DV);
  uint4 *kd = reinterpret_cast<uint4 *>(dst.k + row * DQK);
  uint4 *vd = reinterpret_cast<uint4 *>(dst.v + row * DV);

  if (lane < 4) {
    // dims 8c..8c+7 pair with 32+8c..32+8c+7
    const float4 *tr = reinterpret_cast<const float4 *>(table + p * 64 + 16 * lane);
    float cs[16];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float4 f = tr[u];
      cs[4 * u] = f.x; cs[4 * u + 1] = f.y; cs[4 * u + 2] = f.z; cs[4 * u + 3] = f.w;
    }
    uint4 o1, o2;
    rope_pair8(ks[lane], ks[lane + 4], cs, o1, o2);
    kd[lane] = o1;
    kd[lane + 4] = o2;
  } else if (lane < 20) {
    kd[lane + 4] = ks[lane + 4];  // chunks 8..23: dims 64..191, bit copy
  }
  const int vc0 = lane >= 20 ? lane - 20 : -1;
  const int vc1 = lane < 4 ? lane + 12 : -1;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int c = r == 0 ? vc0 : vc1;
    if (c >= 0) {
      const uint4 x = vs[c];
      const uint16_t *e = reinterpret_cast<const uint16_t *>(&x);
      uint4 y;
      y.x = pack_bf16(bf2f(e[0]) * vscale, bf2f(e[1]) * vscale);
      y.y = pack_bf16(bf2f(e[2]) * vscale, bf2f(e[3]) * vscale);
      y.z = pack_bf16(bf2f(e[4]) * vscale, bf2f(e[5]) * vscale);
      y.w = pack_bf16(bf2f(e[6]) * vscale, bf2f(e[7]) * vscale);
      vd[c] = y;
    }
  }
  if (dst.kind == 1 && h == 0 && lane == 0) dst.slot_pos[(long long)s * WIN + (p & (WIN - 1))] = (int32_t)p;
}

}  // namespace

cudaError_t launch_append(const uint16_t *k, const uint16_t *v, const int64_t *pos, const int32_t *seq,
                          int T, int hkv, const float *table, int64_t max_pos, float value_scale,
                          const KvView &dst, unsigned *status, cudaStream_t st) {
  const long long items = (long long)T * hkv;
  const long long blocks = (items + APPEND_WARPS - 1) / APPEND_WARPS;
  append_kernel<<<(unsigned)blocks, APPEND_WARPS * 32, 0, st>>>(k, v, pos, seq, T, hkv, table, max_pos,
                                                                 value_scale, dst, status);
  return cudaGetLastError();
}

}  // namespace kvr
