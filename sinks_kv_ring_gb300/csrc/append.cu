// append.cu -- fused KV write: rotate-half RoPE of k (dims 0..63), value
// scale of v, bf16 store into a ring slot, a pool page or a staging row.
//
// Follows colibri "MiMo-V2.6", "What the engine implements" (partial RoPE on
// the first 64 of 192 dims, rotate-half; values multiplied by
// attention_value_scale) and "System One mode and prompt reuse" (position p
// lives in ring slot p mod 128, and the ring records which position each slot
// holds).
//
// One warp per APPEND_ITEMS = 8 consecutive (token, KV head) items, i.e. 320
// chunks of 16 bytes (24 of k and 16 of v per item), 10 per lane, split so that
// every phase runs converged across the warp:
//   rope   lane L rotates the chunk pair (c, c+4), c = L mod 4, of item L / 4
//          (dims 8c..8c+7 with 32+8c..32+8c+7);
//   copy   4 chunks per lane of dims 64..191, stored bit for bit;
//   scale  4 chunks per lane of v, multiplied by the value scale.
// Lanes 0..7 resolve the destination row of one item each (position check,
// sequence, block table) while the source chunks are already in flight; the
// phases fetch the row of their item by shuffle.  Pure bandwidth: the
// per-item instruction count is what the layout keeps small.
#include "launch.h"

namespace kvr {
namespace {

constexpr int APPEND_WARPS = 8;
constexpr int APPEND_ITEMS = 8;
constexpr unsigned FULLW = 0xffffffffu;

__device__ __forceinline__ uint4 scale8(const uint4 x, float vscale) {
  const uint16_t *e = reinterpret_cast<const uint16_t *>(&x);
  uint4 y;
  y.x = pack_bf16(bf2f(e[0]) * vscale, bf2f(e[1]) * vscale);
  y.y = pack_bf16(bf2f(e[2]) * vscale, bf2f(e[3]) * vscale);
  y.z = pack_bf16(bf2f(e[4]) * vscale, bf2f(e[5]) * vscale);
  y.w = pack_bf16(bf2f(e[6]) * vscale, bf2f(e[7]) * vscale);
  return y;
}

__global__ void __launch_bounds__(APPEND_WARPS * 32)
    append_kernel(const uint16_t *__restrict__ k, const uint16_t *__restrict__ v,
                  const int64_t *__restrict__ pos, const int32_t *__restrict__ seq, int T, int hkv,
                  const float *__restrict__ table, int64_t max_pos, float vscale, KvView dst,
                  unsigned *status) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const long long total = (long long)T * hkv;
  const long long base = ((long long)blockIdx.x * APPEND_WARPS + (threadIdx.x >> 5)) * APPEND_ITEMS;
  if (base >= total) return;  // warp-uniform
  const int nit = (int)(total - base < APPEND_ITEMS ? total - base : APPEND_ITEMS);

  // 1. source chunks (item-major rows: 24 chunks of k, 16 of v)
  const uint4 *K4 = reinterpret_cast<const uint4 *>(k) + base * (DQK / 8);
  const uint4 *V4 = reinterpret_cast<const uint4 *>(v) + base * (DV / 8);
  const int ri = lane >> 2, rc = lane & 3;
  uint4 r0 = make_uint4(0, 0, 0, 0), r1 = r0, kc[4], vc[4];
  if (ri < nit) {
    r0 = K4[ri * 24 + rc];
    r1 = K4[ri * 24 + rc + 4];
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int q = j * 32 + lane, it = q >> 4;
    if (it < nit) {
      kc[j] = K4[it * 24 + 8 + (q & 15)];
      vc[j] = V4[it * 16 + (q & 15)];
    }
  }

  // 2. destination head-row of item `lane` (lanes 0..7), -1 when it is skipped
  long long row = -1, p = 0;
  if (lane < nit) {
    const long long item = base + lane;
    const int t = (int)(item / hkv);
    const int h = (int)(item - (long long)t * hkv);
    p = pos[t];
    if (p < 0 || p >= max_pos) {
      flag(status, ST_BAD_POS);
    } else if (dst.kind == 3) {
      row = item;
    } else {
      const int s = seq[t];
      if (s < 0 || s >= dst.num_seqs) {
        flag(status, ST_BAD_SEQ);
      } else if (dst.kind == 1) {
        const int slot = (int)(p & (WIN - 1));
        row = ((long long)s * hkv + h) * WIN + slot;
        if (h == 0) dst.slot_pos[(long long)s * WIN + slot] = (int32_t)p;
      } else {
        const long long bi = p / dst.block_size;
        const int blk = bi < dst.max_blocks ? dst.block_table[(long long)s * dst.max_blocks + bi] : -1;
        if (blk < 0 || blk >= dst.num_blocks)
          flag(status, ST_BAD_BLOCK);
        else
          row = ((long long)blk * hkv + h) * dst.block_size + (p - bi * dst.block_size);
      }
    }
  }

  // 3. rope phase
  {
    const long long rr = __shfl_sync(FULLW, row, ri);
    const long long rp = __shfl_sync(FULLW, p, ri);
    if (rr >= 0) {
      const float4 *tr = reinterpret_cast<const float4 *>(table + rp * 64 + 16 * rc);
      float cs[16];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float4 f = tr[u];
        cs[4 * u] = f.x; cs[4 * u + 1] = f.y; cs[4 * u + 2] = f.z; cs[4 * u + 3] = f.w;
      }
      uint4 o1, o2;
      rope_pair8(r0, r1, cs, o1, o2);
      uint4 *kd = reinterpret_cast<uint4 *>(dst.k + rr * DQK);
      kd[rc] = o1;
      kd[rc + 4] = o2;
    }
  }

  // 4. copy and scale phases
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int q = j * 32 + lane;
    const long long rr = __shfl_sync(FULLW, row, q >> 4);
    if (rr >= 0) {
      reinterpret_cast<uint4 *>(dst.k + rr * DQK)[8 + (q & 15)] = kc[j];
      reinterpret_cast<uint4 *>(dst.v + rr * DV)[q & 15] = scale8(vc[j], vscale);
    }
  }
}

}  // namespace

cudaError_t launch_append(const uint16_t *k, const uint16_t *v, const int64_t *pos, const int32_t *seq,
                          int T, int hkv, const float *table, int64_t max_pos, float value_scale,
                          const KvView &dst, unsigned *status, cudaStream_t st) {
  const long long items = (long long)T * hkv;
  const long long per_block = (long long)APPEND_WARPS * APPEND_ITEMS;
  const long long blocks = (items + per_block - 1) / per_block;
  return launch_pdl(append_kernel, dim3((unsigned)blocks), dim3(APPEND_WARPS * 32), 0, st, k, v, pos, seq, T, hkv,
                    table, max_pos, value_scale, dst, status);
}

}  // namespace kvr
