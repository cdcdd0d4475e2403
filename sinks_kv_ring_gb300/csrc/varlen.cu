// varlen.cu -- batches of chunks of different lengths: the device-side work
// plan, and the merge of key-split partials.
//
// A batch holds n chunks; chunk s is C_s rows at positions P0_s .. P0_s+C_s-1
// of sequence seq_s.  With C_s = 1 this is a decode step, with C_s = 2..4 the
// verification of a multi-token-prediction draft (the Chinese Xiaomi article,
// section "Decode加速与多模态优化": the model proposes several tokens per step
// and checks them together), and with large C_s a prefill chunk (section
// "调度与Prefill优化": requests of very different lengths batched by length
// bucket).  The plan is built on the device, so a batch can be launched from
// device-resident lengths and captured in a CUDA graph.
#include <algorithm>

#include "launch.h"

namespace kvr {
namespace {

constexpr int PLAN_THREADS = 1024;

struct PlanArgs {
  VarlenPlan p;
  long long T;          // rows of the batch
  int hq, hkv, G;
  int tile_rows;        // query rows of one CTA item
  long long max_ctx;    // P0 + C must not exceed it
  int num_seqs;
  int short_rows, short_max_c;  // 0: no short-chunk kernel
  unsigned *status;
};

// One CTA: per chunk its mode, item / partial-row counts and short flag,
// then exclusive prefix sums, 1024 chunks at a time.
__global__ void __launch_bounds__(PLAN_THREADS) varlen_plan_kernel(const PlanArgs a) {
  __shared__ int wsum[32][3];
  __shared__ int carry[3];
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) carry[0] = carry[1] = carry[2] = 0;
  __syncthreads();
  for (int base = 0; base < a.p.n; base += PLAN_THREADS) {
    const int s = base + tid;
    int items = 0, prows = 0, shrt = 0;
    if (s < a.p.n) {
      int mode = 1;
      const long long c0 = a.p.cu_rows[s], c1 = a.p.cu_rows[s + 1];
      if (c0 < 0 || c1 < c0 || c1 > a.T) {
        flag(a.status, ST_BAD_ROWS);
        mode = -1;
      } else if (c1 > c0) {
        const long long C = c1 - c0, P0 = a.p.P0[s];
        const int sq = a.p.seq[s];
        const long long tiles = (C * a.G + a.tile_rows - 1) / a.tile_rows;
        bool bad = false;
        if (sq < 0 || sq >= a.num_seqs) { flag(a.status, ST_BAD_SEQ); bad = true; }
        if (P0 < 0 || P0 + C > a.max_ctx) { flag(a.status, ST_BAD_POS); bad = true; }
        if (bad) {
          mode = 0;
          items = (int)(tiles * a.hkv);
        } else if (a.short_rows > 0 && C * a.G <= a.short_rows && C <= a.short_max_c) {
          shrt = 1;
        } else if (a.p.split_len > 0 && tiles == 1) {
          // splits of equal length (a multiple of 128) covering the P0 + C keys
          const long long ctx = P0 + C;
          const long long n0 = (ctx + a.p.split_len - 1) / a.p.split_len;
          const long long L = ((ctx + n0 - 1) / n0 + 127) / 128 * 128;
          const int nsp = (int)((ctx + L - 1) / L);
          mode = nsp;
          a.p.slen[s] = (int)L;
          items = nsp * a.hkv;
          prows = nsp > 1 ? (int)(C * a.hq) : 0;
        } else {
          items = (int)(tiles * a.hkv);
        }
      }
      a.p.mode[s] = mode;
    }
    // block-wide exclusive scan of (items, prows, short)
    int v[3] = {items, prows, shrt};
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        const int t = __shfl_up_sync(0xffffffffu, v[k], d);
        if (lane >= d) v[k] += t;
      }
    }
    if (lane == 31)
      for (int k = 0; k < 3; ++k) wsum[warp][k] = v[k];
    __syncthreads();
    if (warp == 0) {
      int w[3] = {wsum[lane][0], wsum[lane][1], wsum[lane][2]};
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
#pragma unroll
        for (int k = 0; k < 3; ++k) {
          const int t = __shfl_up_sync(0xffffffffu, w[k], d);
          if (lane >= d) w[k] += t;
        }
      }
      for (int k = 0; k < 3; ++k) wsum[lane][k] = w[k];  // inclusive over warps
    }
    __syncthreads();
    if (s < a.p.n) {
      a.p.item_prefix[s] = carry[0] + (warp ? wsum[warp - 1][0] : 0) + v[0] - items;
      a.p.prow_prefix[s] = carry[1] + (warp ? wsum[warp - 1][1] : 0) + v[1] - prows;
      if (shrt) a.p.short_list[carry[2] + (warp ? wsum[warp - 1][2] : 0) + v[2] - 1] = s;
    }
    __syncthreads();
    if (tid == 0)
      for (int k = 0; k < 3; ++k) carry[k] += wsum[31][k];
    __syncthreads();
  }
  if (tid == 0) {
    a.p.item_prefix[a.p.n] = carry[0];
    a.p.prow_prefix[a.p.n] = carry[1];
    a.p.short_list[a.p.n] = carry[2];
  }
}

struct CombineArgs {
  VarlenPlan p;
  int hq;
  uint16_t *out;
};

// One warp per partial row (row, q head) of a split chunk: merge its splits
// by log-sum-exp (Xiaomi "Full-Pipeline Inference Optimization", section 1.2,
// split decode) and write the normalised bf16 row.  Lane = 4 value dims.
__global__ void __launch_bounds__(256) varlen_combine_kernel(const CombineArgs a) {
  pdl_wait();
  pdl_trigger();
  const long long r = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int total = a.p.prow_prefix[a.p.n];
  if (r >= total) return;
  const int s = plan_find(a.p.prow_prefix, a.p.n, r);
  const long long local = r - a.p.prow_prefix[s];
  const long long i = local / a.hq;
  const int h = (int)(local % a.hq);
  const int nsp = a.p.mode[s];
  const long long rec0 = r * a.p.nsp_max;
  float M = -INFINITY;
  for (int k = 0; k < nsp; ++k) M = fmaxf(M, a.p.pml[rec0 + k].x);
  float l = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -INFINITY) {
    for (int k = 0; k < nsp; ++k) {
      const float2 ml = a.p.pml[rec0 + k];
      const float w = ml.x == -INFINITY ? 0.f : ex2(ml.x - M);
      const float4 o = reinterpret_cast<const float4 *>(a.p.po + (rec0 + k) * DV)[lane];
      l += w * ml.y;
      acc.x += w * o.x;
      acc.y += w * o.y;
      acc.z += w * o.z;
      acc.w += w * o.w;
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  uint2 v;
  v.x = pack_bf16(acc.x * inv, acc.y * inv);
  v.y = pack_bf16(acc.z * inv, acc.w * inv);
  reinterpret_cast<uint2 *>(a.out + ((a.p.cu_rows[s] + i) * a.hq + h) * DV)[lane] = v;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

VarlenSizes varlen_sizes(int n, long long T, int hq, int hkv, long long max_ctx, int tile_rows, bool splits) {
  VarlenSizes z{};
  const int G = hq / hkv;
  z.tile_rows = tile_rows;
  z.split_len = 0;
  z.nsp_max = 1;
  const long long small_rows = std::min(T, (long long)n * (tile_rows / G));
  if (splits) {
    // Number of key splits for chunks of one query tile, from a cost model in
    // units of one 128-key tile on one SM (one CTA per SM): items run in
    // waves of `sms`; an item costs a set-up of about 1.6 tiles plus its
    // tiles; each split adds partial records (520 B written and read per row
    // and head) spread over all SMs.  Splits are at least 512 keys.
    const long long sms = num_sms();
    const long long units = (long long)n * hkv;
    const long long tiles = (max_ctx + 127) / 128;
    const double rec_cost = (double)small_rows * hq * 1040.0 / (80.0 * 1024.0 * (double)sms);
    int best = 1;
    double best_cost = 1e300;
    for (int nsp = 1; nsp <= 64 && (nsp == 1 || tiles / nsp >= 4); ++nsp) {
      const double waves = (double)((units * nsp + sms - 1) / sms);
      const double cost = waves * (1.6 + (double)((tiles + nsp - 1) / nsp)) + (nsp > 1 ? nsp * rec_cost : 0.0);
      if (cost < best_cost - 1e-9) {
        best_cost = cost;
        best = nsp;
      }
    }
    long long L = ((max_ctx + best - 1) / best + 127) / 128 * 128;
    z.split_len = L;
    z.nsp_max = (int)((max_ctx + L - 1) / L);
  }
  z.prows_max = z.nsp_max > 1 ? small_rows * hq : 0;
  const long long tiles = (T * G + tile_rows - 1) / tile_rows;
  // tiles: at most one partial tile per chunk; splits: only chunks of one tile
  z.items_max = (long long)hkv * (tiles + n + (splits ? (long long)n * z.nsp_max : 0));
  z.off_prow = align256(((size_t)n + 1) * 4);
  z.off_mode = z.off_prow + align256(((size_t)n + 1) * 4);
  z.off_short = z.off_mode + align256((size_t)n * 4);
  z.off_slen = z.off_short + align256(((size_t)n + 1) * 4);
  z.off_pml = z.off_slen + align256((size_t)n * 4);
  const size_t recs = (size_t)z.prows_max * z.nsp_max;
  z.off_po = z.off_pml + align256(recs * 8);
  z.bytes = z.off_po + recs * DV * 4;
  return z;
}

VarlenPlan varlen_plan_view(const VarlenSizes &z, void *ws, const int32_t *cu_rows, const int64_t *P0,
                            const int32_t *seq, int n) {
  uint8_t *b = static_cast<uint8_t *>(ws);
  VarlenPlan p;
  p.cu_rows = cu_rows;
  p.P0 = P0;
  p.seq = seq;
  p.item_prefix = reinterpret_cast<int32_t *>(b);
  p.prow_prefix = reinterpret_cast<int32_t *>(b + z.off_prow);
  p.mode = reinterpret_cast<int32_t *>(b + z.off_mode);
  p.short_list = reinterpret_cast<int32_t *>(b + z.off_short);
  p.slen = reinterpret_cast<int32_t *>(b + z.off_slen);
  p.pml = reinterpret_cast<float2 *>(b + z.off_pml);
  p.po = reinterpret_cast<float *>(b + z.off_po);
  p.n = n;
  p.nsp_max = z.nsp_max;
  p.split_len = z.split_len;
  return p;
}

cudaError_t launch_varlen_plan(const VarlenPlan &p, long long T, int hq, int hkv, int tile_rows, long long max_ctx,
                               int num_seqs, int short_rows, int short_max_c, unsigned *status, cudaStream_t st) {
  PlanArgs a;
  a.p = p;
  a.T = T;
  a.hq = hq;
  a.hkv = hkv;
  a.G = hq / hkv;
  a.tile_rows = tile_rows;
  a.max_ctx = max_ctx;
  a.num_seqs = num_seqs;
  a.short_rows = short_rows;
  a.short_max_c = short_max_c;
  a.status = status;
  return launch_pdl(varlen_plan_kernel, dim3(1), dim3(PLAN_THREADS), 0, st, a);
}

cudaError_t launch_varlen_combine(const VarlenPlan &p, long long prows_max, int hq, uint16_t *out, cudaStream_t st) {
  if (prows_max <= 0) return cudaSuccess;
  CombineArgs a;
  a.p = p;
  a.hq = hq;
  a.out = out;
  return launch_pdl(varlen_combine_kernel, dim3((unsigned)((prows_max + 7) / 8)), dim3(256), 0, st, a);
}

}  // namespace kvr
