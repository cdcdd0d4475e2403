// prefill.cu -- chunked prefill over a windowed layer: the ring's state
// before the chunk plus the chunk's own rows, with the sink.
//
// gaudi-cookbook "MiMo-V2.6-Flash on Gaudi 2": "What was built" (windowed
// prefill with an fp32 softmax whose denominator includes the sink) and
// "Tiled global-attention prefill" (softmax is per query row, so tiles over
// query rows need no merge).  A row attends at most 128 keys, so the whole
// layer is about 1/1000 of a full layer's products at an 8192-token chunk;
// it runs on the warp-level bf16 MMA (mma.sync) with an online softmax.
// The query rows of one CTA are 64 consecutive (position, head) pairs of one
// KV head's group, so every K/V tile staged in shared memory serves all the
// heads that read it.  The softmax state of a row starts from the sink:
// (m, l, o) = (sink, 1, 0), which puts e^{sink} in the denominator and
// nowhere else.
#include "launch.h"

namespace kvr {
namespace {

constexpr float NEG_INF = -INFINITY;
constexpr int PF_WARPS = 4;
constexpr int PF_ROWS = PF_WARPS * 16;            // 64 query rows per CTA
constexpr int PF_KT = 64;                         // keys per tile
constexpr int PF_TILE_K = PF_KT * DQK * 2;        // 24 KB
constexpr int PF_TILE_V = PF_KT * DV * 2;         // 16 KB
constexpr int PF_STAGE = PF_TILE_K + PF_TILE_V + PF_KT * 4;
constexpr int PF_STAGES = 2;
constexpr int PF_SMEM = PF_ROWS * DQK * 2 + PF_STAGES * PF_STAGE;

// Where key position j of the current sequence lives.
struct SwaSrc {
  const uint16_t *rk, *rv;   // ring of this (sequence, KV head): [128][192], [128][128]
  const int32_t *slot_pos;   // [128] of this sequence
  const uint16_t *ck, *cv;   // chunk rows: [C][hkv][192], [C][hkv][128]
  int hkv, kv;
  long long P0;
  // Point at sequence sq's rings and at the chunk rows from batch row c0.
  __device__ __forceinline__ void rebase(int sq, long long c0, long long p0) {
    rk += (long long)sq * hkv * WIN * DQK;
    rv += (long long)sq * hkv * WIN * DV;
    slot_pos += (long long)sq * WIN;
    ck += c0 * hkv * DQK;
    cv += c0 * hkv * DV;
    P0 = p0;
  }
  __device__ __forceinline__ bool locate(long long j, const uint16_t *&kp, const uint16_t *&vp) const {
    if (j >= P0) {
      const long long row = (j - P0) * hkv + kv;
      kp = ck + row * DQK;
      vp = cv + row * DV;
      return true;
    }
    const int slot = (int)(j & (WIN - 1));
    if (slot_pos[slot] != (int32_t)j) return false;  // the ring no longer (or not yet) holds j
    kp = rk + slot * DQK;
    vp = rv + slot * DV;
    return true;
  }
};

template <int NT>
__device__ __forceinline__ void softmax_update_n(float (&S)[NT][4], float &m0, float &m1, float &l0, float &l1,
                                                 float (&O)[16][4]) {
  float r0 = NEG_INF, r1 = NEG_INF;
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    r0 = fmaxf(r0, fmaxf(S[j][0], S[j][1]));
    r1 = fmaxf(r1, fmaxf(S[j][2], S[j][3]));
  }
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
  for (int j = 0; j < NT; ++j) {
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

// One CTA: 64 (position, head) rows of KV head kv, flat rows
// f0 .. f0+63 of the [C x G] row space (position f / G, head f % G).
// VARLEN: the chunk, row tile and KV head come from the plan, and src0, q
// and out point at sequence 0 / row 0 of the batch.
template <class Src, bool SINK, bool VARLEN>
__global__ void __launch_bounds__(PF_WARPS * 32, 2)
    prefill_kernel(const uint16_t *__restrict__ q, long long P0, int C, int hq, int G, int hkv, Src src0,
                   const float *__restrict__ sinks, const float *__restrict__ table, float scale_log2,
                   uint16_t *__restrict__ out, unsigned *status, const VarlenPlan plan) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *sQ = smem;
  uint8_t *sStage = smem + PF_ROWS * DQK * 2;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int kv;
  long long f0;
  Src src = src0;
  if constexpr (VARLEN) {
    const long long b = blockIdx.x;
    if (b >= plan.item_prefix[plan.n]) return;
    const int s = plan_find(plan.item_prefix, plan.n, b);
    const int local = (int)(b - plan.item_prefix[s]);
    kv = local % hkv;
    f0 = (long long)(local / hkv) * PF_ROWS;
    const long long c0 = plan.cu_rows[s];
    C = (int)(plan.cu_rows[s + 1] - c0);
    q += c0 * hq * DQK;
    out += c0 * hq * DV;
    if (plan.mode[s] <= 0) {  // a position or the sequence id is out of range
      for (int it = tid; it < PF_ROWS * 16; it += blockDim.x) {
        const long long f = f0 + it / 16;
        if (f < (long long)C * G)
          reinterpret_cast<uint4 *>(out + ((f / G) * hq + (long long)kv * G + f % G) * DV)[it % 16] =
              make_uint4(0, 0, 0, 0);
      }
      return;
    }
    P0 = plan.P0[s];
    src.rebase(plan.seq[s], c0, P0);
  } else {
    kv = blockIdx.x % hkv;
    f0 = (long long)(blockIdx.x / hkv) * PF_ROWS;
  }
  const long long nrows = (long long)C * G;
  src.kv = kv;
  if constexpr (SINK) {
    src.rk += (long long)kv * WIN * DQK;
    src.rv += (long long)kv * WIN * DV;
  }

  // Positions covered by this CTA.
  const long long i_first = f0 / G;
  const long long i_last = min(nrows - 1, f0 + PF_ROWS - 1) / G;
  long long key_lo = SINK ? max(0LL, P0 + i_first - (WIN - 1)) : 0LL;
  const long long key_hi = P0 + i_last + 1;  // exclusive
  if (!SINK) key_lo = 0;
  const int ntiles = (int)((key_hi - key_lo + PF_KT - 1) / PF_KT);

  // Stage the rotated Q rows.
  for (int it = tid; it < PF_ROWS * 20; it += blockDim.x) {
    const int r = it / 20, c = it % 20;
    const long long f = f0 + r;
    const bool live = f < nrows;
    const long long i = live ? f / G : 0;
    const int g = live ? (int)(f % G) : 0;
    const uint16_t *qh = q + (i * hq + (long long)kv * G + g) * DQK;
    const uint4 zero = make_uint4(0, 0, 0, 0);
    if (c < 4) {
      uint4 o1 = zero, o2 = zero;
      if (live) {
        const float4 *tr = reinterpret_cast<const float4 *>(table + (P0 + i) * 64 + 16 * c);
        float cs[16];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float4 fv = tr[u];
          cs[4 * u] = fv.x; cs[4 * u + 1] = fv.y; cs[4 * u + 2] = fv.z; cs[4 * u + 3] = fv.w;
        }
        const uint4 *s4 = reinterpret_cast<const uint4 *>(qh);
        rope_pair8(s4[c], s4[c + 4], cs, o1, o2);
      }
      *reinterpret_cast<uint4 *>(sQ + swz<DQK>(r, c)) = o1;
      *reinterpret_cast<uint4 *>(sQ + swz<DQK>(r, c + 4)) = o2;
    } else {
      const int ch = c + 4;
      const uint4 x = live ? reinterpret_cast<const uint4 *>(qh)[ch] : zero;
      *reinterpret_cast<uint4 *>(sQ + swz<DQK>(r, ch)) = x;
    }
  }

  // Tile loader: thread t fills half of key row t/2 (12 K chunks + 8 V chunks).
  auto issue = [&](int t) {
    uint8_t *st = sStage + (t % PF_STAGES) * PF_STAGE;
    const uint32_t kb = smem_u32(st), vb = kb + PF_TILE_K;
    int32_t *sValid = reinterpret_cast<int32_t *>(st + PF_TILE_K + PF_TILE_V);
    const int r = tid >> 1, half = tid & 1;
    const long long j = key_lo + (long long)t * PF_KT + r;
    const uint16_t *kp = nullptr, *vp = nullptr;
    bool ok = j < key_hi && src.locate(j, kp, vp);
    if (!ok) { kp = q; vp = q; }  // any mapped address; zero bytes are read
    const int nb = ok ? 16 : 0;
#pragma unroll
    for (int u = 0; u < 12; ++u) {
      const int ch = half * 12 + u;
      cp_async16(kb + swz<DQK>(r, ch), kp + ch * 8, nb);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int ch = half * 8 + u;
      cp_async16(vb + swz<DV>(r, ch), vp + ch * 8, nb);
    }
    if (half == 0) sValid[r] = ok ? 1 : 0;
  };

  if (ntiles > 0) issue(0);
  cp_async_commit();
  __syncthreads();  // Q staged

  uint32_t qf[12][4];
  {
    const uint32_t base = smem_u32(sQ);
#pragma unroll
    for (int kk = 0; kk < 12; ++kk)
      ldsm_x4(base + swz<DQK>(16 * warp + (lane & 15), 2 * kk + (lane >> 4)), qf[kk][0], qf[kk][1], qf[kk][2],
              qf[kk][3]);
  }

  // This thread's two rows: their positions and heads.
  const int rr0 = 16 * warp + (lane >> 2), rr1 = rr0 + 8;
  const long long fa = f0 + rr0, fb = f0 + rr1;
  const long long pa = P0 + min(fa, nrows - 1) / G, pb = P0 + min(fb, nrows - 1) / G;
  const int ga = (int)(min(fa, nrows - 1) % G), gb = (int)(min(fb, nrows - 1) % G);

  float O[16][4];
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) O[nt][0] = O[nt][1] = O[nt][2] = O[nt][3] = 0.f;
  float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;
  if constexpr (SINK) {
    m0 = sinks[kv * G + ga] * LOG2E;
    m1 = sinks[kv * G + gb] * LOG2E;
    l0 = l1 = (lane & 3) == 0 ? 1.f : 0.f;
  }

  for (int t = 0; t < ntiles; ++t) {
    if (t + 1 < ntiles) issue(t + 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const uint8_t *st = sStage + (t % PF_STAGES) * PF_STAGE;
    const uint32_t kb = smem_u32(st), vb = kb + PF_TILE_K;
    const int32_t *sValid = reinterpret_cast<const int32_t *>(st + PF_TILE_K + PF_TILE_V);
    const long long kbase = key_lo + (long long)t * PF_KT;

    float S[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) S[j][0] = S[j][1] = S[j][2] = S[j][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 12; ++kk) {
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        uint32_t b0, b1, b2, b3;
        const int row = 16 * jj + (lane & 7) + ((lane >> 4) << 3);
        ldsm_x4(kb + swz<DQK>(row, 2 * kk + ((lane >> 3) & 1)), b0, b1, b2, b3);
        mma_bf16(S[2 * jj], qf[kk], b0, b1);
        mma_bf16(S[2 * jj + 1], qf[kk], b2, b3);
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int kr = 8 * j + 2 * (lane & 3) + (e & 1);
        const long long key = kbase + kr;
        const long long pr = e < 2 ? pa : pb;
        bool ok = sValid[kr] != 0 && key <= pr;
        if (SINK) ok = ok && key > pr - WIN;
        S[j][e] = ok ? S[j][e] * scale_log2 : NEG_INF;
      }
    softmax_update_n<8>(S, m0, m1, l0, l1, O);
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      uint32_t a[4];
      a[0] = pack_bf16(S[2 * s][0], S[2 * s][1]);
      a[1] = pack_bf16(S[2 * s][2], S[2 * s][3]);
      a[2] = pack_bf16(S[2 * s + 1][0], S[2 * s + 1][1]);
      a[3] = pack_bf16(S[2 * s + 1][2], S[2 * s + 1][3]);
      const int row = 16 * s + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + swz<DV>(row, 2 * dp + (lane >> 4)), b0, b1, b2, b3);
        mma_bf16(O[2 * dp], a, b0, b1);
        mma_bf16(O[2 * dp + 1], a, b2, b3);
      }
    }
    __syncthreads();  // stage t % 2 is refilled by the next iteration's issue
  }
  cp_async_wait<0>();

  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  const int cq = 2 * (lane & 3);
  if (fa < nrows) {
    uint16_t *o = out + ((pa - P0) * hq + (long long)kv * G + ga) * DV;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
      *reinterpret_cast<uint32_t *>(o + 8 * nt + cq) = pack_bf16(O[nt][0] * inv0, O[nt][1] * inv0);
  }
  if (fb < nrows) {
    uint16_t *o = out + ((pb - P0) * hq + (long long)kv * G + gb) * DV;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
      *reinterpret_cast<uint32_t *>(o + 8 * nt + cq) = pack_bf16(O[nt][2] * inv1, O[nt][3] * inv1);
  }
  (void)status;
}


}  // namespace

cudaError_t launch_swa_prefill(const uint16_t *q, int64_t P0, int C, int seq, int hq, const KvView &chunk,
                               const KvView &ring, const float *sinks, const float *table,
                               int64_t max_pos, float softmax_scale, uint16_t *out, unsigned *status,
                               cudaStream_t st) {
  (void)max_pos;
  const int hkv = ring.hkv, G = hq / hkv;
  auto kern = prefill_kernel<SwaSrc, true, false>;
  cudaError_t e = ensure_smem_limit(3, (const void *)kern, PF_SMEM);
  if (e != cudaSuccess) return e;
  SwaSrc src{ring.k + (long long)seq * hkv * WIN * DQK, ring.v + (long long)seq * hkv * WIN * DV,
             ring.slot_pos + (long long)seq * WIN, chunk.k, chunk.v, hkv, 0, P0};
  const long long tiles = ((long long)C * G + PF_ROWS - 1) / PF_ROWS;
  kern<<<(unsigned)(tiles * hkv), PF_WARPS * 32, PF_SMEM, st>>>(q, P0, C, hq, G, hkv, src, sinks, table,
                                                                 softmax_scale * LOG2E, out, status, VarlenPlan{});
  return cudaGetLastError();
}

cudaError_t launch_swa_varlen(const uint16_t *q, const int32_t *cu_rows, const int64_t *P0, const int32_t *seq,
                              int n, long long T, int hq, const KvView &chunk, const KvView &ring,
                              const float *sinks, const float *table, int64_t max_pos, float softmax_scale,
                              void *ws, uint16_t *out, unsigned *status, cudaStream_t st) {
  const int hkv = ring.hkv, G = hq / hkv;
  auto kern = prefill_kernel<SwaSrc, true, true>;
  cudaError_t e = ensure_smem_limit(5, (const void *)kern, PF_SMEM);
  if (e != cudaSuccess) return e;
  const VarlenSizes z = varlen_sizes(n, T, hq, hkv, max_pos, PF_ROWS, false);
  const VarlenPlan plan = varlen_plan_view(z, ws, cu_rows, P0, seq, n);
  e = launch_varlen_plan(plan, T, hq, hkv, PF_ROWS, max_pos, ring.num_seqs, SWA_SHORT_ROWS, SWA_SHORT_MAX_C, status,
                         st);
  if (e != cudaSuccess) return e;
  // Short chunks (a few tokens per sequence) go to the short-chunk kernel;
  // the rest are tiled here.
  SwaSrc src{ring.k, ring.v, ring.slot_pos, chunk.k, chunk.v, hkv, 0, 0};
  kern<<<(unsigned)z.items_max, PF_WARPS * 32, PF_SMEM, st>>>(q, 0, 0, hq, G, hkv, src, sinks, table,
                                                              softmax_scale * LOG2E, out, status, plan);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_swa_short(q, plan, n, T, hq, chunk, ring, sinks, table, softmax_scale, out, status, st);
}

}  // namespace kvr
