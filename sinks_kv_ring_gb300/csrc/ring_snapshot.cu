// ring_snapshot.cu -- copy the windowed layers' rings of chosen sequences to
// and from snapshot buffers (colibri "MiMo-V2.6 (Xiaomi)", "System One mode
// and prompt reuse": the rings are copied into a snapshot and back).  One CTA
// per (entry, KV head) moves that head's 48 KB of K and 32 KB of V with
// 16-byte accesses, COPY_BATCH loads in flight per thread before their
// stores; the KV-head-0 CTA also moves the 128 slot tags.
#include "launch.h"

namespace kvr {
namespace {

constexpr int COPY_THREADS = 256;
constexpr int COPY_BATCH = 4;

// n16 chunks of 16 bytes from src to dst (n16 a multiple of the batch stride)
__device__ __forceinline__ void copy_chunks(uint4 *__restrict__ dst, const uint4 *__restrict__ src, int n16) {
  for (int e0 = threadIdx.x; e0 < n16; e0 += COPY_THREADS * COPY_BATCH) {
    uint4 v[COPY_BATCH];
#pragma unroll
    for (int u = 0; u < COPY_BATCH; ++u) v[u] = src[e0 + u * COPY_THREADS];
#pragma unroll
    for (int u = 0; u < COPY_BATCH; ++u) dst[e0 + u * COPY_THREADS] = v[u];
  }
}

__global__ void __launch_bounds__(COPY_THREADS)
    ring_copy_kernel(KvView ring, const int32_t *__restrict__ seqs, uint16_t *k_snap, uint16_t *v_snap,
                     int32_t *tags_snap, int to_ring, unsigned *status) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x, kv = blockIdx.y, hkv = ring.hkv;
  const int s = seqs[i];
  if (s < 0 || s >= ring.num_seqs) {
    if (kv == 0 && threadIdx.x == 0) flag(status, ST_BAD_SEQ);
    return;
  }
  uint4 *rk = reinterpret_cast<uint4 *>(ring.k + ((long long)s * hkv + kv) * WIN * DQK);
  uint4 *rv = reinterpret_cast<uint4 *>(ring.v + ((long long)s * hkv + kv) * WIN * DV);
  uint4 *sk = reinterpret_cast<uint4 *>(k_snap + ((long long)i * hkv + kv) * WIN * DQK);
  uint4 *sv = reinterpret_cast<uint4 *>(v_snap + ((long long)i * hkv + kv) * WIN * DV);
  constexpr int NK = WIN * DQK / 8, NV = WIN * DV / 8;
  static_assert(NK % (COPY_THREADS * COPY_BATCH) == 0 && NV % (COPY_THREADS * COPY_BATCH) == 0, "whole batches");
  if (to_ring) {
    copy_chunks(rk, sk, NK);
    copy_chunks(rv, sv, NV);
  } else {
    copy_chunks(sk, rk, NK);
    copy_chunks(sv, rv, NV);
  }
  if (kv == 0 && threadIdx.x < WIN) {
    int32_t *rt = ring.slot_pos + (long long)s * WIN;
    int32_t *st = tags_snap + (long long)i * WIN;
    if (to_ring)
      rt[threadIdx.x] = st[threadIdx.x];
    else
      st[threadIdx.x] = rt[threadIdx.x];
  }
}

}  // namespace

cudaError_t launch_ring_copy(const KvView &ring, const int32_t *seqs, int n, uint16_t *k_snap, uint16_t *v_snap,
                             int32_t *tags_snap, bool to_ring, unsigned *status, cudaStream_t st) {
  dim3 grid((unsigned)n, (unsigned)ring.hkv);
  return launch_pdl(ring_copy_kernel, grid, dim3(COPY_THREADS), 0, st, ring, seqs, k_snap, v_snap, tags_snap,
                    to_ring ? 1 : 0, status);
}

}  // namespace kvr
