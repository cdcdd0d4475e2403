// ring_snapshot.cu -- copy the windowed layers' rings of chosen sequences to
// and from snapshot buffers (colibri "MiMo-V2.6 (Xiaomi)", "System One mode
// and prompt reuse": the rings are copied into a snapshot and back).  One CTA
// per (entry, KV head) moves that head's 48 KB of K and 32 KB of V with
// 16-byte accesses; the KV-head-0 CTA also moves the 128 slot tags.
#include "launch.h"

namespace kvr {
namespace {

__global__ void __launch_bounds__(256)
    ring_copy_kernel(KvView ring, const int32_t *__restrict__ seqs, uint16_t *k_snap, uint16_t *v_snap,
                     int32_t *tags_snap, int to_ring, unsigned *status) {
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
  if (to_ring) {
    for (int e = threadIdx.x; e < NK; e += blockDim.x) rk[e] = sk[e];
    for (int e = threadIdx.x; e < NV; e += blockDim.x) rv[e] = sv[e];
  } else {
    for (int e = threadIdx.x; e < NK; e += blockDim.x) sk[e] = rk[e];
    for (int e = threadIdx.x; e < NV; e += blockDim.x) sv[e] = rv[e];
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
  ring_copy_kernel<<<grid, 256, 0, st>>>(ring, seqs, k_snap, v_snap, tags_snap, to_ring ? 1 : 0, status);
  return cudaGetLastError();
}

}  // namespace kvr
