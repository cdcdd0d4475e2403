// ring_snapshot.cu -- copy the windowed layers' rings of chosen sequences to
// and from snapshot buffers (colibri "MiMo-V2.6 (Xiaomi)", "System One mode
// and prompt reuse": the rings are copied into a snapshot and back).  A KV
// head's ring rows are contiguous on both sides (48 KB of K, 32 KB of V), so
// they move as 16 KB pieces, one CTA each: one bulk copy into shared memory,
// one bulk store out.  The CTA of KV head 0's first piece also moves the 128
// slot tags.
#include "launch.h"
#include "tc_ptx.cuh"

namespace kvr {
namespace {

constexpr int COPY_THREADS = 32;
constexpr int COPY_PIECE = 16384;                         // bytes per CTA
constexpr int COPY_KPIECES = WIN * DQK * 2 / COPY_PIECE;  // K pieces of a head's rows
constexpr int COPY_VPIECES = WIN * DV * 2 / COPY_PIECE;   // V pieces
static_assert(COPY_KPIECES * COPY_PIECE == WIN * DQK * 2 && COPY_VPIECES * COPY_PIECE == WIN * DV * 2,
              "whole pieces");
constexpr unsigned COPY_ST_TIMEOUT = 8u;                  // KVR_DEV_TIMEOUT

__global__ void __launch_bounds__(COPY_THREADS)
    ring_copy_kernel(KvView ring, const int32_t *__restrict__ seqs, uint16_t *k_snap, uint16_t *v_snap,
                     int32_t *tags_snap, int to_ring, unsigned *status, unsigned long long stall_ns) {
  __shared__ __align__(128) uint8_t buf[COPY_PIECE];
  __shared__ __align__(8) uint64_t s_bar, s_stall;
  __shared__ uint32_t s_abort;
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x, kv = blockIdx.y, piece = blockIdx.z, hkv = ring.hkv, lane = threadIdx.x;
  const int s = seqs[i];
  if (s < 0 || s >= ring.num_seqs) {
    if (kv == 0 && piece == 0 && lane == 0) flag(status, ST_BAD_SEQ);
    return;
  }
  const bool isv = piece >= COPY_KPIECES;
  const long long off = (long long)(isv ? piece - COPY_KPIECES : piece) * COPY_PIECE;  // bytes into the head's rows
  uint8_t *ringp = isv ? reinterpret_cast<uint8_t *>(ring.v + ((long long)s * hkv + kv) * WIN * DV)
                       : reinterpret_cast<uint8_t *>(ring.k + ((long long)s * hkv + kv) * WIN * DQK);
  uint8_t *snapp = isv ? reinterpret_cast<uint8_t *>(v_snap + ((long long)i * hkv + kv) * WIN * DV)
                       : reinterpret_cast<uint8_t *>(k_snap + ((long long)i * hkv + kv) * WIN * DQK);
  const uint8_t *src = (to_ring ? snapp : ringp) + off;
  uint8_t *dst = (to_ring ? ringp : snapp) + off;
  if (lane == 0) {
    const uint32_t bar = smem_u32(&s_bar), stall_bar = smem_u32(&s_stall), sb = smem_u32(buf);
    tc::mbar_init(bar, 1);
    tc::mbar_init(stall_bar, 1);
    s_abort = 0;
    tc::fence_mbar_init();
    tc::mbar_expect_tx(bar, COPY_PIECE);
    tc::bulk_load(sb, src, COPY_PIECE, bar);
    // a copy that does not land within 2 s: flagged, nothing stored, and
    // still waited for (bounded) before the CTA leaves.  Test hook
    // (stall_ns != 0): the first CTA waits instead on a barrier nothing
    // completes, with that limit, and takes the same exit.
    const bool stall = stall_ns && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0;
    if (stall ? tc::mbar_wait(stall_bar, 0, &s_abort, stall_ns) : tc::mbar_wait(bar, 0, &s_abort)) {
      tc::fence_proxy_async_smem();
      tc::bulk_store(dst, sb, COPY_PIECE);
      tc::bulk_commit();
      tc::bulk_wait_read_all();  // the piece is read before the CTA leaves (the grid's end covers the writes)
    } else {
      flag(status, COPY_ST_TIMEOUT);
      uint32_t never = 0;
      tc::mbar_wait(bar, 0, &never);
    }
  }
  if (kv == 0 && piece == 0) {
    int32_t *rt = ring.slot_pos + (long long)s * WIN;
    int32_t *st = tags_snap + (long long)i * WIN;
    for (int c = lane; c < WIN; c += COPY_THREADS) {
      if (to_ring)
        rt[c] = st[c];
      else
        st[c] = rt[c];
    }
  }
}

}  // namespace

cudaError_t launch_ring_copy(const KvView &ring, const int32_t *seqs, int n, uint16_t *k_snap, uint16_t *v_snap,
                             int32_t *tags_snap, bool to_ring, unsigned *status, cudaStream_t st) {
  dim3 grid((unsigned)n, (unsigned)ring.hkv, COPY_KPIECES + COPY_VPIECES);
  return launch_pdl(ring_copy_kernel, grid, dim3(COPY_THREADS), 0, st, ring, seqs, k_snap, v_snap, tags_snap,
                    to_ring ? 1 : 0, status, take_stall());
}

}  // namespace kvr
