// pages.cu -- pool management of a windowed layer kept in pages.
//
// release: Xiaomi "Full-Pipeline Inference Optimization for MiMo-V2.5
// Series", section 2.1 ("SWA KVCache Management": the SWA pool is bounded by
// the window; "SWA-Aware Prefix Cache Tree": the end of a prefill chunk, the
// end of a request and every N decoded tokens release the SWA KV that has
// left the window) and gaudi-cookbook "Windowed KV groups" (the sliding
// layers' out-of-window blocks are freed).  A query at q reads q-W+1..q, so
// with the next query of a sequence at P, the blocks whose positions all lie
// below P-W+1 are read by no later query.
//
// gather: colibri "System One mode and prompt reuse": position p sits in ring
// slot p mod 128 and the ring records which position each slot holds; the
// ring of a sequence whose positions 0..E-1 were appended in order holds, in
// slot c, the last of them congruent to c.
#include "launch.h"
#include "tc_ptx.cuh"

namespace kvr {
namespace {

constexpr int RL_THREADS = 1024;
constexpr int RL_WARPS = RL_THREADS / 32;
constexpr unsigned FULLW = 0xffffffffu;

struct ReleaseArgs {
  int32_t *table;
  int num_seqs, max_blocks, block_size, num_blocks;
  const int32_t *seqs;
  const int64_t *next_pos;
  int32_t *lo;  // [num_seqs] or null
  int n, window;
  int32_t *free_ids;
  int32_t *free_count;
  int free_cap;
};

// Table range [a, b) that entry i looks at; false for a bad sequence id.
__device__ __forceinline__ bool release_range(const ReleaseArgs &A, int i, int &s, int &a, int &b) {
  s = A.seqs[i];
  if (s < 0 || s >= A.num_seqs) return false;
  const long long first_kept = A.next_pos[i] - A.window + 1;  // earliest position a later query reads
  long long hi = first_kept > 0 ? first_kept / A.block_size : 0;
  if (hi > A.max_blocks) hi = A.max_blocks;
  int lo = A.lo ? A.lo[s] : 0;
  if (lo < 0) lo = 0;
  if (lo > A.max_blocks) lo = A.max_blocks;
  a = lo;
  b = (int)hi;
  return true;
}

// Live (releasable) entries of one range, counted by a warp.
__device__ __forceinline__ int warp_count_live(const ReleaseArgs &A, const int32_t *row, int a, int b, int lane,
                                               bool &bad) {
  int cnt = 0;
  for (int c0 = a; c0 < b; c0 += 32) {
    const int bi = c0 + lane;
    const int id = bi < b ? row[bi] : -1;
    if (id >= A.num_blocks) bad = true;
    cnt += __popc(__ballot_sync(FULLW, id >= 0 && id < A.num_blocks));
  }
  return cnt;
}

// One CTA: pass 1 counts what the whole call releases (all or nothing
// against the free list's capacity); pass 2 walks the entries in rounds of
// 32 (one per warp), takes each entry's offset from a scan of the round's
// counts, and writes the ids in (entry, block index) order.
__global__ void __launch_bounds__(RL_THREADS) pages_release_kernel(ReleaseArgs A, unsigned *status) {
  __shared__ int s_cnt[RL_WARPS];
  __shared__ int s_off[RL_WARPS];
  __shared__ int s_total, s_base;
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  // pass 1
  int mine = 0;
  bool bad_seq = false, bad_blk = false;
  for (int i = warp; i < A.n; i += RL_WARPS) {
    int s, a, b;
    if (!release_range(A, i, s, a, b)) {
      bad_seq = true;
      continue;
    }
    mine += warp_count_live(A, A.table + (long long)s * A.max_blocks, a, b, lane, bad_blk);
  }
  if (lane == 0) s_cnt[warp] = mine;
  if (threadIdx.x == 0) s_base = *A.free_count;
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = 0;
    for (int w = 0; w < RL_WARPS; ++w) t += s_cnt[w];
    s_total = t;
  }
  if (bad_seq && lane == 0) flag(status, ST_BAD_SEQ);
  if (__any_sync(FULLW, bad_blk) && lane == 0) flag(status, ST_BAD_BLOCK);
  __syncthreads();
  const int base0 = s_base, total = s_total;
  if (base0 < 0 || (long long)base0 + total > A.free_cap) {
    if (threadIdx.x == 0) flag(status, ST_FREE_FULL);
    return;  // nothing released, nothing changed
  }

  // pass 2
  int base = base0;
  for (int r0 = 0; r0 < A.n; r0 += RL_WARPS) {
    const int i = r0 + warp;
    int s = -1, a = 0, b = 0;
    const bool ok = i < A.n && release_range(A, i, s, a, b);
    bool dummy = false;
    const int cnt = ok ? warp_count_live(A, A.table + (long long)s * A.max_blocks, a, b, lane, dummy) : 0;
    if (lane == 0) s_cnt[warp] = cnt;
    __syncthreads();
    if (threadIdx.x == 0) {
      int t = 0;
      for (int w = 0; w < RL_WARPS; ++w) {
        s_off[w] = t;
        t += s_cnt[w];
      }
      s_total = t;
    }
    __syncthreads();
    if (ok) {
      int32_t *row = A.table + (long long)s * A.max_blocks;
      int at = base + s_off[warp];
      for (int c0 = a; c0 < b; c0 += 32) {
        const int bi = c0 + lane;
        const int id = bi < b ? row[bi] : -1;
        const bool live = id >= 0 && id < A.num_blocks;
        const unsigned m = __ballot_sync(FULLW, live);
        if (live) {
          A.free_ids[at + __popc(m & ((1u << lane) - 1u))] = id;
          row[bi] = -1;
        }
        at += __popc(m);
      }
      if (A.lo && lane == 0 && A.lo[s] < b) A.lo[s] = b;
    }
    base += s_total;
    __syncthreads();  // s_cnt / s_off / s_total are rewritten by the next round
  }
  if (threadIdx.x == 0) *A.free_count = base;
}

// One CTA per (entry, KV head, K or V), one thread per ring slot.  Slot c is
// resolved to its source row (-1 when the slot gets no position); the slots
// form runs whose source rows are consecutive in the pool (positions of one
// block in slot order, or of neighbouring blocks where their rows adjoin),
// at most (128 / block size) + 2 of them.  The thread at the head of a run
// copies it with one bulk copy into the CTA's image of the ring's K (or V),
// then, once every run has landed, back out to the ring with one bulk store:
// each byte crosses the SM once, in copies of a block's rows or more.  Slots
// without a position keep what the ring held.  The CTA of KV head 0's K also
// writes the slot tags.
constexpr int GATHER_THREADS = WIN;
constexpr int GATHER_SMEM = WIN * DQK * 2;  // the image of one ring's K (or V: the first 32 KB)
constexpr unsigned GATHER_ST_TIMEOUT = 8u;           // KVR_DEV_TIMEOUT

__global__ void __launch_bounds__(GATHER_THREADS, 4)
    ring_gather_kernel(KvView pages, KvView ring, const int32_t *__restrict__ src_seqs,
                       const int32_t *__restrict__ dst_seqs, const int64_t *__restrict__ end, unsigned *status,
                       unsigned long long stall_ns) {
  extern __shared__ __align__(128) uint8_t g_img[];
  __shared__ long long s_row[WIN];
  __shared__ unsigned s_brk[WIN / 32];
  __shared__ __align__(8) uint64_t s_bar, s_stall;
  __shared__ uint32_t s_abort;
  const int i = blockIdx.x, kv = blockIdx.y, hkv = ring.hkv, c = threadIdx.x;
  const bool isv = blockIdx.z != 0;
  const int width = isv ? DV : DQK;                             // elements per row
  const uint16_t *src = isv ? pages.v : pages.k;
  uint16_t *dstr = isv ? ring.v : ring.k;
  const uint32_t bar = smem_u32(&s_bar), stall_bar = smem_u32(&s_stall);
  // Before the wait for the kernel ahead (which may still run): the window's
  // rows requested into L2, block by block (thread j: the window's j-th
  // block), from the end, source sequence and block ids read early (see
  // ld_early_s32: a stale value only wastes a prefetch; all is read again
  // below).  Anything outside the pool is skipped.
  if (c < 32) {
    const long long e = ld_early_s64(end + i);
    const int ss = ld_early_s32(src_seqs + i), bsz = pages.block_size;
    if (e > 0 && ss >= 0 && ss < pages.num_seqs) {
      const long long lo = e > WIN ? e - WIN : 0, b0 = lo / bsz, bj = b0 + c;
      if (bj <= (e - 1) / bsz && bj < pages.max_blocks) {
        const int blk = ld_early_s32(pages.block_table + (long long)ss * pages.max_blocks + bj);
        if (blk >= 0 && blk < pages.num_blocks) {
          const long long r0 = max(lo, bj * bsz), r1 = min(e - 1, bj * bsz + bsz - 1);
          const long long row = ((long long)blk * pages.hkv + kv) * bsz + (r0 - bj * bsz);
          prefetch_l2(src + row * width, (uint32_t)(r1 - r0 + 1) * width * 2);
        }
      }
    }
  }
  if (c == 0) {
    tc::mbar_init(bar, 1);
    tc::mbar_init(stall_bar, 1);
    s_abort = 0;
    tc::fence_mbar_init();
  }
  pdl_wait();
  pdl_trigger();
  const int ss = src_seqs[i], ds = dst_seqs[i];
  if (ss < 0 || ss >= pages.num_seqs || ds < 0 || ds >= ring.num_seqs) {
    if (kv == 0 && !isv && c == 0) flag(status, ST_BAD_SEQ);
    return;
  }
  {
    const long long e = end[i];
    // the position slot c holds: the largest p < e with p mod 128 == c
    const long long p = e - 1 - (long long)(((e - 1 - c) % WIN + WIN) % WIN);
    long long row = -1;
    int32_t tag = -1;
    if (e > 0 && p >= 0) {
      const long long bi = p / pages.block_size;
      const int blk = bi < pages.max_blocks ? pages.block_table[(long long)ss * pages.max_blocks + bi] : -1;
      if (blk >= 0 && blk < pages.num_blocks) {
        row = ((long long)blk * pages.hkv + kv) * pages.block_size + (p - bi * pages.block_size);
        tag = (int32_t)p;
      } else if (kv == 0 && !isv) {
        flag(status, ST_BAD_BLOCK);
      }
    }
    s_row[c] = row;
    if (kv == 0 && !isv) ring.slot_pos[(long long)ds * WIN + c] = tag;
  }
  __syncthreads();  // (also: the barrier's initialisation before any use)
  // Slot c continues a run when its row follows slot c-1's; every other slot
  // (a head, or one without a position) ends the run before it.
  const long long row = s_row[c];
  const bool cont = row >= 0 && c > 0 && s_row[c - 1] == row - 1;
  const unsigned brk = __ballot_sync(FULLW, !cont);
  if ((c & 31) == 0) s_brk[c >> 5] = brk;
  const int nslots = __syncthreads_count(row >= 0);
  if (nslots == 0) return;
  int len = 0;  // slots in the run this thread heads (0: none): up to the next break
  if (row >= 0 && !cont) {
    len = WIN - c;
    for (int k = c + 1, w = k >> 5; w < WIN / 32; ++w) {
      const unsigned m = w == (k >> 5) ? s_brk[w] & (FULLW << (k & 31)) : s_brk[w];
      if (m) {
        len = 32 * w + __ffs((int)m) - 1 - c;
        break;
      }
    }
  }
  if (c == 0) tc::mbar_expect_tx(bar, (uint32_t)nslots * width * 2);
  __syncthreads();  // the expected bytes are set before any copy can complete
  const uint32_t img = smem_u32(g_img);
  if (len) tc::bulk_load(img + c * width * 2, src + row * width, (uint32_t)len * width * 2, bar);
  // A wait that gives up (2 s) flags the call and still lets the copies
  // land (bounded again) before the CTA leaves; nothing is stored then.
  // Test hook (stall_ns != 0): the first CTA waits instead on a barrier
  // nothing completes, with that limit, and takes the same exit.
  const bool stall = stall_ns && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0;
  if (!(stall ? tc::mbar_wait(stall_bar, 0, &s_abort, stall_ns) : tc::mbar_wait(bar, 0, &s_abort))) {
    if (c == 0) flag(status, GATHER_ST_TIMEOUT);
    uint32_t never = 0;
    tc::mbar_wait(bar, 0, &never);
    return;
  }
  if (len) {
    tc::fence_proxy_async_smem();
    tc::bulk_store(dstr + (((long long)ds * hkv + kv) * WIN + c) * width, img + c * width * 2, (uint32_t)len * width * 2);
    tc::bulk_commit();
    tc::bulk_wait_read_all();  // the image is read before the CTA leaves (the grid's end covers the writes)
  }
}

}  // namespace

cudaError_t launch_pages_release(int32_t *table, int num_seqs, int max_blocks, int block_size, int num_blocks,
                                 const int32_t *seqs, const int64_t *next_pos, int32_t *lo, int n, int window,
                                 int32_t *free_ids, int32_t *free_count, int free_cap, unsigned *status,
                                 cudaStream_t st) {
  ReleaseArgs A{table, num_seqs, max_blocks, block_size, num_blocks, seqs, next_pos, lo, n, window,
                free_ids, free_count, free_cap};
  return launch_pdl(pages_release_kernel, dim3(1), dim3(RL_THREADS), 0, st, A, status);
}

cudaError_t launch_ring_gather(const KvView &pages, const KvView &ring, const int32_t *src_seqs,
                               const int32_t *dst_seqs, const int64_t *end, int n, unsigned *status,
                               cudaStream_t st) {
  cudaError_t e = ensure_smem_limit(15, (const void *)ring_gather_kernel, GATHER_SMEM, true);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)n, (unsigned)ring.hkv, 2);
  return launch_pdl(ring_gather_kernel, grid, dim3(GATHER_THREADS), GATHER_SMEM, st, pages, ring, src_seqs, dst_seqs,
                    end, status, take_stall());
}

}  // namespace kvr
