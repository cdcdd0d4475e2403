/*
 * kvring.h -- C ABI of the hybrid-SWA attention hot path (sm_103a).
 *
 * MiMo-V2-style hybrid attention: most layers attend over a sliding window
 * of W = 128 positions with a learned per-head sink logit, kept in a ring of
 * 128 slots; a few layers attend over the whole context, kept in a paged pool.
 * Heads are GQA with 192-wide q/k and 128-wide v; RoPE is rotate-half on the
 * first 64 dims (theta 1e4 on windowed layers, 1e7 on full layers); v is
 * multiplied by the value scale when it is written.  Sources: colibri
 * "MiMo-V2.6", sections "What the engine implements" and "System One mode and
 * prompt reuse"; gaudi-cookbook "MiMo-V2.6-Flash on Gaudi 2", sections "What
 * was built" and "The RoPE fix for large positions"; Xiaomi "Full-Pipeline
 * Inference Optimization for MiMo-V2.5 Series", section 2.1 (dual KV pools).
 *
 * Conventions for every call:
 *  - bf16 tensors are IEEE bfloat16 bit patterns (kvr_bf16), row-major,
 *    densely packed.  All tensor pointers are DEVICE pointers unless the
 *    argument says "host".  The caller owns every buffer, including
 *    workspaces; the library allocates and frees nothing on the device.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  Buffers must stay valid until the stream has run the
 *    work.  Calls on one stream execute in order.  The decode-path kernels
 *    are launched with programmatic stream serialisation: one may be
 *    scheduled while the kernel before it on the stream is still running,
 *    but touches no global memory until that kernel has completed and its
 *    writes are visible, so stream order holds as for a plain launch.
 *  - Arguments are validated on the host before anything is launched; a bad
 *    argument returns a negative kvr_status and launches nothing.  A launch
 *    failure returns KVR_ECUDA.  kvr_last_error() gives a message (thread
 *    local).  The library never aborts or traps.
 *  - Values only the device can see (positions, sequence ids, block-table
 *    entries, ring tags) are checked by the kernels: an access that would
 *    leave its buffer is skipped, the affected output row is written as
 *    zeros, and a bit is set in the device status word (kvr_device_status).
 *  - Positions are 0-based absolute token positions.  Head h of a layer with
 *    Hq query heads and Hkv KV heads reads KV head h / (Hq / Hkv).
 *
 * Head geometry is fixed: Dqk = 192, Dv = 128, rotary dims = 64, W = 128.
 */
#ifndef KVRING_H
#define KVRING_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t kvr_bf16;
typedef int kvr_status;

enum {
  KVR_OK = 0,
  KVR_EINVAL = -1,       /* null pointer, bad size, Hq not a multiple of Hkv, wrong layout kind */
  KVR_ERANGE = -2,       /* a host-known position or length past the RoPE table or the pool */
  KVR_EWORKSPACE = -3,   /* workspace missing or smaller than the size query returned */
  KVR_EUNSUPPORTED = -4, /* a shape the library does not handle (e.g. Hq/Hkv > 16) */
  KVR_ECUDA = -5         /* a CUDA runtime call or launch failed */
};

#define KVR_DQK 192
#define KVR_DV 128
#define KVR_DROT 64
#define KVR_WINDOW 128

/* Device status bits (kvr_device_status). */
#define KVR_DEV_BAD_POS 1u    /* a position < 0 or >= the RoPE table length */
#define KVR_DEV_BAD_SEQ 2u    /* a sequence id outside the layout */
#define KVR_DEV_BAD_BLOCK 4u  /* a block-table entry outside the pool, or a context past the table */
#define KVR_DEV_TIMEOUT 8u    /* a kernel gave up waiting on its own pipeline (bounded wait) and returned */
#define KVR_DEV_BAD_ROWS 16u  /* varlen: cu_rows not non-decreasing within [0, T]; that chunk is skipped */
#define KVR_DEV_FREE_FULL 32u /* kv_pages_release_window: the free list could not take the released ids */

/* KV storage kinds. */
enum {
  KVR_LAYOUT_RING = 1,   /* SWA pool: one ring of 128 slots per (sequence, KV head) */
  KVR_LAYOUT_PAGED = 2,  /* Full pool (or a windowed layer kept in pages): pages of block_size positions */
  KVR_LAYOUT_LINEAR = 3  /* staging: rows in call order (a prefill chunk) */
};

/*
 * Where one layer's K/V live.
 *
 * RING   (colibri "System One mode and prompt reuse": position p sits in slot
 *        p mod 128, and the ring records the position each slot holds):
 *        k [num_seqs][Hkv][128][192], v [num_seqs][Hkv][128][128],
 *        slot_pos [num_seqs][128] int32, -1 = empty.  slot_pos is shared by
 *        the KV heads of a sequence and is written by kv_ring_append_rope.
 *        k, v and slot_pos must be 16-byte aligned.
 * PAGED  (the Full KV pool of Xiaomi section 2.1, grown on demand; a
 *        windowed layer may be kept this way too, its out-of-window pages
 *        released by kv_pages_release_window):
 *        k [num_blocks][Hkv][block_size][192], v [num_blocks][Hkv][block_size][128],
 *        block_table [num_seqs][max_blocks] int32: position p of sequence s is
 *        row p % block_size of block block_table[s][p / block_size].
 *        block_size is a multiple of 16 in [16, 1024].
 * LINEAR k [num_rows][Hkv][192], v [num_rows][Hkv][128]; row r of a call is
 *        the r-th token of that call.
 *
 * Fields a kind does not use are ignored.  The struct itself is host memory
 * read during the call only.
 */
typedef struct kvr_kv_layout {
  int32_t kind;
  int32_t num_kv_heads;
  kvr_bf16 *k;
  kvr_bf16 *v;
  int32_t *slot_pos;           /* RING */
  const int32_t *block_table;  /* PAGED */
  int32_t num_seqs;            /* RING, PAGED */
  int32_t max_blocks;          /* PAGED */
  int32_t block_size;          /* PAGED */
  int32_t num_blocks;          /* PAGED */
  int64_t num_rows;            /* LINEAR */
} kvr_kv_layout;

/*
 * Every call that launches work looks up, on its first use on a device (and
 * again after cudaDeviceReset), the device address of the library's status
 * word; that first call must not run while its stream is being captured
 * into a CUDA graph: it then returns KVR_EINVAL and launches nothing.
 */

/* Message for the last failing call on this thread ("" if none). */
const char *kvr_last_error(void);

/*
 * Read the device status word of the current device into *flags (host) and,
 * if reset != 0, clear it.  Synchronises the device.  Returns KVR_OK or
 * KVR_ECUDA.
 */
kvr_status kvr_device_status(uint32_t *flags, int reset);

/*
 * Test hook for the bounded waits (no counterpart on the pages).  The next
 * `launches` kernels started by swa_sink_decode (over a RING layout, or over
 * a PAGED one with up to 8 q heads per KV head), by the short-chunk part of
 * swa_sink_prefill_varlen, by full_attn_prefill_chunk, by
 * kv_ring_gather_pages or by kv_ring_snapshot / kv_ring_restore, in this
 * process, stall on purpose: once their loads are in flight (and, for the
 * prefill, with its tensor memory held), one warp group (for the copies: the
 * first CTA) waits on an internal barrier that nothing completes, with a
 * time limit of limit_ns nanoseconds.  When the limit passes the kernel takes
 * the exit a real stall would take -- the other warps see the abort, the
 * loads and products already issued finish, tensor memory is freed, a copy
 * stores nothing -- and sets KVR_DEV_TIMEOUT; that call's output is
 * unspecified.  launches = 0
 * turns the hook off.  KVR_EINVAL unless 0 <= launches and
 * 1000 <= limit_ns <= 1e9.  For tests of that exit path only.
 */
kvr_status kvr_debug_stall_next(int32_t launches, int64_t limit_ns);

/*
 * RoPE cos/sin table, computed on the host in fp64 and stored as fp32
 * (gaudi-cookbook "The RoPE fix for large positions": a table built with
 * fp32 cos/sin goes wrong past about 1.5e5 radians, so it is built on the CPU
 * in float64).
 *   host_out [max_pos][32][2] fp32 host memory: host_out[p][i] =
 *   (cos, sin)(p * theta^(-2i/64)).  Copy it to the device once per theta.
 * nthreads <= 0 uses the hardware concurrency.  KVR_EINVAL on a null
 * pointer, max_pos <= 0 or theta <= 1.
 */
kvr_status kvr_rope_table_build(double theta, int64_t max_pos, float *host_out, int nthreads);

/*
 * Fused KV write (colibri "What the engine implements": partial rotate-half
 * RoPE on the first 64 dims; values multiplied by attention_value_scale).
 * For each token t and KV head h:
 *   k'[0:32]  = k[0:32]*c - k[32:64]*s,  k'[32:64] = k[32:64]*c + k[0:32]*s
 *   (c, s) = rope_cos_sin[pos[t]][i]; k'[64:192] = k[64:192] (bit copy);
 *   v' = v * value_scale;  fp32 arithmetic, one round-to-nearest-even to bf16.
 * and writes them to `dst`:
 *   RING   slot pos[t] % 128 of sequence seq[t], and slot_pos[seq][slot] = pos[t];
 *   PAGED  row pos[t] % block_size of block block_table[seq[t]][pos[t]/block_size];
 *   LINEAR row t (seq may be NULL; dst->num_rows >= T).
 * k [T][Hkv][192], v [T][Hkv][128] bf16; pos [T] int64; seq [T] int32.
 * rope_cos_sin [max_pos][32][2] fp32 (kvr_rope_table_build).  Hkv must equal
 * dst->num_kv_heads.  For RING, two tokens of one call must not map to the
 * same (sequence, slot); which one lands is then unspecified.  T = 0 is a
 * no-op.
 */
kvr_status kv_ring_append_rope(const kvr_bf16 *k, const kvr_bf16 *v, const int64_t *pos,
                               const int32_t *seq, int32_t T, int32_t Hkv,
                               const float *rope_cos_sin, int64_t max_pos, float value_scale,
                               const kvr_kv_layout *dst, void *stream);

/*
 * Decode over a windowed layer (colibri "What the engine implements": the
 * sink joins the softmax denominator and nothing else; gaudi-cookbook "What
 * was built": the window is exactly the last 128 positions).  For sequence
 * b at position p = pos[b] (whose K/V were already appended) and q head h:
 *   s_j = (rope(q)[h] . k'_j) * softmax_scale over ring slots j with
 *         p - 128 < slot_pos[seq[b]][j] <= p,
 *   out[b][h] = sum_j e^{s_j - m} v'_j / (e^{sinks[h] - m} + sum_j e^{s_j - m}).
 * q [B][Hq][192] bf16 un-rotated (rotated here with rope_cos_sin row p and
 * rounded to bf16); ring: a RING layout; sinks [Hq] fp32 (raw logits, not
 * multiplied by softmax_scale); out [B][Hq][128] bf16.  Hq/Hkv <= 16.
 * The sink is counted once, in the final normalisation.
 *
 * `ring` may also be a PAGED layout holding the windowed layer in pages
 * (gaudi-cookbook "Windowed KV groups": vLLM's paged sliding-window groups):
 * the keys are positions max(0, p-127)..p of sequence seq[b], read through
 * its block table; no entry for a position below p-127 rounded down to a
 * multiple of 16 is read, so pages released by kv_pages_release_window with
 * next_pos <= p are never touched.  p must be < max_blocks*block_size (else
 * the row is zeroed and KVR_DEV_BAD_POS set).
 */
kvr_status swa_sink_decode(const kvr_bf16 *q, const int64_t *pos, const int32_t *seq, int32_t B,
                           int32_t Hq, const kvr_kv_layout *ring, const float *sinks,
                           const float *rope_cos_sin, int64_t max_pos, float softmax_scale,
                           kvr_bf16 *out, void *stream);

/*
 * Workspace bytes full_attn_decode needs for B sequences whose contexts
 * (pos + 1) are at most max_ctx.  Returns 0 on bad arguments.
 */
size_t full_attn_decode_workspace_size(int32_t B, int32_t Hq, int32_t Hkv, int64_t max_ctx);

/*
 * Decode over a full-attention layer: causal attention of the token at
 * p = pos[b] over positions 0..p of the paged pool, no sink.  Split-K
 * (flash-decode): the context is cut into splits that run in parallel and
 * write (max, denominator, numerator) partials to the workspace; a second
 * kernel merges them by log-sum-exp (Xiaomi section 1.2: decode is
 * memory-bound, its time set by the KV bytes read).
 * q [B][Hq][192] bf16 un-rotated; pool: a PAGED layout; out [B][Hq][128] bf16.
 * Every pos[b] + 1 must be <= max_ctx (else the row is zeroed and
 * KVR_DEV_BAD_POS set); max_ctx <= max_pos and <= max_blocks*block_size.
 * workspace: device memory of at least
 * full_attn_decode_workspace_size(B, Hq, Hkv, max_ctx) bytes, 256-byte
 * aligned, used as scratch; its contents need no initialisation.
 */
kvr_status full_attn_decode(const kvr_bf16 *q, const int64_t *pos, const int32_t *seq, int32_t B,
                            int32_t Hq, const kvr_kv_layout *pool, const float *rope_cos_sin,
                            int64_t max_pos, float softmax_scale, int64_t max_ctx,
                            void *workspace, size_t workspace_bytes, kvr_bf16 *out, void *stream);

/*
 * Ring snapshot and restore (colibri "MiMo-V2.6 (Xiaomi)", "System One mode
 * and prompt reuse": a snapshot of a prompt holds the windowed layers' rings,
 * copied out and later copied back, because the next prompt overwrites the
 * slots of the snapshot's last positions; the full layers' rows stay in place).
 *   seqs [n] int32 (device): the ring rows to copy (sequence ids of `ring`);
 *   k_snap [n][Hkv][128][192], v_snap [n][Hkv][128][128] bf16 and
 *   tags_snap [n][128] int32: the snapshot buffers (device), entry i for
 *   seqs[i].
 * kv_ring_snapshot copies ring -> snapshot; kv_ring_restore copies
 * snapshot -> ring (slot contents and slot tags, bit for bit).  A sequence
 * id outside the ring sets KVR_DEV_BAD_SEQ and its entry is skipped.  The
 * rows move as bulk copies through shared memory; a piece that does not land
 * within 2 s sets KVR_DEV_TIMEOUT and is not stored.  k_snap and v_snap must
 * be 16-byte aligned (KVR_EINVAL otherwise).  Two entries of one restore must
 * not name the same sequence.  n = 0 is a no-op.
 */
kvr_status kv_ring_snapshot(const kvr_kv_layout *ring, const int32_t *seqs, int32_t n, kvr_bf16 *k_snap,
                            kvr_bf16 *v_snap, int32_t *tags_snap, void *stream);
kvr_status kv_ring_restore(const kvr_kv_layout *ring, const int32_t *seqs, int32_t n, const kvr_bf16 *k_snap,
                           const kvr_bf16 *v_snap, const int32_t *tags_snap, void *stream);

/*
 * Out-of-window release of a windowed layer kept in pages (Xiaomi
 * "Full-Pipeline Inference Optimization", section 2.1: the SWA pool is kept
 * at window size -- the end of each prefill chunk, the end of a request and
 * every N decoded tokens release the SWA KV that has left the window;
 * gaudi-cookbook "Windowed KV groups": the out-of-window blocks are freed).
 * A query at q reads positions q-window+1..q, so once the next query of a
 * sequence is at P, table entries bi with (bi+1)*block_size <= P-window+1
 * hold only positions no later query reads.
 *   block_table [num_seqs][max_blocks] int32 (device, read and written);
 *   seqs [n] int32, next_pos [n] int64 (device): entry i names sequence
 *     seqs[i] and the position of its next query; no two entries of one call
 *     may name the same sequence; next_pos must not decrease from one call
 *     to the next for a sequence (release with the committed position, not
 *     one a rejected draft could roll back);
 *   lo [num_seqs] int32 (device, read and written) or NULL: entries below
 *     lo[s] were handled by earlier calls and are not looked at again; the
 *     call sets lo[s] = max(lo[s], bound) (keep it 0 for a new sequence);
 *   free_ids [free_cap] int32, free_count [1] int32 (device): the free list.
 * Every entry in [max(lo[s], 0), bound) holding a block id in
 * [0, num_blocks) is released: the id is written at free_ids[*free_count +
 * k] and the entry set to -1; *free_count grows by the number released.
 * Ids are appended in the order (call entry i, block index).  Entries
 * holding -1 are skipped; ids >= num_blocks are left in place and set
 * KVR_DEV_BAD_BLOCK; a sequence id outside [0, num_seqs) sets
 * KVR_DEV_BAD_SEQ.  If the ids the whole call would release do not fit in
 * free_cap, the call changes nothing and sets KVR_DEV_FREE_FULL.  One CTA;
 * the work per call is the entries between lo and the bound.  n = 0 is a
 * no-op.
 */
kvr_status kv_pages_release_window(int32_t *block_table, int32_t num_seqs, int32_t max_blocks,
                                   int32_t block_size, int32_t num_blocks, const int32_t *seqs,
                                   const int64_t *next_pos, int32_t *lo, int32_t n, int32_t window,
                                   int32_t *free_ids, int32_t *free_count, int32_t free_cap, void *stream);

/*
 * Ring from pages (colibri "System One mode and prompt reuse": position p
 * lives in ring slot p mod 128, and the ring records the position each slot
 * holds).  For entry i, ring sequence dst_seqs[i] receives the window of
 * paged sequence src_seqs[i] that ends before position end[i]: slot c gets
 * the row of the largest position p < end[i] with p mod 128 == c (K and V,
 * bit for bit) and slot_pos = p; a slot with no such position (end[i] <= c)
 * gets slot_pos -1 and keeps its rows.  The result equals the ring that
 * appending positions 0..end[i]-1 in order would leave, so the ring-based
 * calls (swa_sink_prefill_chunk, swa_sink_prefill_varlen) can continue a
 * sequence kept in pages.  A needed position whose block entry is not a
 * block id of the pool gets slot_pos -1 and sets KVR_DEV_BAD_BLOCK; a
 * sequence id outside either layout sets KVR_DEV_BAD_SEQ and the entry is
 * skipped.  The rows move as bulk copies through shared memory; if they do
 * not land within 2 s, KVR_DEV_TIMEOUT is set and that entry's K or V rows
 * are left as they were.  pages: PAGED; ring: RING with the same
 * num_kv_heads; src_seqs, dst_seqs [n] int32 and end [n] int64 are device
 * arrays; no two entries may name the same dst sequence.  n = 0 is a no-op.
 */
kvr_status kv_ring_gather_pages(const kvr_kv_layout *pages, const kvr_kv_layout *ring, const int32_t *src_seqs,
                                const int32_t *dst_seqs, const int64_t *end, int32_t n, void *stream);

/*
 * Size of the fixed device scratch array used by full_attn_decode_noalloc:
 * 32 MiB.  It is part of the library's device image, so a device holds it
 * from the first call of any kind into this library on that device (not only
 * the first no-allocation call) until the process exits.
 */
#define KVR_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * full_attn_decode for callers that cannot allocate device memory.  The
 * pages describe no such call: it exists for callers that are handed only
 * their input and output buffers, with no allocator and no workspace --
 * e.g. a plugin whose host passes tensors but owns all device memory, or a
 * server that reserves the whole GPU for KV pools at start-up and forbids
 * allocations afterwards.
 *
 * Same arguments and results as full_attn_decode, minus the workspace: the
 * split partials go to a fixed array inside the library's device image
 * (KVR_NOALLOC_SCRATCH_BYTES).  Nothing is allocated or freed, on the device
 * or through any library.  A call whose partials would not fit, i.e.
 * full_attn_decode_workspace_size(B, Hq, Hkv, max_ctx) >
 * KVR_NOALLOC_SCRATCH_BYTES, returns KVR_EWORKSPACE and launches nothing.
 *
 * The array is shared by every call in the process and keeps whatever the
 * last call left in it; no part of it needs to start at zero (each partial
 * the merge reads is written earlier in the same call).  Calls that can
 * overlap on the GPU -- on different streams, or from different host
 * threads without ordering -- race on the array and give wrong results:
 * order them (for example, issue them all on one stream).
 *
 * The first call on each device looks up the array's device address with
 * cudaGetSymbolAddress (with that device current); make that first call
 * before any stream capture begins.  A first call made while its stream is
 * being captured returns KVR_EINVAL (with a message saying so) and launches
 * nothing.  The looked-up address belongs to the device's current context:
 * after cudaDeviceReset it is looked up again on the next call (which again
 * must not be inside a capture).
 */
kvr_status full_attn_decode_noalloc(const kvr_bf16 *q, const int64_t *pos, const int32_t *seq, int32_t B,
                                    int32_t Hq, const kvr_kv_layout *pool, const float *rope_cos_sin,
                                    int64_t max_pos, float softmax_scale, int64_t max_ctx, kvr_bf16 *out,
                                    void *stream);

/*
 * Chunked prefill over a windowed layer (gaudi-cookbook "What was built":
 * banded tiles with an fp32 softmax that includes the sink).  Row i of the
 * chunk is position P0 + i of sequence `seq`; it attends positions
 * (P0 + i - 128, P0 + i]: those below P0 from the ring (its state before the
 * chunk, slot tags checked), those from P0 on from chunk_kv row (pos - P0).
 * The softmax starts from the sink, so the sink joins the denominator only.
 * q [C][Hq][192] bf16 un-rotated; chunk_kv: LINEAR, num_rows >= C, holding
 * this chunk's K/V as written by kv_ring_append_rope; ring: RING;
 * out [C][Hq][128] bf16.  Afterwards the caller appends the chunk's last
 * min(C, 128) tokens to the ring.
 */
kvr_status swa_sink_prefill_chunk(const kvr_bf16 *q, int64_t P0, int32_t C, int32_t seq, int32_t Hq,
                                  const kvr_kv_layout *chunk_kv, const kvr_kv_layout *ring,
                                  const float *sinks, const float *rope_cos_sin, int64_t max_pos,
                                  float softmax_scale, kvr_bf16 *out, void *stream);

/*
 * Chunked prefill over a full-attention layer (gaudi-cookbook "Tiled
 * global-attention prefill": softmax is per query row, so query tiles need no
 * merge).  Row i of the chunk is position P0 + i of sequence `seq` and
 * attends positions 0..P0 + i of the paged pool, into which the chunk's own
 * K/V were already appended.  No sink.
 * q [C][Hq][192] bf16 un-rotated; pool: PAGED; out [C][Hq][128] bf16.
 * P0 + C <= max_pos and <= max_blocks*block_size.
 */
kvr_status full_attn_prefill_chunk(const kvr_bf16 *q, int64_t P0, int32_t C, int32_t seq, int32_t Hq,
                                   const kvr_kv_layout *pool, const float *rope_cos_sin,
                                   int64_t max_pos, float softmax_scale, kvr_bf16 *out,
                                   void *stream);

/*
 * Batches of chunks of different lengths ("varlen"), for both layer kinds.
 * Chunk s (s < n) is C_s = cu_rows[s+1] - cu_rows[s] query rows at positions
 * P0[s] .. P0[s] + C_s - 1 of sequence seq[s]; its q rows are rows
 * cu_rows[s] .. cu_rows[s+1]-1 of q, and its outputs the same rows of out.
 * Each row attends exactly as in the single-chunk calls above.  Uses:
 *  - multi-token-prediction verification (the Chinese Xiaomi article,
 *    section "Decode加速与多模态优化": the model proposes several tokens per
 *    step and they are checked in one pass): C_s = 2..4 draft tokens per
 *    sequence, causal within the draft, each sequence's K/V read once;
 *  - batched prefill of requests of different lengths (section
 *    "调度与Prefill优化": length buckets 0-64K / 64K-256K / 256K-1M);
 *  - mixed batches of prefill chunks and single decode tokens (C_s = 1).
 * cu_rows [n+1] int32, P0 [n] int64, seq [n] int32 are DEVICE arrays, read
 * by the kernels (the work plan is built on the device, so the call can be
 * captured in a CUDA graph and the lengths can change between replays).
 * T (host) is the number of rows of q/out; cu_rows must be non-decreasing
 * within [0, T] (else that chunk is skipped and KVR_DEV_BAD_ROWS set).  A
 * chunk whose sequence id is outside the layout (KVR_DEV_BAD_SEQ) or whose
 * P0 < 0 or P0 + C_s exceeds the bound (KVR_DEV_BAD_POS) has its rows written
 * as zeros.  Rows of q/out outside every chunk are neither read nor written.
 * q [T][Hq][192] bf16 un-rotated; out [T][Hq][128] bf16.
 * workspace: device scratch (16-byte aligned, no initialisation needed) of
 * the size the matching *_workspace_size call returns; it holds the plan
 * (and for full layers the key-split partials).  n = 0 or T = 0 is a no-op.
 */

/* Workspace bytes for full_attn_prefill_varlen (0 on bad arguments). */
size_t full_attn_prefill_varlen_workspace_size(int32_t n, int64_t T, int32_t Hq, int32_t Hkv, int64_t max_ctx);

/*
 * Full-attention layer, varlen: chunk s attends positions 0..P0[s] + i of
 * the paged pool, into which its K/V were already appended.  Every
 * P0[s] + C_s must be <= max_ctx; max_ctx <= max_pos and
 * <= max_blocks*block_size.  Runs on the tensor cores; a chunk of at most
 * 256 / (Hq/Hkv) rows (a decode or draft-verification chunk) is also cut
 * along its keys into splits that run in parallel and are merged by
 * log-sum-exp, like full_attn_decode.
 */
kvr_status full_attn_prefill_varlen(const kvr_bf16 *q, const int32_t *cu_rows, const int64_t *P0,
                                    const int32_t *seq, int32_t n, int64_t T, int32_t Hq,
                                    const kvr_kv_layout *pool, const float *rope_cos_sin, int64_t max_pos,
                                    float softmax_scale, int64_t max_ctx, void *workspace,
                                    size_t workspace_bytes, kvr_bf16 *out, void *stream);

/* Workspace bytes for swa_sink_prefill_varlen (0 on bad arguments). */
size_t swa_sink_prefill_varlen_workspace_size(int32_t n);

/*
 * Windowed layer, varlen: row i of chunk s attends positions
 * (P0[s] + i - 128, P0[s] + i]: those below P0[s] from sequence seq[s]'s ring
 * (its state before the chunk, slot tags checked), those from P0[s] on from
 * chunk_kv row cu_rows[s] + (pos - P0[s]).  Sink as in swa_sink_prefill_chunk.
 * chunk_kv: LINEAR with num_rows >= T, the batch's K/V as written by
 * kv_ring_append_rope; P0[s] + C_s must be <= max_pos.  For a draft
 * verification, the draft's K/V go to chunk_kv and the ring is left as it was
 * before the draft; the accepted tokens are appended to the ring afterwards.
 */
kvr_status swa_sink_prefill_varlen(const kvr_bf16 *q, const int32_t *cu_rows, const int64_t *P0,
                                   const int32_t *seq, int32_t n, int64_t T, int32_t Hq,
                                   const kvr_kv_layout *chunk_kv, const kvr_kv_layout *ring,
                                   const float *sinks, const float *rope_cos_sin, int64_t max_pos,
                                   float softmax_scale, void *workspace, size_t workspace_bytes,
                                   kvr_bf16 *out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KVRING_H */
