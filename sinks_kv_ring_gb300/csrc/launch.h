// launch.h -- internal launchers called by the C ABI (api.cu) after it has
// validated every host-visible argument.  Each returns the cudaError_t of its
// launch.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace kvr {

// 2-D tensor map over a bf16 tensor viewed as [rows][width], box of 64
// elements x box_rows rows, 128-byte swizzle.  False if encoding fails.
bool make_tma_map_2d(CUtensorMap *m, const void *ptr, long long rows, int width, int box_rows);

// 3-D tensor map over [rows][width] bf16 viewed as [rows][width/64][64]: one
// box brings box_rows whole rows (every 64-element part), so a row is read
// in one pass; in shared memory the box is [row][part][64] with the 128-byte
// swizzle applied per 128-byte segment (segment index = row * parts + part).
// With one_part a box brings a single 64-element part of box_rows rows
// ([row][64], segment index = row); the part is the box's y coordinate.
bool make_tma_map_rows3d(CUtensorMap *m, const void *ptr, long long rows, int width, int box_rows,
                         bool one_part = false);

// Raise a kernel's dynamic shared-memory limit once per (kernel slot, device);
// later launches make no attribute call (so they can sit in a stream capture).
// `slot` is a small distinct integer per kernel.  max_carveout: also ask for
// the largest shared-memory carveout (a kernel that fits two CTAs per SM only
// with it).
cudaError_t ensure_smem_limit(int slot, const void *func, int bytes, bool max_carveout = false);

// Launch with programmatic stream serialisation: the kernel may be scheduled
// before the work ahead of it on the stream has finished, and waits for it on
// the device (pdl_wait) before touching global memory.  This hides the launch
// gap between back-to-back kernels.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// The wait limit of a launch that kvr_debug_stall_next asked to stall (one
// taken per call), or 0 for a normal launch.
void set_stall(int launches, unsigned long long ns);
unsigned long long take_stall();

cudaError_t launch_append(const uint16_t *k, const uint16_t *v, const int64_t *pos, const int32_t *seq,
                          int T, int hkv, const float *table, int64_t max_pos, float value_scale,
                          const KvView &dst, unsigned *status, cudaStream_t st);

cudaError_t launch_swa_decode(const uint16_t *q, const int64_t *pos, const int32_t *seq, int B, int hq,
                              const KvView &ring, const float *sinks, const float *table,
                              int64_t max_pos, float softmax_scale, uint16_t *out, unsigned *status,
                              cudaStream_t st);

// Windowed decode over a PAGED layout: groups of up to 8 q heads per KV head
// go to launch_swa_paged; larger ones run the split decode kernel with the key
// range p-127..p, one split, the sink in the final normalisation.
cudaError_t launch_swa_decode_paged(const uint16_t *q, const int64_t *pos, const int32_t *seq, int B, int hq,
                                    const KvView &pool, const float *sinks, const float *table, int64_t max_pos,
                                    float softmax_scale, uint16_t *out, unsigned *status, cudaStream_t st);
// the same for G <= 8 q heads per KV head (swa_paged.cu: keys as the MMA rows)
cudaError_t launch_swa_paged(const uint16_t *q, const int64_t *pos, const int32_t *seq, int B, int hq,
                             const KvView &pool, const float *sinks, const float *table, int64_t max_pos,
                             float softmax_scale, uint16_t *out, unsigned *status, cudaStream_t st);

// Split plan of the full-attention decode: contexts up to max_ctx are cut
// into at most `splits` pieces of `split_len` keys (a multiple of 64).
struct DecodePlan {
  int splits;
  int split_len;
};
DecodePlan full_decode_plan(int B, int hkv, long long max_ctx);
size_t full_decode_workspace(int B, int hq, int hkv, long long max_ctx);

cudaError_t launch_full_decode(const uint16_t *q, const int64_t *pos, const int32_t *seq, int B, int hq,
                               const KvView &pool, const float *table, int64_t max_pos,
                               float softmax_scale, long long max_ctx, void *ws, uint16_t *out,
                               unsigned *status, cudaStream_t st);

cudaError_t launch_full_prefill(const uint16_t *q, int64_t P0, int C, int seq, int hq, const KvView &pool,
                                const float *table, int64_t max_pos, float softmax_scale, uint16_t *out,
                                unsigned *status, cudaStream_t st);

// Windowed chunked prefill on the tensor cores (prefill_tc.cu).
cudaError_t launch_swa_prefill_tc(const uint16_t *q, int64_t P0, int C, int seq, int hq, const KvView &chunk,
                                  const KvView &ring, const float *sinks, const float *table, float softmax_scale,
                                  uint16_t *out, unsigned *status, cudaStream_t st);
// Windowed chunked prefill for group sizes G >= 8 dividing 128 (swa_band.cu):
// *taken is false when the call does not fit it (nothing launched).
cudaError_t launch_swa_band(const uint16_t *q, int64_t P0, int C, int seq, int hq, const KvView &chunk,
                            const KvView &ring, const float *sinks, const float *table, float softmax_scale,
                            uint16_t *out, unsigned *status, cudaStream_t st, bool *taken);
// The same for a batch of chunks (builds the plan in `ws`, then the band
// kernel for the long chunks and the short-chunk kernel for the others).
cudaError_t launch_swa_band_varlen(const uint16_t *q, const int32_t *cu_rows, const int64_t *P0, const int32_t *seq,
                                   int n, long long T, int hq, const KvView &chunk, const KvView &ring,
                                   const float *sinks, const float *table, int64_t max_pos, float softmax_scale,
                                   void *ws, uint16_t *out, unsigned *status, cudaStream_t st, bool *taken);
// Sizes of the workspace of a varlen call (see VarlenPlan): n chunks, T rows,
// contexts up to max_ctx, CTA items of tile_rows query rows; with `splits`,
// chunks of one item are cut along the keys.
struct VarlenSizes {
  int tile_rows;
  long long split_len;
  int nsp_max;
  long long prows_max;   // partial rows the workspace holds
  long long items_max;   // bound on the CTA items of any plan (the grid size)
  size_t off_prow, off_mode, off_short, off_slen, off_pml, off_po, bytes;
};
VarlenSizes varlen_sizes(int n, long long T, int hq, int hkv, long long max_ctx, int tile_rows, bool splits);
VarlenPlan varlen_plan_view(const VarlenSizes &z, void *ws, const int32_t *cu_rows, const int64_t *P0,
                            const int32_t *seq, int n);
// short_rows > 0: chunks of at most short_rows query rows (C * G) and at most
// short_max_c rows go to short_list instead of getting items.
cudaError_t launch_varlen_plan(const VarlenPlan &p, long long T, int hq, int hkv, int tile_rows, long long max_ctx,
                               int num_seqs, int short_rows, int short_max_c, unsigned *status, cudaStream_t st);
cudaError_t launch_varlen_combine(const VarlenPlan &p, long long prows_max, int hq, uint16_t *out, cudaStream_t st);

// Varlen attention: rows of chunk s are q/out rows cu_rows[s] ..; the plan
// in `ws` is built by the launcher.
cudaError_t launch_full_varlen(const uint16_t *q, const int32_t *cu_rows, const int64_t *P0, const int32_t *seq,
                               int n, long long T, int hq, const KvView &pool, const float *table,
                               float softmax_scale, long long max_ctx, void *ws, uint16_t *out, unsigned *status,
                               cudaStream_t st);
cudaError_t launch_swa_varlen(const uint16_t *q, const int32_t *cu_rows, const int64_t *P0, const int32_t *seq,
                              int n, long long T, int hq, const KvView &chunk, const KvView &ring,
                              const float *sinks, const float *table, int64_t max_pos, float softmax_scale,
                              void *ws, uint16_t *out, unsigned *status, cudaStream_t st);

// Windowed attention of the short chunks of a varlen plan (short_list).
cudaError_t launch_swa_short(const uint16_t *q, const VarlenPlan &plan, int n, long long T, int hq,
                             const KvView &chunk, const KvView &ring, const float *sinks, const float *table,
                             float softmax_scale, uint16_t *out, unsigned *status, cudaStream_t st);
constexpr int SWA_SHORT_ROWS = 32;   // C * G of a short chunk
constexpr int SWA_SHORT_MAX_C = 16;  // C of a short chunk

// 4-D tensor map over LINEAR rows [T][hkv][width] bf16 viewed as
// [T][hkv][width/64][64]: one box brings box_rows consecutive tokens of one
// KV head, every 64-element part (smem [token][part][64], 128-byte swizzle),
// or with one_part a single 64-element part (smem [token][64]).  With
// heads_per_box > 1 (rows of [T][heads][width], e.g. q) a box brings that
// many consecutive heads of each token: smem [token][head][part][64].
bool make_tma_map_tokens4d(CUtensorMap *m, const void *ptr, long long T, int hkv, int width, int box_rows,
                           bool one_part = false, int heads_per_box = 1);

// 3-D tensor map over [rows][hq][width] bf16 (q: width 192, out: width 128)
// for the tensor-core kernel's query tiles: a box of 64 dims x G heads x
// 128/G rows is 128 tile rows (row = position * G + head) of 128 bytes,
// 128-byte swizzled.  False when G does not divide 128 (those group sizes
// move q and out with plain copies).
bool make_tma_map_heads3d(CUtensorMap *m, const void *ptr, long long rows, int hq, int width, int G);

cudaError_t launch_ring_copy(const KvView &ring, const int32_t *seqs, int n, uint16_t *k_snap, uint16_t *v_snap,
                             int32_t *tags_snap, bool to_ring, unsigned *status, cudaStream_t st);

cudaError_t launch_pages_release(int32_t *table, int num_seqs, int max_blocks, int block_size, int num_blocks,
                                 const int32_t *seqs, const int64_t *next_pos, int32_t *lo, int n, int window,
                                 int32_t *free_ids, int32_t *free_count, int free_cap, unsigned *status,
                                 cudaStream_t st);

cudaError_t launch_ring_gather(const KvView &pages, const KvView &ring, const int32_t *src_seqs,
                               const int32_t *dst_seqs, const int64_t *end, int n, unsigned *status,
                               cudaStream_t st);

int num_sms();

}  // namespace kvr
