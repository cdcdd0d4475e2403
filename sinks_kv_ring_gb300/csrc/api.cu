// api.cu -- the C ABI declared in include/kvring.h: host-side validation of
// every argument the host can see, then the kernel launches.  Nothing here
// allocates device memory.
#include <atomic>
#include <cuda.h>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/kvring.h"
#include "launch.h"

namespace kvr {
void rope_table_fill(double theta, int64_t max_pos, float *out, int nthreads);
}

namespace {

thread_local std::string g_err;

kvr_status fail(kvr_status code, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

kvr_status ok() {
  g_err.clear();
  return KVR_OK;
}

kvr_status cuda_fail(cudaError_t e, const char *what) {
  return fail(KVR_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Device status word, one per device that loads the library.
__device__ unsigned int g_status_word;

constexpr int MAX_DEV = 64;
std::mutex g_mu;
int g_sms[MAX_DEV];

// The calling thread's current CUDA context (the driver's cuCtxGetCurrent,
// looked up once through the runtime, so the library does not link the
// driver library).  Device addresses of this library's symbols belong to the
// context they were looked up in: after cudaDeviceReset, or with another
// context current, they are looked up again.
void *current_ctx() {
  typedef CUresult (*Fn)(CUcontext *);
  static Fn fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<Fn>(p);
  }();
  CUcontext c = nullptr;
  if (fn) fn(&c);
  return c;
}

// Per device: the context its cached addresses belong to, the status word's
// address and the no-allocation scratch array's address (null: not looked up).
struct DevSyms {
  void *ctx;
  void *status;
  void *scratch;
};
DevSyms g_syms[MAX_DEV];

// A lookup that would have run while the caller's stream is captured.
constexpr cudaError_t ERR_CAPTURE = cudaErrorStreamCaptureUnsupported;

// Under g_mu: the entry of the current device, emptied when the context
// current now is not the one its addresses were looked up in.
cudaError_t cur_syms(DevSyms **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= MAX_DEV) return cudaErrorInvalidDevice;
  DevSyms &d = g_syms[dev];
  const void *ctx = current_ctx();
  if (d.ctx != ctx) d = DevSyms{nullptr, nullptr, nullptr};
  *out = &d;
  return cudaSuccess;
}

// Whether work issued to `stream` is being captured into a graph (for the
// legacy default stream: whether any global capture is under way).
bool capturing(void *stream) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cs) != cudaSuccess) {
    (void)cudaGetLastError();  // the query's own error must not reach the launch check
    return true;
  }
  return cs != cudaStreamCaptureStatusNone;
}

// Device address of `sym` for the current device and context, cached in
// `slot`; the lookup (cudaGetSymbolAddress) never runs inside a capture.
template <class T>
cudaError_t symbol_addr(void *DevSyms::*slot, const T &sym, void *stream, void **out) {
  std::lock_guard<std::mutex> lk(g_mu);
  DevSyms *d = nullptr;
  cudaError_t e = cur_syms(&d);
  if (e != cudaSuccess) return e;
  if (!(d->*slot)) {
    if (capturing(stream)) return ERR_CAPTURE;
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, sym);
    if (e != cudaSuccess) return e;
    d->ctx = current_ctx();  // the lookup may have made the primary context current
    d->*slot = p;
  }
  *out = d->*slot;
  return cudaSuccess;
}

// Device address of the status word on the current device (host code may
// not use the symbol itself as an address).
cudaError_t status_ptr(unsigned **out, void *stream) {
  void *p = nullptr;
  const cudaError_t e = symbol_addr(&DevSyms::status, g_status_word, stream, &p);
  *out = static_cast<unsigned *>(p);
  return e;
}

kvr_status state_fail(cudaError_t e, const char *what) {
  if (e == ERR_CAPTURE)
    return fail(KVR_EINVAL,
                "%s: the first call on a device (and the first after a device reset) looks up the library's device "
                "symbols, which cannot happen while its stream is being captured; make one call before capturing",
                what);
  return cuda_fail(e, what);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kvr::KvView view(const kvr_kv_layout &L) {
  kvr::KvView v;
  v.kind = L.kind;
  v.hkv = L.num_kv_heads;
  v.k = L.k;
  v.v = L.v;
  v.slot_pos = L.slot_pos;
  v.block_table = L.block_table;
  v.num_seqs = L.num_seqs;
  v.max_blocks = L.max_blocks;
  v.block_size = L.block_size;
  v.num_blocks = L.num_blocks;
  v.num_rows = L.num_rows;
  return v;
}

kvr_status check_layout(const kvr_kv_layout *L, int want_kind, const char *name) {
  if (!L) return fail(KVR_EINVAL, "%s: layout is NULL", name);
  if (want_kind && L->kind != want_kind) return fail(KVR_EINVAL, "%s: layout kind %d, expected %d", name, L->kind, want_kind);
  if (L->num_kv_heads < 1) return fail(KVR_EINVAL, "%s: num_kv_heads %d", name, L->num_kv_heads);
  if (!L->k || !L->v) return fail(KVR_EINVAL, "%s: k/v pointer is NULL", name);
  if (!aligned16(L->k) || !aligned16(L->v)) return fail(KVR_EINVAL, "%s: k/v not 16-byte aligned", name);
  switch (L->kind) {
    case KVR_LAYOUT_RING:
      if (!L->slot_pos) return fail(KVR_EINVAL, "%s: ring slot_pos is NULL", name);
      if (!aligned16(L->slot_pos)) return fail(KVR_EINVAL, "%s: ring slot_pos not 16-byte aligned", name);
      if (L->num_seqs < 1) return fail(KVR_EINVAL, "%s: num_seqs %d", name, L->num_seqs);
      break;
    case KVR_LAYOUT_PAGED:
      if (!L->block_table) return fail(KVR_EINVAL, "%s: block_table is NULL", name);
      if (L->num_seqs < 1 || L->max_blocks < 1 || L->num_blocks < 1)
        return fail(KVR_EINVAL, "%s: num_seqs/max_blocks/num_blocks must be >= 1", name);
      if (L->block_size < 16 || L->block_size > 1024 || L->block_size % 16)
        return fail(KVR_EUNSUPPORTED, "%s: block_size %d (needs a multiple of 16 in [16, 1024])", name, L->block_size);
      break;
    case KVR_LAYOUT_LINEAR:
      if (L->num_rows < 0) return fail(KVR_EINVAL, "%s: num_rows %lld", name, (long long)L->num_rows);
      break;
    default:
      return fail(KVR_EINVAL, "%s: unknown layout kind %d", name, L->kind);
  }
  return KVR_OK;
}

kvr_status check_table(const float *table, int64_t max_pos) {
  if (!table) return fail(KVR_EINVAL, "rope_cos_sin is NULL");
  if (!aligned16(table)) return fail(KVR_EINVAL, "rope_cos_sin not 16-byte aligned");
  if (max_pos < 1 || max_pos > INT32_MAX) return fail(KVR_ERANGE, "max_pos %lld outside [1, 2^31)", (long long)max_pos);
  return KVR_OK;
}

kvr_status check_heads(int32_t Hq, int32_t Hkv, int max_group) {
  if (Hq < 1 || Hkv < 1 || Hq % Hkv) return fail(KVR_EINVAL, "Hq %d is not a positive multiple of Hkv %d", Hq, Hkv);
  if (max_group && Hq / Hkv > max_group)
    return fail(KVR_EUNSUPPORTED, "Hq/Hkv = %d; this call handles at most %d query heads per KV head", Hq / Hkv, max_group);
  return KVR_OK;
}

cudaStream_t as_stream(void *s) { return static_cast<cudaStream_t>(s); }

}  // namespace

namespace kvr {
namespace {
std::atomic<int> g_stall_left{0};
std::atomic<unsigned long long> g_stall_ns{0};
}  // namespace

void set_stall(int launches, unsigned long long ns) {
  g_stall_ns.store(ns);
  g_stall_left.store(launches);
}

unsigned long long take_stall() {
  int left = g_stall_left.load();
  while (left > 0 && !g_stall_left.compare_exchange_weak(left, left - 1)) {
  }
  return left > 0 ? g_stall_ns.load() : 0ull;
}

namespace {
constexpr int MAX_KSLOT = 16;
unsigned char g_smem_done[MAX_DEV][MAX_KSLOT];
void *g_smem_ctx[MAX_DEV];  // the context g_smem_done[dev] is for
}  // namespace

cudaError_t ensure_smem_limit(int slot, const void *func, int bytes, bool max_carveout) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= MAX_DEV || slot < 0 || slot >= MAX_KSLOT) return cudaErrorInvalidValue;
  std::lock_guard<std::mutex> lk(g_mu);
  void *ctx = current_ctx();
  if (g_smem_ctx[dev] != ctx) {  // a new context: its kernels' attributes start from the defaults
    for (int i = 0; i < MAX_KSLOT; ++i) g_smem_done[dev][i] = 0;
    g_smem_ctx[dev] = ctx;
  }
  if (g_smem_done[dev][slot]) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && max_carveout)
    e = cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess) g_smem_done[dev][slot] = 1;
  return e;
}

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEV) return 152;
  if (!g_sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 152;
    g_sms[dev] = n;
  }
  return g_sms[dev];
}
}  // namespace kvr

extern "C" {

const char *kvr_last_error(void) { return g_err.c_str(); }

kvr_status kvr_device_status(uint32_t *flags, int reset) {
  if (!flags) return fail(KVR_EINVAL, "flags is NULL");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "kvr_device_status");
  unsigned v = 0;
  e = cudaMemcpyFromSymbol(&v, g_status_word, sizeof v);
  if (e != cudaSuccess) return cuda_fail(e, "kvr_device_status");
  *flags = v;
  if (reset) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof zero);
    if (e != cudaSuccess) return cuda_fail(e, "kvr_device_status");
  }
  return ok();
}

kvr_status kvr_debug_stall_next(int32_t launches, int64_t limit_ns) {
  if (launches < 0 || limit_ns < 1000 || limit_ns > 1000000000LL)
    return fail(KVR_EINVAL, "launches %d, limit_ns %lld", launches, (long long)limit_ns);
  kvr::set_stall(launches, (unsigned long long)limit_ns);
  return ok();
}

kvr_status kvr_rope_table_build(double theta, int64_t max_pos, float *host_out, int nthreads) {
  if (!host_out) return fail(KVR_EINVAL, "host_out is NULL");
  if (max_pos < 1) return fail(KVR_EINVAL, "max_pos %lld", (long long)max_pos);
  if (!(theta > 1.0)) return fail(KVR_EINVAL, "theta %g", theta);
  kvr::rope_table_fill(theta, max_pos, host_out, nthreads);
  return ok();
}

kvr_status kv_ring_append_rope(const kvr_bf16 *k, const kvr_bf16 *v, const int64_t *pos, const int32_t *seq,
                               int32_t T, int32_t Hkv, const float *rope_cos_sin, int64_t max_pos,
                               float value_scale, const kvr_kv_layout *dst, void *stream) {
  if (T < 0) return fail(KVR_EINVAL, "T %d", T);
  kvr_status s = check_layout(dst, 0, "dst");
  if (s) return s;
  if (Hkv != dst->num_kv_heads) return fail(KVR_EINVAL, "Hkv %d != dst->num_kv_heads %d", Hkv, dst->num_kv_heads);
  if ((s = check_table(rope_cos_sin, max_pos))) return s;
  if (T == 0) return ok();
  if (!k || !v || !pos) return fail(KVR_EINVAL, "k/v/pos is NULL");
  if (!aligned16(k) || !aligned16(v)) return fail(KVR_EINVAL, "k/v not 16-byte aligned");
  if (dst->kind != KVR_LAYOUT_LINEAR && !seq) return fail(KVR_EINVAL, "seq is NULL");
  if (dst->kind == KVR_LAYOUT_LINEAR && dst->num_rows < T)
    return fail(KVR_EINVAL, "LINEAR dst has %lld rows, T = %d", (long long)dst->num_rows, T);
  unsigned *st = nullptr;
  cudaError_t e = status_ptr(&st, stream);
  if (e != cudaSuccess) return state_fail(e, "kv_ring_append_rope");
  e = kvr::launch_append(k, v, pos, seq, T, Hkv, rope_cos_sin, max_pos, value_scale, view(*dst), st,
                         as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kv_ring_append_rope launch");
  return ok();
}

kvr_status swa_sink_decode(const kvr_bf16 *q, const int64_t *pos, const int32_t *seq, int32_t B, int32_t Hq,
                           const kvr_kv_layout *ring, const float *sinks, const float *rope_cos_sin,
                           int64_t max_pos, float softmax_scale, kvr_bf16 *out, void *stream) {
  if (B < 0) return fail(KVR_EINVAL, "B %d", B);
  kvr_status s = check_layout(ring, 0, "ring");
  if (s) return s;
  if (ring->kind != KVR_LAYOUT_RING && ring->kind != KVR_LAYOUT_PAGED)
    return fail(KVR_EINVAL, "ring: layout kind %d, expected RING or PAGED", ring->kind);
  if ((s = check_heads(Hq, ring->num_kv_heads, 16))) return s;
  if (Hq > 1024) return fail(KVR_EUNSUPPORTED, "Hq %d > 1024", Hq);
  if ((s = check_table(rope_cos_sin, max_pos))) return s;
  if (B == 0) return ok();
  if (!q || !pos || !seq || !sinks || !out) return fail(KVR_EINVAL, "q/pos/seq/sinks/out is NULL");
  if (!aligned16(q) || !aligned16(out)) return fail(KVR_EINVAL, "q/out not 16-byte aligned");
  unsigned *st = nullptr;
  cudaError_t e = status_ptr(&st, stream);
  if (e != cudaSuccess) return state_fail(e, "swa_sink_decode");
  if (ring->kind == KVR_LAYOUT_PAGED)
    e = kvr::launch_swa_decode_paged(q, pos, seq, B, Hq, view(*ring), sinks, rope_cos_sin, max_pos, softmax_scale,
                                     out, st, as_stream(stream));
  else
    e = kvr::launch_swa_decode(q, pos, seq, B, Hq, view(*ring), sinks, rope_cos_sin, max_pos, softmax_scale, out,
                               st, as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "swa_sink_decode launch");
  return ok();
}

size_t full_attn_decode_workspace_size(int32_t B, int32_t Hq, int32_t Hkv, int64_t max_ctx) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || max_ctx < 1) return 0;
  return kvr::full_decode_workspace(B, Hq, Hkv, max_ctx);
}

kvr_status full_attn_decode(const kvr_bf16 *q, const int64_t *pos, const int32_t *seq, int32_t B, int32_t Hq,
                            const kvr_kv_layout *pool, const float *rope_cos_sin, int64_t max_pos,
                            float softmax_scale, int64_t max_ctx, void *workspace, size_t workspace_bytes,
                            kvr_bf16 *out, void *stream) {
  if (B < 0) return fail(KVR_EINVAL, "B %d", B);
  kvr_status s = check_layout(pool, KVR_LAYOUT_PAGED, "pool");
  if (s) return s;
  if ((s = check_heads(Hq, pool->num_kv_heads, 16))) return s;
  if ((s = check_table(rope_cos_sin, max_pos))) return s;
  if (max_ctx < 1 || max_ctx > max_pos)
    return fail(KVR_ERANGE, "max_ctx %lld outside [1, max_pos=%lld]", (long long)max_ctx, (long long)max_pos);
  if (max_ctx > (int64_t)pool->max_blocks * pool->block_size)
    return fail(KVR_ERANGE, "max_ctx %lld exceeds max_blocks*block_size = %lld", (long long)max_ctx,
                (long long)pool->max_blocks * pool->block_size);
  if (B == 0) return ok();
  if (!q || !pos || !seq || !out) return fail(KVR_EINVAL, "q/pos/seq/out is NULL");
  if (!aligned16(q) || !aligned16(out)) return fail(KVR_EINVAL, "q/out not 16-byte aligned");
  const size_t need = kvr::full_decode_workspace(B, Hq, pool->num_kv_heads, max_ctx);
  if (!workspace || workspace_bytes < need)
    return fail(KVR_EWORKSPACE, "workspace %zu bytes, need %zu", workspace ? workspace_bytes : (size_t)0, need);
  if (!aligned16(workspace)) return fail(KVR_EINVAL, "workspace not 16-byte aligned");
  unsigned *st = nullptr;
  cudaError_t e = status_ptr(&st, stream);
  if (e != cudaSuccess) return state_fail(e, "full_attn_decode");
  e = kvr::launch_full_decode(q, pos, seq, B, Hq, view(*pool), rope_cos_sin, max_pos, softmax_scale, max_ctx,
                              workspace, out, st, as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "full_attn_decode launch");
  return ok();
}

kvr_status swa_sink_prefill_chunk(const kvr_bf16 *q, int64_t P0, int32_t C, int32_t seq, int32_t Hq,
                                  const kvr_kv_layout *chunk_kv, const kvr_kv_layout *ring, const float *sinks,
                                  const float *rope_cos_sin, int64_t max_pos, float softmax_scale, kvr_bf16 *out,
                                  void *stream) {
  if (C < 0 || P0 < 0) return fail(KVR_EINVAL, "C %d, P0 %lld", C, (long long)P0);
  kvr_status s = check_layout(ring, KVR_LAYOUT_RING, "ring");
  if (s) return s;
  if ((s = check_layout(chunk_kv, KVR_LAYOUT_LINEAR, "chunk_kv"))) return s;
  if (chunk_kv->num_kv_heads != ring->num_kv_heads)
    return fail(KVR_EINVAL, "chunk_kv has %d KV heads, ring %d", chunk_kv->num_kv_heads, ring->num_kv_heads);
  if ((s = check_heads(Hq, ring->num_kv_heads, 0))) return s;
  if ((s = check_table(rope_cos_sin, max_pos))) return s;
  if (seq < 0 || seq >= ring->num_seqs) return fail(KVR_EINVAL, "seq %d outside [0, %d)", seq, ring->num_seqs);
  if (P0 + C > max_pos) return fail(KVR_ERANGE, "P0 + C = %lld > max_pos %lld", (long long)(P0 + C), (long long)max_pos);
  if (chunk_kv->num_rows < C) return fail(KVR_EINVAL, "chunk_kv has %lld rows, C = %d", (long long)chunk_kv->num_rows, C);
  if (C == 0) return ok();
  if (!q || !sinks || !out) return fail(KVR_EINVAL, "q/sinks/out is NULL");
  if (!aligned16(q) || !aligned16(out)) return fail(KVR_EINVAL, "q/out not 16-byte aligned");
  unsigned *st = nullptr;
  cudaError_t e = status_ptr(&st, stream);
  if (e != cudaSuccess) return state_fail(e, "swa_sink_prefill_chunk");
  e = kvr::launch_swa_prefill_tc(q, P0, C, seq, Hq, view(*chunk_kv), view(*ring), sinks, rope_cos_sin, softmax_scale,
                                 out, st, as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "swa_sink_prefill_chunk launch");
  return ok();
}

kvr_status full_attn_prefill_chunk(const kvr_bf16 *q, int64_t P0, int32_t C, int32_t seq, int32_t Hq,
                                   const kvr_kv_layout *pool, const float *rope_cos_sin, int64_t max_pos,
                                   float softmax_scale, kvr_bf16 *out, void *stream) {
  if (C < 0 || P0 < 0) return fail(KVR_EINVAL, "C %d, P0 %lld", C, (long long)P0);
  kvr_status s = check_layout(pool, KVR_LAYOUT_PAGED, "pool");
  if (s) return s;
  if ((s = check_heads(Hq, pool->num_kv_heads, 0))) return s;
  if ((s = check_table(rope_cos_sin, max_pos))) return s;
  if (seq < 0 || seq >= pool->num_seqs) return fail(KVR_EINVAL, "seq %d outside [0, %d)", seq, pool->num_seqs);
  if (P0 + C > max_pos) return fail(KVR_ERANGE, "P0 + C = %lld > max_pos %lld", (long long)(P0 + C), (long long)max_pos);
  if (P0 + C > (int64_t)pool->max_blocks * pool->block_size)
    return fail(KVR_ERANGE, "P0 + C = %lld exceeds max_blocks*block_size", (long long)(P0 + C));
  if (C == 0) return ok();
  if (!q || !out) return fail(KVR_EINVAL, "q/out is NULL");
  if (!aligned16(q) || !aligned16(out)) return fail(KVR_EINVAL, "q/out not 16-byte aligned");
  unsigned *st = nullptr;
  cudaError_t e = status_ptr(&st, stream);
  if (e != cudaSuccess) return state_fail(e, "full_attn_prefill_chunk");
  e = kvr::launch_full_prefill(q, P0, C, seq, Hq, view(*pool), rope_cos_sin, max_pos, softmax_scale, out, st,
                               as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "full_attn_prefill_chunk launch");
  return ok();
}

static kvr_status ring_copy(const char *name, const kvr_kv_layout *ring, const int32_t *seqs, int32_t n,
                            const kvr_bf16 *k_snap, const kvr_bf16 *v_snap, const int32_t *tags_snap, bool to_ring,
                            void *stream) {
  if (n < 0) return fail(KVR_EINVAL, "%s: n %d", name, n);
  kvr_status s = check_layout(ring, KVR_LAYOUT_RING, "ring");
  if (s) return s;
  if (n == 0) return ok();
  if (!seqs || !k_snap || !v_snap || !tags_snap) return fail(KVR_EINVAL, "%s: a pointer is NULL", name);
  if (!aligned16(k_snap) || !aligned16(v_snap)) return fail(KVR_EINVAL, "%s: snapshot k/v not 16-byte aligned", name);
  if (n > 65535) return fail(KVR_EUNSUPPORTED, "%s: n %d > 65535", name, n);
  unsigned *st = nullptr;
  cudaError_t e = status_ptr(&st, stream);
  if (e != cudaSuccess) return state_fail(e, name);
  e = kvr::launch_ring_copy(view(*ring), seqs, n, const_cast<uint16_t *>(k_snap), const_cast<uint16_t *>(v_snap),
                            const_cast<int32_t *>(tags_snap), to_ring, st, as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, name);
  return ok();
}

kvr_status kv_ring_snapshot(const kvr_kv_layout *ring, const int32_t *seqs, int32_t n, kvr_bf16 *k_snap,
                            kvr_bf16 *v_snap, int32_t *tags_snap, void *stream) {
  return ring_copy("kv_ring_snapshot", ring, seqs, n, k_snap, v_snap, tags_snap, false, stream);
}

namespace {

kvr_status check_varlen(const char *who, const kvr_bf16 *q, const int32_t *cu_rows, const int64_t *P0,
                        const int32_t *seq, int32_t n, int64_t T, const kvr_bf16 *out) {
  if (n < 0 || T < 0 || T > INT32_MAX) return fail(KVR_EINVAL, "%s: n %d, T %lld", who, n, (long long)T);
  if (n == 0 || T == 0) return KVR_OK;
  if (!q || !cu_rows || !P0 || !seq || !out) return fail(KVR_EINVAL, "%s: q/cu_rows/P0/seq/out is NULL", who);
  if (!aligned16(q) || !aligned16(out)) return fail(KVR_EINVAL, "%s: q/out not 16-byte aligned", who);
  return KVR_OK;
}

}  // namespace

size_t full_attn_prefill_varlen_workspace_size(int32_t n, int64_t T, int32_t Hq, int32_t Hkv, int64_t max_ctx) {
  if (n < 1 || T < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv || max_ctx < 1) return 0;
  return kvr::varlen_sizes(n, T, Hq, Hkv, max_ctx, 256, true).bytes;
}

size_t swa_sink_prefill_varlen_workspace_size(int32_t n) {
  if (n < 1) return 0;
  return kvr::varlen_sizes(n, 0, 1, 1, 1, 256, false).bytes;
}

kvr_status full_attn_prefill_varlen(const kvr_bf16 *q, const int32_t *cu_rows, const int64_t *P0, const int32_t *seq,
                                    int32_t n, int64_t T, int32_t Hq, const kvr_kv_layout *pool,
                                    const float *rope_cos_sin, int64_t max_pos, float softmax_scale, int64_t max_ctx,
                                    void *workspace, size_t workspace_bytes, kvr_bf16 *out, void *stream) {
  const char *who = "full_attn_prefill_varlen";
  kvr_status s = check_layout(pool, KVR_LAYOUT_PAGED, "pool");
  if (s) return s;
  if ((s = check_heads(Hq, pool->num_kv_heads, 0))) return s;
  if ((s = check_table(rope_cos_sin, max_pos))) return s;
  if (max_ctx < 1 || max_ctx > max_pos)
    return fail(KVR_ERANGE, "max_ctx %lld outside [1, max_pos=%lld]", (long long)max_ctx, (long long)max_pos);
  if (max_ctx > (int64_t)pool->max_blocks * pool->block_size)
    return fail(KVR_ERANGE, "max_ctx %lld exceeds max_blocks*block_size = %lld", (long long)max_ctx,
                (long long)pool->max_blocks * pool->block_size);
  if ((s = check_varlen(who, q, cu_rows, P0, seq, n, T, out))) return s;
  if (n == 0 || T == 0) return ok();
  const kvr::VarlenSizes z = kvr::varlen_sizes(n, T, Hq, pool->num_kv_heads, max_ctx, 256, true);
  if (z.items_max >= INT32_MAX || z.prows_max * z.nsp_max >= INT32_MAX)
    return fail(KVR_EUNSUPPORTED, "%s: batch too large for one call (n %d, T %lld)", who, n, (long long)T);
  if (!workspace || workspace_bytes < z.bytes)
    return fail(KVR_EWORKSPACE, "workspace %zu bytes, need %zu", workspace ? workspace_bytes : (size_t)0, z.bytes);
  if (!aligned16(workspace)) return fail(KVR_EINVAL, "workspace not 16-byte aligned");
  unsigned *st = nullptr;
  cudaError_t e = status_ptr(&st, stream);
  if (e != cudaSuccess) return state_fail(e, who);
  e = kvr::launch_full_varlen(q, cu_rows, P0, seq, n, T, Hq, view(*pool), rope_cos_sin, softmax_scale, max_ctx,
                              workspace, out, st, as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "full_attn_prefill_varlen launch");
  return ok();
}

kvr_status swa_sink_prefill_varlen(const kvr_bf16 *q, const int32_t *cu_rows, const int64_t *P0, const int32_t *seq,
                                   int32_t n, int64_t T, int32_t Hq, const kvr_kv_layout *chunk_kv,
                                   const kvr_kv_layout *ring, const float *sinks, const float *rope_cos_sin,
                                   int64_t max_pos, float softmax_scale, void *workspace, size_t workspace_bytes,
                                   kvr_bf16 *out, void *stream) {
  const char *who = "swa_sink_prefill_varlen";
  kvr_status s = check_layout(ring, KVR_LAYOUT_RING, "ring");
  if (s) return s;
  if ((s = check_layout(chunk_kv, KVR_LAYOUT_LINEAR, "chunk_kv"))) return s;
  if (chunk_kv->num_kv_heads != ring->num_kv_heads)
    return fail(KVR_EINVAL, "chunk_kv has %d KV heads, ring %d", chunk_kv->num_kv_heads, ring->num_kv_heads);
  if ((s = check_heads(Hq, ring->num_kv_heads, 0))) return s;
  if ((s = check_table(rope_cos_sin, max_pos))) return s;
  if ((s = check_varlen(who, q, cu_rows, P0, seq, n, T, out))) return s;
  if (chunk_kv->num_rows < T)
    return fail(KVR_EINVAL, "chunk_kv has %lld rows, T = %lld", (long long)chunk_kv->num_rows, (long long)T);
  if (n == 0 || T == 0) return ok();
  if (!sinks) return fail(KVR_EINVAL, "sinks is NULL");
  const kvr::VarlenSizes z = kvr::varlen_sizes(n, T, Hq, ring->num_kv_heads, max_pos, 256, false);
  if (z.items_max >= INT32_MAX)
    return fail(KVR_EUNSUPPORTED, "%s: batch too large for one call (n %d, T %lld)", who, n, (long long)T);
  if (!workspace || workspace_bytes < z.bytes)
    return fail(KVR_EWORKSPACE, "workspace %zu bytes, need %zu", workspace ? workspace_bytes : (size_t)0, z.bytes);
  if (!aligned16(workspace)) return fail(KVR_EINVAL, "workspace not 16-byte aligned");
  unsigned *st = nullptr;
  cudaError_t e = status_ptr(&st, stream);
  if (e != cudaSuccess) return state_fail(e, who);
  e = kvr::launch_swa_varlen(q, cu_rows, P0, seq, n, T, Hq, view(*chunk_kv), view(*ring), sinks, rope_cos_sin,
                             max_pos, softmax_scale, workspace, out, st, as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "swa_sink_prefill_varlen launch");
  return ok();
}

kvr_status kv_ring_restore(const kvr_kv_layout *ring, const int32_t *seqs, int32_t n, const kvr_bf16 *k_snap,
                           const kvr_bf16 *v_snap, const int32_t *tags_snap, void *stream) {
  return ring_copy("kv_ring_restore", ring, seqs, n, k_snap, v_snap, tags_snap, true, stream);
}

kvr_status kv_pages_release_window(int32_t *block_table, int32_t num_seqs, int32_t max_blocks, int32_t block_size,
                                   int32_t num_blocks, const int32_t *seqs, const int64_t *next_pos, int32_t *lo,
                                   int32_t n, int32_t window, int32_t *free_ids, int32_t *free_count,
                                   int32_t free_cap, void *stream) {
  if (n < 0) return fail(KVR_EINVAL, "kv_pages_release_window: n %d", n);
  if (num_seqs < 1 || max_blocks < 1 || num_blocks < 1 || block_size < 1)
    return fail(KVR_EINVAL, "kv_pages_release_window: num_seqs/max_blocks/num_blocks/block_size must be >= 1");
  if (window < 1) return fail(KVR_EINVAL, "kv_pages_release_window: window %d", window);
  if (free_cap < 0) return fail(KVR_EINVAL, "kv_pages_release_window: free_cap %d", free_cap);
  if (!block_table || !free_count) return fail(KVR_EINVAL, "kv_pages_release_window: block_table/free_count is NULL");
  if (n == 0) return ok();
  if (!seqs || !next_pos) return fail(KVR_EINVAL, "kv_pages_release_window: seqs/next_pos is NULL");
  if (free_cap > 0 && !free_ids) return fail(KVR_EINVAL, "kv_pages_release_window: free_ids is NULL");
  unsigned *st = nullptr;
  cudaError_t e = status_ptr(&st, stream);
  if (e != cudaSuccess) return state_fail(e, "kv_pages_release_window");
  e = kvr::launch_pages_release(block_table, num_seqs, max_blocks, block_size, num_blocks, seqs, next_pos, lo, n,
                                window, free_ids, free_count, free_cap, st, as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kv_pages_release_window launch");
  return ok();
}

kvr_status kv_ring_gather_pages(const kvr_kv_layout *pages, const kvr_kv_layout *ring, const int32_t *src_seqs,
                                const int32_t *dst_seqs, const int64_t *end, int32_t n, void *stream) {
  kvr_status s = check_layout(pages, KVR_LAYOUT_PAGED, "pages");
  if (s) return s;
  if ((s = check_layout(ring, KVR_LAYOUT_RING, "ring"))) return s;
  if (pages->num_kv_heads != ring->num_kv_heads)
    return fail(KVR_EINVAL, "pages have %d KV heads, ring %d", pages->num_kv_heads, ring->num_kv_heads);
  if (n < 0) return fail(KVR_EINVAL, "kv_ring_gather_pages: n %d", n);
  if (n == 0) return ok();
  if (!src_seqs || !dst_seqs || !end) return fail(KVR_EINVAL, "kv_ring_gather_pages: src_seqs/dst_seqs/end is NULL");
  unsigned *st = nullptr;
  cudaError_t e = status_ptr(&st, stream);
  if (e != cudaSuccess) return state_fail(e, "kv_ring_gather_pages");
  e = kvr::launch_ring_gather(view(*pages), view(*ring), src_seqs, dst_seqs, end, n, st, as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kv_ring_gather_pages launch");
  return ok();
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Decode without a caller-provided workspace.
//
// Some callers get only their input and output buffers and may not allocate
// device memory (no allocator handed to them, or all memory reserved up front).
// For them full_attn_decode_noalloc keeps its split partials in this fixed
// array, which lives in the library's device image on every device that loads
// the library.  Host code must not use the symbol as an address: the device
// address is looked up once per device with cudaGetSymbolAddress.

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[KVR_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on the current device; looked up on the
// first call made on that device (and again after a device reset).
cudaError_t noalloc_scratch(void **out, void *stream) {
  return symbol_addr(&DevSyms::scratch, g_noalloc_scratch, stream, out);
}

}  // namespace

extern "C" kvr_status full_attn_decode_noalloc(const kvr_bf16 *q, const int64_t *pos, const int32_t *seq,
                                               int32_t B, int32_t Hq, const kvr_kv_layout *pool,
                                               const float *rope_cos_sin, int64_t max_pos, float softmax_scale,
                                               int64_t max_ctx, kvr_bf16 *out, void *stream) {
  if (B < 0) return fail(KVR_EINVAL, "B %d", B);
  kvr_status s = check_layout(pool, KVR_LAYOUT_PAGED, "pool");
  if (s) return s;
  if ((s = check_heads(Hq, pool->num_kv_heads, 16))) return s;
  if ((s = check_table(rope_cos_sin, max_pos))) return s;
  if (max_ctx < 1 || max_ctx > max_pos)
    return fail(KVR_ERANGE, "max_ctx %lld outside [1, max_pos=%lld]", (long long)max_ctx, (long long)max_pos);
  if (max_ctx > (int64_t)pool->max_blocks * pool->block_size)
    return fail(KVR_ERANGE, "max_ctx %lld exceeds max_blocks*block_size = %lld", (long long)max_ctx,
                (long long)pool->max_blocks * pool->block_size);
  if (B == 0) return ok();
  if (!q || !pos || !seq || !out) return fail(KVR_EINVAL, "q/pos/seq/out is NULL");
  if (!aligned16(q) || !aligned16(out)) return fail(KVR_EINVAL, "q/out not 16-byte aligned");
  const size_t need = kvr::full_decode_workspace(B, Hq, pool->num_kv_heads, max_ctx);
  if (need > (size_t)KVR_NOALLOC_SCRATCH_BYTES)
    return fail(KVR_EWORKSPACE,
                "full_attn_decode_noalloc: this batch needs %zu bytes of scratch, the fixed array holds %zu; "
                "use full_attn_decode with a workspace, or a smaller batch or max_ctx",
                need, (size_t)KVR_NOALLOC_SCRATCH_BYTES);
  void *scratch = nullptr;
  cudaError_t e = noalloc_scratch(&scratch, stream);
  if (e != cudaSuccess) return state_fail(e, "full_attn_decode_noalloc: cudaGetSymbolAddress");
  unsigned *st = nullptr;
  e = status_ptr(&st, stream);
  if (e != cudaSuccess) return state_fail(e, "full_attn_decode_noalloc");
  e = kvr::launch_full_decode(q, pos, seq, B, Hq, view(*pool), rope_cos_sin, max_pos, softmax_scale, max_ctx,
                              scratch, out, st, as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "full_attn_decode_noalloc launch");
  return ok();
}
