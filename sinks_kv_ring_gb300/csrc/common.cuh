// common.cuh -- device helpers shared by the attention kernels (sm_103a).
//
// Small wrappers over PTX: bf16 packing, cp.async (16-byte global->shared
// copies), ldmatrix, the m16n8k16 bf16 tensor-core MMA with fp32
// accumulation, and ex2.approx.  Plus the device-side views of a KV layout.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

namespace kvr {

constexpr int DQK = 192;
constexpr int DV = 128;
constexpr int DROT = 64;
constexpr int HALF = 32;
constexpr int WIN = 128;
constexpr float LOG2E = 1.4426950408889634f;

// status bits (mirrors KVR_DEV_* in kvring.h)
constexpr unsigned ST_BAD_POS = 1u;
constexpr unsigned ST_BAD_SEQ = 2u;
constexpr unsigned ST_BAD_BLOCK = 4u;
constexpr unsigned ST_BAD_ROWS = 16u;
constexpr unsigned ST_FREE_FULL = 32u;

// Programmatic dependent launch (kernels launched through launch_pdl).
// pdl_wait returns once the kernel before this one on the stream has
// completed and its writes are visible (at once for a plain launch); a kernel
// calls it before its first global-memory access.  pdl_trigger lets a kernel
// launched the same way after this one be scheduled as this one's CTAs leave;
// it is called only after pdl_wait, so a dependent never runs beside this
// kernel's own predecessor.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Prefetch ahead of pdl_wait.  A kernel may read, before its pdl_wait, an
// index that the kernel ahead of it could still be writing, and use it only
// to choose bytes to bring into L2: such a read may see an old value, which
// costs nothing but a useless prefetch, since every value the kernel computes
// with is read again after pdl_wait.  The early read bypasses L1 (.cg), so no
// stale line stays there for the later one.  The prefetch itself is
// prefetch_l2 below.
__device__ __forceinline__ int ld_early_s32(const int32_t *p) {
  int v;
  asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ long long ld_early_s64(const int64_t *p) {
  long long v;
  asm volatile("ld.global.cg.s64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void flag(unsigned *status, unsigned bits) {
  if (status) atomicOr(status, bits);
}

__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

__device__ __forceinline__ uint16_t f2bf(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// two fp32 -> packed bf16x2 (lo in the low half), round to nearest even
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max of three fp32 values (one instruction on sm_100+)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Packed pairs of fp32 (one instruction each on sm_100+): x * y + z and
// x + y element-wise, round to nearest, as fmaf / + on each element.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f32x2_split(uint64_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t x, uint64_t y, uint64_t z) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(x), "l"(y), "l"(z));
  return r;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t x, uint64_t y) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(x), "l"(y));
  return r;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte async copy global -> shared; src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes = 16) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }
// Bulk prefetch of [src, src + bytes) into L2 (both 16-byte multiples); no
// completion to wait for.
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(src), "r"(bytes) : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D = A(16x16, row) * B(16x8, col) + D, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float *d, const uint32_t *a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Shared-memory tiles of bf16 rows, 16-byte chunks XOR-swizzled by (row & 7)
// so that ldmatrix reads of 8 rows at one column hit 8 different banks.
// Row lengths (192 or 128 elements) are multiples of 8 chunks, so the XOR
// stays inside the row.
template <int ROW_ELEMS>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)(row * ROW_ELEMS * 2 + ((chunk ^ (row & 7)) << 4));
}

// Byte offset of 16-byte chunk ch of row r in a [rows][PARTS][128 B] tile
// written by a 3-D (or 4-D) TMA box with the 128-byte swizzle: segment
// seg = r * PARTS + ch / 8, chunk (ch % 8) ^ (seg % 8).  For PARTS = 3 the 8
// rows an ldmatrix reads at one chunk land on 8 different bank groups.
template <int PARTS>
__device__ __forceinline__ uint32_t swrow(int r, int ch) {
  const int seg = r * PARTS + (ch >> 3);
  return (uint32_t)(seg * 128 + (((ch & 7) ^ (seg & 7)) << 4));
}

// Rotate-half RoPE of 8 + 8 elements (dims 8c..8c+7 and 32+8c..32+8c+7 of a
// head).  cs16 holds (cos, sin) of frequencies 8c..8c+7, interleaved; results
// are rounded to bf16 and packed.
__device__ __forceinline__ void rope_pair8(const uint4 &x1v, const uint4 &x2v, const float *cs16,
                                           uint4 &o1, uint4 &o2) {
  const uint16_t *x1 = reinterpret_cast<const uint16_t *>(&x1v);
  const uint16_t *x2 = reinterpret_cast<const uint16_t *>(&x2v);
  uint32_t r1[4], r2[4];
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    float a[2], b[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const float cz = cs16[2 * (e + u)], sn = cs16[2 * (e + u) + 1];
      const float v1 = bf2f(x1[e + u]), v2 = bf2f(x2[e + u]);
      a[u] = v1 * cz - v2 * sn;
      b[u] = v2 * cz + v1 * sn;
    }
    r1[e / 2] = pack_bf16(a[0], a[1]);
    r2[e / 2] = pack_bf16(b[0], b[1]);
  }
  o1 = make_uint4(r1[0], r1[1], r1[2], r1[3]);
  o2 = make_uint4(r2[0], r2[1], r2[2], r2[3]);
}

// Work plan of a batch of chunks of different lengths (written on the device
// by varlen_plan_kernel into the caller's workspace).  Chunk s holds rows
// cu_rows[s] .. cu_rows[s+1]-1 of the batch; its CTA work items are
// item_prefix[s] .. item_prefix[s+1]-1; mode[s] is -1 (rows not addressable:
// nothing is written), 0 (a position or sequence id out of range: its rows
// are written as zeros), or k >= 1 (the keys are cut into k splits).
// Split chunks own partial rows prow_prefix[s] .. prow_prefix[s+1]-1, one per
// (row, q head), each with nsp_max records (m, l) + o[128].  Chunks listed in
// short_list have no items: a kernel for short chunks takes them whole.
struct VarlenPlan {
  const int32_t *cu_rows;
  const int64_t *P0;
  const int32_t *seq;
  int32_t *item_prefix;  // [n+1]
  int32_t *prow_prefix;  // [n+1]
  int32_t *mode;         // [n]
  int32_t *short_list;   // [n+1]: ids of the chunks taken by the short-chunk kernel; count at [n]
  int32_t *slen;         // [n]: keys per split of chunk s (a multiple of 128; mode[s] >= 2 only)
  float2 *pml;           // [prows][nsp_max]: (max in log2 units, sum of exponentials)
  float *po;             // [prows][nsp_max][128]: unnormalised numerators
  int n;
  int nsp_max;
  long long split_len;   // keys per split (a multiple of 128); 0 = no splits
};

// Chunk s of work item b: the last s with item_prefix[s] <= b (the caller
// has checked b < item_prefix[n]).
__device__ __forceinline__ int plan_find(const int32_t *prefix, int n, long long b) {
  int lo = 0, hi = n;  // prefix[lo] <= b < prefix[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= b) lo = mid; else hi = mid;
  }
  return lo;
}

// Device view of a KV layout (see kvr_kv_layout).
struct KvView {
  int kind;
  int hkv;
  uint16_t *k;
  uint16_t *v;
  int32_t *slot_pos;
  const int32_t *block_table;
  int num_seqs;
  int max_blocks;
  int block_size;
  int num_blocks;
  long long num_rows;
};

}  // namespace kvr
