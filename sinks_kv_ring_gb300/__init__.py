"""Hybrid-SWA attention with sinks over a ring KV cache, for GB300 (sm_103a).

Thin Python binding over the C ABI of ``libkvring.so`` (``include/kvring.h``).
It only marshals arguments: every step of the attention path runs in the
library's CUDA kernels.  PyTorch supplies device memory and streams.  There
is no fallback: if the library is missing, every call raises.

The five calls (colibri "MiMo-V2.6", "What the engine implements";
gaudi-cookbook "MiMo-V2.6-Flash on Gaudi 2", "What was built"):

  kv_ring_append_rope     RoPE k (dims 0..63), scale v, write ring / pages / rows
  swa_sink_decode         one token over a 128-slot ring with a per-head sink
  full_attn_decode        one token over a paged pool, split-K + LSE combine
  swa_sink_prefill_chunk  a chunk over ring + chunk rows, sink in the softmax
  full_attn_prefill_chunk a chunk over a paged pool, causal

and the batched forms of the two prefill calls, ``swa_sink_prefill_varlen``
and ``full_attn_prefill_varlen``: n chunks of different lengths in one call
(multi-token-prediction draft verification, mixed prefill/decode batches).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "KvrError", "RingLayout", "PagedLayout", "LinearLayout", "lib", "rope_table",
    "kv_ring_append_rope", "swa_sink_decode", "full_attn_decode", "full_attn_decode_workspace_size",
    "swa_sink_prefill_chunk", "full_attn_prefill_chunk", "device_status", "full_attn_decode_noalloc",
    "kv_ring_snapshot", "kv_ring_restore", "ring_snapshot_alloc",
    "full_attn_prefill_varlen", "swa_sink_prefill_varlen", "full_attn_prefill_varlen_workspace_size",
    "swa_sink_prefill_varlen_workspace_size",
    "DQK", "DV", "DROT", "WINDOW",
]

DQK, DV, DROT, WINDOW = 192, 128, 64, 128
LAYOUT_RING, LAYOUT_PAGED, LAYOUT_LINEAR = 1, 2, 3
DEV_BAD_POS, DEV_BAD_SEQ, DEV_BAD_BLOCK, DEV_TIMEOUT, DEV_BAD_ROWS, DEV_FREE_FULL = 1, 2, 4, 8, 16, 32

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvring.so")
_lib = None
_lock = threading.Lock()


class KvrError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"kvring error {code}: {msg}")
        self.code = code


class _Layout(ctypes.Structure):
    _fields_ = [
        ("kind", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("slot_pos", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p),
        ("num_seqs", ctypes.c_int32),
        ("max_blocks", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32),
        ("num_rows", ctypes.c_int64),
    ]


def lib():
    """The loaded libkvring.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise ImportError(f"{LIB_PATH} is missing: build it with sinks_kv_ring_gb300.build.build()")
                L = ctypes.CDLL(LIB_PATH)
                p, i32, i64, f32, f64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_double
                L.kvr_last_error.restype = ctypes.c_char_p
                L.kvr_last_error.argtypes = []
                L.kvr_device_status.restype = ctypes.c_int
                L.kvr_device_status.argtypes = [p, ctypes.c_int]
                L.kvr_debug_stall_next.restype = ctypes.c_int
                L.kvr_debug_stall_next.argtypes = [i32, i64]
                L.kvr_rope_table_build.restype = ctypes.c_int
                L.kvr_rope_table_build.argtypes = [f64, i64, p, ctypes.c_int]
                L.kv_ring_append_rope.restype = ctypes.c_int
                L.kv_ring_append_rope.argtypes = [p, p, p, p, i32, i32, p, i64, f32, p, p]
                L.swa_sink_decode.restype = ctypes.c_int
                L.swa_sink_decode.argtypes = [p, p, p, i32, i32, p, p, p, i64, f32, p, p]
                L.full_attn_decode_workspace_size.restype = ctypes.c_size_t
                L.full_attn_decode_workspace_size.argtypes = [i32, i32, i32, i64]
                L.full_attn_decode.restype = ctypes.c_int
                L.full_attn_decode.argtypes = [p, p, p, i32, i32, p, p, i64, f32, i64, p, ctypes.c_size_t, p, p]
                L.kv_ring_snapshot.restype = ctypes.c_int
                L.kv_ring_snapshot.argtypes = [p, p, i32, p, p, p, p]
                L.kv_ring_restore.restype = ctypes.c_int
                L.kv_ring_restore.argtypes = [p, p, i32, p, p, p, p]
                L.full_attn_decode_noalloc.restype = ctypes.c_int
                L.full_attn_decode_noalloc.argtypes = [p, p, p, i32, i32, p, p, i64, f32, i64, p, p]
                L.swa_sink_prefill_chunk.restype = ctypes.c_int
                L.swa_sink_prefill_chunk.argtypes = [p, i64, i32, i32, i32, p, p, p, p, i64, f32, p, p]
                L.full_attn_prefill_chunk.restype = ctypes.c_int
                L.full_attn_prefill_chunk.argtypes = [p, i64, i32, i32, i32, p, p, i64, f32, p, p]
                L.full_attn_prefill_varlen_workspace_size.restype = ctypes.c_size_t
                L.full_attn_prefill_varlen_workspace_size.argtypes = [i32, i64, i32, i32, i64]
                L.full_attn_prefill_varlen.restype = ctypes.c_int
                L.full_attn_prefill_varlen.argtypes = [p, p, p, p, i32, i64, i32, p, p, i64, f32, i64, p,
                                                       ctypes.c_size_t, p, p]
                L.swa_sink_prefill_varlen_workspace_size.restype = ctypes.c_size_t
                L.swa_sink_prefill_varlen_workspace_size.argtypes = [i32]
                L.swa_sink_prefill_varlen.restype = ctypes.c_int
                L.swa_sink_prefill_varlen.argtypes = [p, p, p, p, i32, i64, i32, p, p, p, p, i64, f32, p,
                                                      ctypes.c_size_t, p, p]
                L.kv_pages_release_window.restype = ctypes.c_int
                L.kv_pages_release_window.argtypes = [p, i32, i32, i32, i32, p, p, p, i32, i32, p, p, i32, p]
                L.kv_ring_gather_pages.restype = ctypes.c_int
                L.kv_ring_gather_pages.argtypes = [p, p, p, p, p, i32, p]
                _lib = L
    return _lib


def _check(rc: int):
    if rc != 0:
        raise KvrError(rc, lib().kvr_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _want(t, name, dtype, dim=None, cuda=True):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if dim is not None and t.dim() != dim:
        raise ValueError(f"{name} must have {dim} dims, got shape {tuple(t.shape)}")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# The C ABI takes bare pointers, so the sizes the kernels index by are
# checked here, before any launch.

def _want_q(q):
    _want(q, "q", torch.bfloat16, 3)
    if q.shape[2] != DQK:
        raise ValueError(f"q must be [rows, Hq, {DQK}], got shape {tuple(q.shape)}")


def _want_table(table):
    _want(table, "table", torch.float32, 3)
    if tuple(table.shape[1:]) != (DROT // 2, 2):
        raise ValueError(f"table must be [max_pos, {DROT // 2}, 2] (cos, sin), got shape {tuple(table.shape)}")


def _want_len(t, name, n):
    if t.shape[0] != n:
        raise ValueError(f"{name} must have {n} entries, got {t.shape[0]}")


def _out(out, rows, hq, like):
    if out is None:
        return torch.empty(rows, hq, DV, dtype=torch.bfloat16, device=like.device)
    _want(out, "out", torch.bfloat16, 3)
    if tuple(out.shape) != (rows, hq, DV):
        raise ValueError(f"out must be [{rows}, {hq}, {DV}], got shape {tuple(out.shape)}")
    return out


def _same_device(first, *rest):
    """The library launches on the current CUDA device and reads every pointer
    of a call there, so all of the call's tensors must live on that device."""
    dev = first.device
    cur = torch.cuda.current_device()
    if dev.index != cur:
        raise ValueError(f"the call's tensors are on {dev} but the current device is cuda:{cur} "
                         "(make it current with torch.cuda.device)")
    for t in rest:
        if t is not None and t.device != dev:
            raise ValueError(f"a tensor of the call is on {t.device}, the others on {dev}")


class RingLayout:
    """SWA pool of one layer: k [S, Hkv, 128, 192], v [S, Hkv, 128, 128] bf16,
    slot_pos [S, 128] int32 (-1 = empty)."""

    def __init__(self, k, v, slot_pos):
        _want(k, "ring.k", torch.bfloat16, 4)
        _want(v, "ring.v", torch.bfloat16, 4)
        _want(slot_pos, "ring.slot_pos", torch.int32, 2)
        S, H, W, D = k.shape
        if W != WINDOW or D != DQK or tuple(v.shape) != (S, H, WINDOW, DV) or tuple(slot_pos.shape) != (S, WINDOW):
            raise ValueError("ring tensors have inconsistent shapes")
        self.k, self.v, self.slot_pos = k, v, slot_pos
        self.num_seqs, self.num_kv_heads = S, H

    def tensors(self):
        return self.k, self.v, self.slot_pos

    @classmethod
    def empty(cls, num_seqs, num_kv_heads, device="cuda"):
        k = torch.zeros(num_seqs, num_kv_heads, WINDOW, DQK, dtype=torch.bfloat16, device=device)
        v = torch.zeros(num_seqs, num_kv_heads, WINDOW, DV, dtype=torch.bfloat16, device=device)
        sp = torch.full((num_seqs, WINDOW), -1, dtype=torch.int32, device=device)
        return cls(k, v, sp)

    @staticmethod
    def bytes_per_layer(num_seqs, num_kv_heads, elem_bytes=2):
        """Ring K+V bytes of one layer (slot tags not counted)."""
        return num_seqs * num_kv_heads * WINDOW * (DQK + DV) * elem_bytes

    def c(self):
        return _Layout(LAYOUT_RING, self.num_kv_heads, self.k.data_ptr(), self.v.data_ptr(),
                       self.slot_pos.data_ptr(), None, self.num_seqs, 0, 0, 0, 0)


class PagedLayout:
    """Full pool of one layer: k [nblk, Hkv, Bsz, 192], v [nblk, Hkv, Bsz, 128]
    bf16, block_table [S, max_blocks] int32."""

    def __init__(self, k, v, block_table):
        _want(k, "pool.k", torch.bfloat16, 4)
        _want(v, "pool.v", torch.bfloat16, 4)
        _want(block_table, "pool.block_table", torch.int32, 2)
        nb, H, bsz, D = k.shape
        if D != DQK or tuple(v.shape) != (nb, H, bsz, DV):
            raise ValueError("pool tensors have inconsistent shapes")
        self.k, self.v, self.block_table = k, v, block_table
        self.num_blocks, self.num_kv_heads, self.block_size = nb, H, bsz
        self.num_seqs, self.max_blocks = block_table.shape

    def tensors(self):
        return self.k, self.v, self.block_table

    @classmethod
    def contiguous(cls, num_seqs, num_kv_heads, max_ctx, block_size=64, device="cuda", zero=True):
        """A pool where sequence s owns blocks s*mb .. s*mb+mb-1 in order."""
        mb = (max_ctx + block_size - 1) // block_size
        nb = num_seqs * mb
        alloc = torch.zeros if zero else torch.empty
        k = alloc(nb, num_kv_heads, block_size, DQK, dtype=torch.bfloat16, device=device)
        v = alloc(nb, num_kv_heads, block_size, DV, dtype=torch.bfloat16, device=device)
        bt = torch.arange(nb, dtype=torch.int32, device=device).reshape(num_seqs, mb)
        return cls(k, v, bt)

    @staticmethod
    def bytes_per_token(num_kv_heads, elem_bytes=2, v_width=DV):
        """Pool K+V bytes one token adds per layer (v_width=192 models V zero-padded to 192)."""
        return num_kv_heads * (DQK + v_width) * elem_bytes

    def c(self):
        return _Layout(LAYOUT_PAGED, self.num_kv_heads, self.k.data_ptr(), self.v.data_ptr(), None,
                       self.block_table.data_ptr(), self.num_seqs, self.max_blocks, self.block_size,
                       self.num_blocks, 0)


class LinearLayout:
    """Staging rows: k [T, Hkv, 192], v [T, Hkv, 128] bf16."""

    def __init__(self, k, v):
        _want(k, "linear.k", torch.bfloat16, 3)
        _want(v, "linear.v", torch.bfloat16, 3)
        T, H, D = k.shape
        if D != DQK or tuple(v.shape) != (T, H, DV):
            raise ValueError("linear tensors have inconsistent shapes")
        self.k, self.v = k, v
        self.num_rows, self.num_kv_heads = T, H

    def tensors(self):
        return self.k, self.v

    @classmethod
    def empty(cls, rows, num_kv_heads, device="cuda"):
        return cls(torch.empty(rows, num_kv_heads, DQK, dtype=torch.bfloat16, device=device),
                   torch.empty(rows, num_kv_heads, DV, dtype=torch.bfloat16, device=device))

    def c(self):
        return _Layout(LAYOUT_LINEAR, self.num_kv_heads, self.k.data_ptr(), self.v.data_ptr(), None, None,
                       0, 0, 0, 0, self.num_rows)


def rope_table(theta: float, max_pos: int, device="cuda", nthreads: int = 0) -> torch.Tensor:
    """[max_pos, 32, 2] fp32 (cos, sin) table, evaluated on the host in fp64
    by the library, then copied to `device`."""
    host = torch.empty((max_pos, 32, 2), dtype=torch.float32)
    _check(lib().kvr_rope_table_build(float(theta), int(max_pos), _ptr(host), int(nthreads)))
    return host if str(device) == "cpu" else host.to(device)


def kv_ring_append_rope(k, v, pos, seq, table, value_scale, dst, stream=None):
    _want(k, "k", torch.bfloat16, 3)
    _want(v, "v", torch.bfloat16, 3)
    _want(pos, "pos", torch.int64, 1)
    if seq is not None:
        _want(seq, "seq", torch.int32, 1)
    _want_table(table)
    T, H = k.shape[0], k.shape[1]
    if tuple(k.shape) != (T, H, DQK) or tuple(v.shape) != (T, H, DV) or pos.shape[0] != T:
        raise ValueError("k/v/pos shapes disagree")
    if seq is not None and seq.shape[0] != T:
        raise ValueError("seq shape disagrees")
    _same_device(k, v, pos, seq, table, *dst.tensors())
    c = dst.c()
    _check(lib().kv_ring_append_rope(_ptr(k), _ptr(v), _ptr(pos), _ptr(seq), T, H, _ptr(table),
                                     table.shape[0], float(value_scale), ctypes.byref(c), _stream(stream)))


def swa_sink_decode(q, pos, seq, ring, sinks, table, softmax_scale, out=None, stream=None):
    _want_q(q)
    _want(pos, "pos", torch.int64, 1)
    _want(seq, "seq", torch.int32, 1)
    _want(sinks, "sinks", torch.float32, 1)
    _want_table(table)
    B, Hq, _ = q.shape
    _want_len(pos, "pos", B)
    _want_len(seq, "seq", B)
    _want_len(sinks, "sinks", Hq)
    out = _out(out, B, Hq, q)
    _same_device(q, pos, seq, sinks, table, out, *ring.tensors())
    c = ring.c()
    _check(lib().swa_sink_decode(_ptr(q), _ptr(pos), _ptr(seq), B, Hq, ctypes.byref(c), _ptr(sinks),
                                 _ptr(table), table.shape[0], float(softmax_scale), _ptr(out), _stream(stream)))
    return out


def full_attn_decode_workspace_size(B, Hq, Hkv, max_ctx) -> int:
    return int(lib().full_attn_decode_workspace_size(int(B), int(Hq), int(Hkv), int(max_ctx)))


def full_attn_decode(q, pos, seq, pool, table, softmax_scale, max_ctx, workspace=None, out=None, stream=None):
    _want_q(q)
    _want(pos, "pos", torch.int64, 1)
    _want(seq, "seq", torch.int32, 1)
    _want_table(table)
    B, Hq, _ = q.shape
    _want_len(pos, "pos", B)
    _want_len(seq, "seq", B)
    if workspace is None:
        n = full_attn_decode_workspace_size(B, Hq, pool.num_kv_heads, max_ctx)
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=q.device)
    _want(workspace, "workspace", torch.uint8, 1)
    out = _out(out, B, Hq, q)
    _same_device(q, pos, seq, table, workspace, out, *pool.tensors())
    c = pool.c()
    _check(lib().full_attn_decode(_ptr(q), _ptr(pos), _ptr(seq), B, Hq, ctypes.byref(c), _ptr(table),
                                  table.shape[0], float(softmax_scale), int(max_ctx), _ptr(workspace),
                                  workspace.numel(), _ptr(out), _stream(stream)))
    return out


NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


def full_attn_decode_noalloc(q, pos, seq, pool, table, softmax_scale, max_ctx, out=None, stream=None):
    """full_attn_decode for callers that may not allocate device memory: the
    split partials go to a fixed 32 MiB array inside the library instead of a
    workspace.  Calls that may run at the same time on the GPU share that
    array and must be ordered (e.g. one stream).  The first call on a device
    looks the array up; make it before any stream capture."""
    _want_q(q)
    _want(pos, "pos", torch.int64, 1)
    _want(seq, "seq", torch.int32, 1)
    _want_table(table)
    B, Hq, _ = q.shape
    _want_len(pos, "pos", B)
    _want_len(seq, "seq", B)
    out = _out(out, B, Hq, q)
    _same_device(q, pos, seq, table, out, *pool.tensors())
    c = pool.c()
    _check(lib().full_attn_decode_noalloc(_ptr(q), _ptr(pos), _ptr(seq), B, Hq, ctypes.byref(c), _ptr(table),
                                          table.shape[0], float(softmax_scale), int(max_ctx), _ptr(out),
                                          _stream(stream)))
    return out


def swa_sink_prefill_chunk(q, P0, seq, chunk_kv, ring, sinks, table, softmax_scale, out=None, stream=None):
    _want_q(q)
    _want(sinks, "sinks", torch.float32, 1)
    _want_table(table)
    C, Hq, _ = q.shape
    _want_len(sinks, "sinks", Hq)
    out = _out(out, C, Hq, q)
    _same_device(q, sinks, table, out, *chunk_kv.tensors(), *ring.tensors())
    cc, rc = chunk_kv.c(), ring.c()
    _check(lib().swa_sink_prefill_chunk(_ptr(q), int(P0), C, int(seq), Hq, ctypes.byref(cc), ctypes.byref(rc),
                                        _ptr(sinks), _ptr(table), table.shape[0], float(softmax_scale), _ptr(out),
                                        _stream(stream)))
    return out


def full_attn_prefill_chunk(q, P0, seq, pool, table, softmax_scale, out=None, stream=None):
    _want_q(q)
    _want_table(table)
    C, Hq, _ = q.shape
    out = _out(out, C, Hq, q)
    _same_device(q, table, out, *pool.tensors())
    c = pool.c()
    _check(lib().full_attn_prefill_chunk(_ptr(q), int(P0), C, int(seq), Hq, ctypes.byref(c), _ptr(table),
                                         table.shape[0], float(softmax_scale), _ptr(out), _stream(stream)))
    return out


def full_attn_prefill_varlen_workspace_size(n, T, Hq, Hkv, max_ctx) -> int:
    return int(lib().full_attn_prefill_varlen_workspace_size(int(n), int(T), int(Hq), int(Hkv), int(max_ctx)))


def swa_sink_prefill_varlen_workspace_size(n) -> int:
    return int(lib().swa_sink_prefill_varlen_workspace_size(int(n)))


def _varlen_args(q, cu_rows, P0, seq):
    _want_q(q)
    _want(cu_rows, "cu_rows", torch.int32, 1)
    _want(P0, "P0", torch.int64, 1)
    _want(seq, "seq", torch.int32, 1)
    n = seq.numel()
    if cu_rows.numel() != n + 1 or P0.numel() != n:
        raise ValueError(f"cu_rows must have n+1 = {n + 1} entries and P0 n = {n}")
    return n


def full_attn_prefill_varlen(q, cu_rows, P0, seq, pool, table, softmax_scale, max_ctx, workspace=None, out=None,
                             stream=None):
    """n chunks over a full layer's paged pool: chunk s is q rows
    cu_rows[s]..cu_rows[s+1]-1 at positions P0[s].. of sequence seq[s]
    (device int32 / int64 / int32 tensors)."""
    n = _varlen_args(q, cu_rows, P0, seq)
    _want_table(table)
    T, Hq, _ = q.shape
    if workspace is None:
        nb = full_attn_prefill_varlen_workspace_size(n, T, Hq, pool.num_kv_heads, max_ctx)
        workspace = torch.empty(max(nb, 1), dtype=torch.uint8, device=q.device)
    _want(workspace, "workspace", torch.uint8, 1)
    out = _out(out, T, Hq, q)
    _same_device(q, cu_rows, P0, seq, table, workspace, out, *pool.tensors())
    c = pool.c()
    _check(lib().full_attn_prefill_varlen(_ptr(q), _ptr(cu_rows), _ptr(P0), _ptr(seq), n, T, Hq, ctypes.byref(c),
                                          _ptr(table), table.shape[0], float(softmax_scale), int(max_ctx),
                                          _ptr(workspace), workspace.numel(), _ptr(out), _stream(stream)))
    return out


def swa_sink_prefill_varlen(q, cu_rows, P0, seq, chunk_kv, ring, sinks, table, softmax_scale, workspace=None,
                            out=None, stream=None):
    """n chunks over a windowed layer: ring state before each chunk plus the
    batch's own rows in chunk_kv (row cu_rows[s] + i for chunk s)."""
    n = _varlen_args(q, cu_rows, P0, seq)
    _want(sinks, "sinks", torch.float32, 1)
    _want_table(table)
    T, Hq, _ = q.shape
    _want_len(sinks, "sinks", Hq)
    if workspace is None:
        nb = swa_sink_prefill_varlen_workspace_size(n)
        workspace = torch.empty(max(nb, 1), dtype=torch.uint8, device=q.device)
    _want(workspace, "workspace", torch.uint8, 1)
    out = _out(out, T, Hq, q)
    _same_device(q, cu_rows, P0, seq, sinks, table, workspace, out, *chunk_kv.tensors(), *ring.tensors())
    cc, rc = chunk_kv.c(), ring.c()
    _check(lib().swa_sink_prefill_varlen(_ptr(q), _ptr(cu_rows), _ptr(P0), _ptr(seq), n, T, Hq, ctypes.byref(cc),
                                         ctypes.byref(rc), _ptr(sinks), _ptr(table), table.shape[0],
                                         float(softmax_scale), _ptr(workspace), workspace.numel(), _ptr(out),
                                         _stream(stream)))
    return out


def ring_snapshot_alloc(n, num_kv_heads, device="cuda"):
    """Snapshot buffers for n rings: (k [n, Hkv, 128, 192], v [n, Hkv, 128, 128], tags [n, 128])."""
    return (torch.empty(n, num_kv_heads, WINDOW, DQK, dtype=torch.bfloat16, device=device),
            torch.empty(n, num_kv_heads, WINDOW, DV, dtype=torch.bfloat16, device=device),
            torch.empty(n, WINDOW, dtype=torch.int32, device=device))


def _ring_copy(fn, ring, seqs, snap, stream):
    _want(seqs, "seqs", torch.int32, 1)
    k, v, t = snap
    n = seqs.shape[0]
    _want(k, "k_snap", torch.bfloat16, 4)
    _want(v, "v_snap", torch.bfloat16, 4)
    _want(t, "tags_snap", torch.int32, 2)
    if k.shape[0] < n or v.shape[0] < n or t.shape[0] < n or k.shape[1] != ring.num_kv_heads:
        raise ValueError("snapshot buffers too small for the ring / sequence list")
    _same_device(seqs, k, v, t, *ring.tensors())
    c = ring.c()
    _check(fn(ctypes.byref(c), _ptr(seqs), n, _ptr(k), _ptr(v), _ptr(t), _stream(stream)))


def kv_ring_snapshot(ring, seqs, snap, stream=None):
    """Copy the rings (slots + tags) of sequences `seqs` into snapshot buffers."""
    _ring_copy(lib().kv_ring_snapshot, ring, seqs, snap, stream)


def kv_ring_restore(ring, seqs, snap, stream=None):
    """Copy snapshot buffers back into the rings of sequences `seqs`."""
    _ring_copy(lib().kv_ring_restore, ring, seqs, snap, stream)


def kv_pages_release_window(block_table, num_blocks, block_size, seqs, next_pos, free_ids, free_count, lo=None,
                            window=WINDOW, stream=None):
    """Release the pages of a windowed layer kept in pages that no query at or
    after next_pos[i] reads: their ids (entries of block_table, int32
    [num_seqs, max_blocks], ids < num_blocks) are appended to free_ids (int32
    [cap]) at free_count (int32 [1], advanced), their entries set to -1, and
    lo (int32 [num_seqs], optional) advanced.  Everything stays on the
    device."""
    _want(block_table, "block_table", torch.int32, 2)
    _want(seqs, "seqs", torch.int32, 1)
    _want(next_pos, "next_pos", torch.int64, 1)
    _want(free_ids, "free_ids", torch.int32, 1)
    _want(free_count, "free_count", torch.int32, 1)
    S, mb = block_table.shape
    if lo is not None:
        _want(lo, "lo", torch.int32, 1)
        if lo.shape[0] != S:
            raise ValueError("lo must have one entry per sequence of the block table")
    n = seqs.shape[0]
    if next_pos.shape[0] != n or free_count.shape[0] != 1:
        raise ValueError("seqs/next_pos/free_count shapes disagree")
    _same_device(block_table, seqs, next_pos, free_ids, free_count, lo)
    _check(lib().kv_pages_release_window(_ptr(block_table), S, mb, int(block_size), int(num_blocks), _ptr(seqs),
                                         _ptr(next_pos), _ptr(lo), n, int(window), _ptr(free_ids),
                                         _ptr(free_count), free_ids.shape[0], _stream(stream)))


def kv_ring_gather_pages(pages, ring, src_seqs, dst_seqs, end, stream=None):
    """Fill ring rows dst_seqs[i] with the window of paged sequence
    src_seqs[i] that ends before position end[i] (slot p mod 128 <- row p)."""
    _want(src_seqs, "src_seqs", torch.int32, 1)
    _want(dst_seqs, "dst_seqs", torch.int32, 1)
    _want(end, "end", torch.int64, 1)
    n = src_seqs.shape[0]
    if dst_seqs.shape[0] != n or end.shape[0] != n:
        raise ValueError("src_seqs/dst_seqs/end shapes disagree")
    _same_device(src_seqs, dst_seqs, end, *pages.tensors(), *ring.tensors())
    pc, rc = pages.c(), ring.c()
    _check(lib().kv_ring_gather_pages(ctypes.byref(pc), ctypes.byref(rc), _ptr(src_seqs), _ptr(dst_seqs), _ptr(end),
                                      n, _stream(stream)))


def debug_stall_next(launches: int, limit_ns: int) -> None:
    """Test hook: the next `launches` windowed decodes (ring layout) or
    single-chunk full-attention prefills stall on purpose and leave by their
    bounded-wait exit after limit_ns, setting DEV_TIMEOUT (kvr_debug_stall_next)."""
    _check(lib().kvr_debug_stall_next(int(launches), int(limit_ns)))


def device_status(reset: bool = True) -> int:
    """Device status bits (DEV_BAD_POS | DEV_BAD_SEQ | DEV_BAD_BLOCK); synchronises."""
    flags = ctypes.c_uint32(0)
    _check(lib().kvr_device_status(ctypes.byref(flags), 1 if reset else 0))
    return int(flags.value)
