"""fp64 CPU oracle for hybrid-SWA attention with sinks.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
path (``sinks_kv_ring_gb300``) never imports it and shares no code with it.

``oracle.c`` is the definition written out in plain C (compiled here with
gcc, OpenMP over (query, head) rows); ``dense.py`` is an independent numpy
formulation with the sink as a zero-valued extra key.  This module builds the
C library and wraps it for numpy.

Parity pins (tests/test_oracle_pins.py) tie it to what the pages fix; none is
unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, -O2, OpenMP, IEEE math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        p = ctypes.c_void_p
        L.orc_round_bf16.restype = ctypes.c_uint16
        L.orc_round_bf16.argtypes = [ctypes.c_double]
        L.orc_rope_cos_sin.restype = None
        L.orc_rope_cos_sin.argtypes = [ctypes.c_double, ctypes.c_int64, p]
        L.orc_rope_heads.restype = None
        L.orc_rope_heads.argtypes = [p, p, ctypes.c_int64, ctypes.c_double, p]
        L.orc_kv_store_bf16.restype = None
        L.orc_kv_store_bf16.argtypes = [p, p, p, ctypes.c_int64, ctypes.c_int, ctypes.c_double,
                                        ctypes.c_double, p, p]
        L.orc_attend_seq.restype = ctypes.c_int
        L.orc_attend_seq.argtypes = [p, p, ctypes.c_int64, ctypes.c_int, p, p, ctypes.c_int64,
                                     ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_double,
                                     ctypes.c_double, ctypes.c_int64, p, p, p, ctypes.c_int]
        L.orc_max_threads.restype = ctypes.c_int
        L.orc_max_threads.argtypes = []
        _lib = L
    return _lib


def _u16(a) -> np.ndarray:
    """bf16 data (torch bf16 tensor, or uint16 bits) -> contiguous uint16 numpy."""
    if hasattr(a, "dtype") and str(getattr(a, "dtype")) == "torch.bfloat16":
        import torch
        a = a.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)
    return np.ascontiguousarray(np.asarray(a), dtype=np.uint16)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def round_bf16(x: float) -> int:
    return int(lib().orc_round_bf16(float(x)))


def rope_cos_sin(theta: float, pos: int) -> np.ndarray:
    """[32, 2] fp64 (cos, sin) of each rotary frequency at one position."""
    out = np.zeros((32, 2))
    lib().orc_rope_cos_sin(float(theta), int(pos), _ptr(out))
    return out


def rope_heads(x, pos, theta: float) -> np.ndarray:
    """fp64 RoPE of raw bf16 heads x [n, 192] at positions pos [n]."""
    x = _u16(x).reshape(-1, 192)
    pos = np.ascontiguousarray(pos, dtype=np.int64)
    out = np.zeros((x.shape[0], 192))
    lib().orc_rope_heads(_ptr(x), _ptr(pos), x.shape[0], float(theta), _ptr(out))
    return out


def kv_store_bf16(k, v, pos, theta: float, value_scale: float):
    """Stored (bf16 bits) form of a KV write: RNE(rope(k)), RNE(v*scale)."""
    k = _u16(k)
    v = _u16(v)
    n, hkv = k.shape[0], k.shape[1]
    pos = np.ascontiguousarray(pos, dtype=np.int64)
    ko = np.zeros_like(k)
    vo = np.zeros_like(v)
    lib().orc_kv_store_bf16(_ptr(k), _ptr(v), _ptr(pos), n, hkv, float(theta), float(value_scale),
                            _ptr(ko), _ptr(vo))
    return ko, vo


def attend_seq(q, qpos, k, v, k0, theta, value_scale, softmax_scale, window, sinks=None,
               nthreads: int = 0, with_stats: bool = False):
    """fp64 attention of one sequence (see orc_attend_seq in oracle.c).

    q [nq, hq, 192], k [nk, hkv, 192], v [nk, hkv, 128] raw bf16; key row r is
    position k0 + r.  window 0 = full layer.  sinks [hq] or None.
    Returns out [nq, hq, 128] (and stats [nq, hq, 2] = (m, Z) if asked).
    """
    q, k, v = _u16(q), _u16(k), _u16(v)
    nq, hq = q.shape[0], q.shape[1]
    nk, hkv = k.shape[0], k.shape[1]
    qpos = np.ascontiguousarray(qpos, dtype=np.int64)
    out = np.zeros((nq, hq, 128))
    stats = np.zeros((nq, hq, 2))
    s = None
    if sinks is not None:
        s = np.ascontiguousarray(np.asarray(sinks, dtype=np.float64))
    rc = lib().orc_attend_seq(_ptr(q), _ptr(qpos), nq, hq, _ptr(k), _ptr(v), int(k0), nk, hkv,
                              float(theta), float(value_scale), float(softmax_scale), int(window),
                              _ptr(s) if s is not None else None, _ptr(out), _ptr(stats),
                              int(nthreads))
    if rc != 0:
        raise ValueError("orc_attend_seq: bad arguments")
    return (out, stats) if with_stats else out


def max_threads() -> int:
    return int(lib().orc_max_threads())
