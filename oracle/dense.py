"""Dense numpy formulation of windowed attention with a sink (fp64).

TEST INFRASTRUCTURE ONLY -- a second, independent statement of the same
definition as ``oracle.c``, used to check that one against another
formulation.  It shares no code with ``oracle.c`` or with the CUDA path.

Here the sink is a virtual extra key whose logit is the sink value and whose
value vector is zero: a column appended to the [nq, nk] logit matrix.  The
softmax over that widened row puts the sink in the denominator only, which is
what colibri's "MiMo-V2.6" page ("What the engine implements") says the sink
does.  Masked pairs (outside the causal window) get -inf.  RoPE is rotate-half
on the first 64 dims with inv_freq_i = theta^(-2i/64), evaluated in fp64.
"""
from __future__ import annotations

import numpy as np

DQK, DV, DROT = 192, 128, 64


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float64, exactly."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate-half RoPE on dims 0..63 of x[..., 192] (positions broadcast on axis 0)."""
    half = DROT // 2
    inv = theta ** (-(2.0 * np.arange(half)) / DROT)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv[None, :]
    shape = (len(pos),) + (1,) * (x.ndim - 2) + (half,)
    c, s = np.cos(ang).reshape(shape), np.sin(ang).reshape(shape)
    y = x.copy()
    x1, x2 = x[..., :half], x[..., half:DROT]
    y[..., :half] = x1 * c - x2 * s
    y[..., half:DROT] = x2 * c + x1 * s
    return y


def attend(q, qpos, k, v, k0, theta, value_scale, softmax_scale, window, sinks=None,
           pad_v_to=None):
    """Dense attention of one sequence.

    q [nq, hq, 192] and k [nk, hkv, 192] and v [nk, hkv, 128] are bf16 bit
    arrays (uint16) or float64 arrays; key row r is position k0 + r.
    window 0 = full causal attention.  sinks [hq] or None.  pad_v_to: if set,
    V is zero-padded to that width before the product and the extra output
    columns are dropped afterwards (the gaudi-cookbook layout).
    Returns out [nq, hq, 128] float64.
    """
    def as64(a):
        a = np.asarray(a)
        return bf16_bits_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)

    q, k, v = as64(q), as64(k), as64(v)
    qpos = np.asarray(qpos, dtype=np.int64)
    nq, hq, _ = q.shape
    nk, hkv, _ = k.shape
    g = hq // hkv
    kpos = k0 + np.arange(nk, dtype=np.int64)
    qr = rope(q, qpos, theta)
    kr = rope(k, kpos, theta)
    vr = v * value_scale
    if pad_v_to is not None:
        vr = np.concatenate([vr, np.zeros(vr.shape[:-1] + (pad_v_to - DV,))], axis=-1)
    allowed = kpos[None, :] <= qpos[:, None]
    if window:
        allowed &= kpos[None, :] > qpos[:, None] - window
    out = np.zeros((nq, hq, DV))
    for h in range(hq):
        kv = h // g
        logits = qr[:, h, :] @ kr[:, kv, :].T * softmax_scale          # [nq, nk]
        logits = np.where(allowed, logits, -np.inf)
        vals = vr[:, kv, :]
        if sinks is not None:
            logits = np.concatenate([logits, np.full((nq, 1), float(sinks[h]))], axis=1)
            vals = np.concatenate([vals, np.zeros((1, vals.shape[1]))], axis=0)
        m = logits.max(axis=1, keepdims=True)
        m = np.where(np.isfinite(m), m, 0.0)
        e = np.exp(logits - m)
        z = e.sum(axis=1, keepdims=True)
        o = (e @ vals) / np.where(z > 0, z, 1.0)
        out[:, h, :] = o[:, :DV]
    return out
