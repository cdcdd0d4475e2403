"""Shared set-up for the GPU parity tests: seeded raw K/V by position,
filling rings and pools through the library, and the comparison bar.

Raw keys/values of (layer, sequence) are drawn in aligned blocks of BLK
positions, so any position range can be regenerated for the oracle without
keeping copies (the draws happen on the GPU; the oracle gets a host copy of
the same draw, never a value computed by the CUDA path).
"""
from __future__ import annotations

import math

import numpy as np
import torch

import sinks_kv_ring_gb300 as kvr
from sinks_kv_ring_gb300.synth import Synth

BLK = 4096
SCALE = 1.0 / math.sqrt(192.0)

# the parity bar for bf16 outputs with fp32 accumulation
MAX_ABS = 2e-2
REL_RMS = 1e-2


def raw_kv(syn: Synth, hkv: int, seq: int, lo: int, hi: int):
    """Raw bf16 k [hi-lo, hkv, 192] and v [hi-lo, hkv, 128] for positions lo..hi-1."""
    if hi <= lo:
        dev = syn.device
        return (torch.empty(0, hkv, 192, dtype=torch.bfloat16, device=dev),
                torch.empty(0, hkv, 128, dtype=torch.bfloat16, device=dev))
    ks, vs = [], []
    for b in range(lo // BLK, (hi - 1) // BLK + 1):
        ks.append(syn.k(BLK, hkv, seq=seq, start=b * BLK))
        vs.append(syn.v(BLK, hkv, seq=seq, start=b * BLK))
    k = torch.cat(ks)
    v = torch.cat(vs)
    off = lo - (lo // BLK) * BLK
    return k[off:off + hi - lo].contiguous(), v[off:off + hi - lo].contiguous()


def fill_paged(pool, syn: Synth, seqs, ctx_lens, table, vscale, chunk=65536):
    """Append positions 0..ctx-1 of each sequence into the paged pool."""
    dev = pool.k.device
    for s, n in zip(seqs, ctx_lens):
        for lo in range(0, n, chunk):
            hi = min(n, lo + chunk)
            k, v = raw_kv(syn, pool.num_kv_heads, s, lo, hi)
            pos = torch.arange(lo, hi, dtype=torch.int64, device=dev)
            sq = torch.full((hi - lo,), s, dtype=torch.int32, device=dev)
            kvr.kv_ring_append_rope(k, v, pos, sq, table, vscale, pool)


def fill_ring(ring, syn: Synth, seqs, last_pos, table, vscale):
    """Append positions max(0, p-127)..p of each sequence into the ring."""
    dev = ring.k.device
    for s, p in zip(seqs, last_pos):
        lo = max(0, p - 127)
        k, v = raw_kv(syn, ring.num_kv_heads, s, lo, p + 1)
        pos = torch.arange(lo, p + 1, dtype=torch.int64, device=dev)
        sq = torch.full((p + 1 - lo,), s, dtype=torch.int32, device=dev)
        kvr.kv_ring_append_rope(k, v, pos, sq, table, vscale, ring)


def compare(got, want, what=""):
    """Assert the accuracy bar: max |err| <= 2e-2 and relative RMS <= 1e-2."""
    g = got.float().cpu().double().numpy() if isinstance(got, torch.Tensor) else np.asarray(got, dtype=np.float64)
    w = np.asarray(want, dtype=np.float64)
    assert g.shape == w.shape, (g.shape, w.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - w)
    mx = float(err.max()) if err.size else 0.0
    denom = float(np.sqrt(np.mean(w * w))) if w.size else 0.0
    rel = float(np.sqrt(np.mean(err * err)) / denom) if denom > 0 else float(np.sqrt(np.mean(err * err)))
    assert mx <= MAX_ABS, f"{what}: max|err| {mx:.3e} > {MAX_ABS}"
    assert rel <= REL_RMS, f"{what}: rel RMS {rel:.3e} > {REL_RMS}"
    return mx, rel


def compare_rows_vec(got, want, what=""):
    """The bar of compare_rows (max |err| and relative RMS of every (token,
    head) output vector on its own), vectorised for large cases."""
    g = got.float().cpu().double().numpy().reshape(-1, got.shape[-1])
    w = np.asarray(want, dtype=np.float64).reshape(-1, g.shape[-1])
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - w)
    assert err.max() <= MAX_ABS, f"{what}: max|err| {err.max():.3e}"
    rms_w = np.sqrt(np.mean(w * w, axis=1))
    rms_e = np.sqrt(np.mean(err * err, axis=1))
    rel = np.where(rms_w > 0, rms_e / np.where(rms_w > 0, rms_w, 1.0), rms_e)
    worst = int(np.argmax(rel))
    assert rel[worst] <= REL_RMS, f"{what}: row {worst} rel RMS {rel[worst]:.3e}"
    return float(rel[worst])


def compare_rows(got, want, what=""):
    """The bar row by row (each (token, head) output vector on its own), so a
    tiny-valued row (the sink taking the mass) is still held to 1e-2."""
    g = got.float().cpu().double().numpy()
    w = np.asarray(want, dtype=np.float64)
    g2 = g.reshape(-1, g.shape[-1])
    w2 = w.reshape(-1, w.shape[-1])
    worst = 0.0
    for i in range(g2.shape[0]):
        _, rel = compare(g2[i], w2[i], f"{what} row {i}")
        worst = max(worst, rel)
    return worst
