"""Windowed chunked prefill for GQA groups of 8 or more q heads (the band
kernel, one 144-key band per tile of 128 query rows): every output row
against the fp64 oracle, over the cases a band meets -- a full ring before
the chunk, a chunk near position 0, no ring at all, stale ring slots, a
ragged last tile, chunks shorter than one tile, G = 8 .. 128, many items per
CTA (bands sliding along the ring, ranges crossing KV heads) -- plus
chunking invariance.  The other ring sequence and the staging rows past the
chunk hold NaN bits, so a read of either shows up as a non-finite output."""
import numpy as np
import pytest
import torch

import oracle
import sinks_kv_ring_gb300 as kvr
from sinks_kv_ring_gb300.synth import Synth

from kvr_cases import SCALE, compare, compare_rows, compare_rows_vec, fill_ring, raw_kv

pytestmark = pytest.mark.gpu

DEV = "cuda"
NAN_BF16 = 0x7FC0


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sinks_kv_ring_gb300 import build
    build.build()
    kvr.device_status(reset=True)
    yield


@pytest.fixture(scope="module")
def table():
    return kvr.rope_table(1e4, 8192)


def _nan_fill(t):
    t.view(torch.int16).fill_(NAN_BF16)


def _ring_for(syn, hkv, P0, table, vscale, stale=0):
    """Ring of 2 sequences: sequence 1 holds positions P0-128..P0-1 (minus the
    `stale` oldest, whose tags say -1); sequence 0 holds NaN rows tagged
    with the same positions."""
    ring = kvr.RingLayout.empty(2, hkv)
    if P0 > 0:
        fill_ring(ring, syn, [1], [P0 - 1], table, vscale)
        for p in range(max(0, P0 - 128), max(0, P0 - 128 + stale)):
            ring.slot_pos[1, p % 128] = -1
    _nan_fill(ring.k[0])
    _nan_fill(ring.v[0])
    ring.slot_pos[0].copy_(ring.slot_pos[1])
    return ring


def _stage_for(syn, hkv, P0, C, table, vscale, extra=64):
    """Staged chunk rows P0..P0+C-1 of sequence 1, then `extra` NaN rows."""
    stage = kvr.LinearLayout.empty(C + extra, hkv)
    _nan_fill(stage.k)
    _nan_fill(stage.v)
    k, v = raw_kv(syn, hkv, 1, P0, P0 + C)
    kvr.kv_ring_append_rope(k, v, torch.arange(P0, P0 + C, device=DEV), None, table, vscale, stage)
    return stage


@pytest.mark.parametrize("hq,hkv,P0,C,stale", [
    (64, 8, 1000, 300, 0),    # full ring, several tiles, ragged last tile (300 = 18 x 16 + 12)
    (64, 8, 1000, 37, 0),     # shorter than one tile: every item reaches into the ring
    (64, 8, 50, 200, 0),      # the window reaches below position 0
    (64, 8, 0, 161, 0),       # no ring
    (64, 8, 128, 144, 0),     # the ring holds exactly positions 0..127
    (64, 8, 1000, 150, 40),   # the 40 oldest ring slots are stale
    (64, 8, 777, 129, 127),   # only the newest ring slot is live
    (128, 8, 700, 200, 0),    # G = 16: 8 positions per tile
    (64, 4, 333, 129, 0),     # G = 16 with 4 KV heads
    (64, 2, 500, 300, 0),     # G = 32: four positions per tile
    (128, 2, 700, 77, 3),     # G = 64: two positions per tile, stale slots
    (256, 2, 300, 40, 0),     # G = 128: one position per tile
    (8, 1, 400, 90, 0),       # one KV head
    # many items per CTA: bands slide along the ring, ranges cross KV heads
    (64, 8, 1000, 4096, 0),   # 2048 items
    (64, 8, 50, 4096, 0),     # 13-14 items per CTA, the window reaches below position 0
    (64, 8, 1000, 2500, 40),  # 8-9 items per CTA, the 40 oldest ring slots stale
    (64, 8, 130, 3035, 3),    # 10 items per CTA, the last tile 11 rows
    (128, 8, 300, 2000, 5),   # G = 16: the band moves every other item
    (64, 4, 60, 3000, 0),     # G = 16, the window reaches below position 0
])
def test_swa_band_prefill_matches_oracle(hq, hkv, P0, C, stale, table):
    syn = Synth(4100 + hq + P0 + C, dist="plain", device=DEV)
    vscale = 0.707
    sinks = syn.sinks(hq).to(DEV)
    ring = _ring_for(syn, hkv, P0, table, vscale, stale)
    stage = _stage_for(syn, hkv, P0, C, table, vscale)
    q = syn.q(C, hq, hkv, seq=1, start=P0)
    out = kvr.swa_sink_prefill_chunk(q, P0, 1, stage, ring, sinks, table, SCALE)
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    lo = max(0, P0 - 128 + stale)  # positions below lo are absent (stale or before 0)
    k, v = raw_kv(syn, hkv, 1, lo, P0 + C)
    want = oracle.attend_seq(q, np.arange(P0, P0 + C), k, v, lo, 1e4, vscale, SCALE, 128,
                             sinks.double().cpu().numpy())
    compare(out, want, "band prefill")
    compare_rows_vec(out, want, "band prefill")


def test_swa_band_prefill_ring_bands_repeat_bit_for_bit():
    # 27 items per CTA, as in the 8192-row chunk: three calls agree bit for
    # bit, and every row against the oracle.
    hq, hkv, P0, C = 64, 8, 700, 8192
    table = kvr.rope_table(1e4, P0 + C)
    syn = Synth(4150, dist="plain", device=DEV)
    sinks = syn.sinks(hq).to(DEV)
    ring = _ring_for(syn, hkv, P0, table, 0.707)
    stage = _stage_for(syn, hkv, P0, C, table, 0.707)
    q = syn.q(C, hq, hkv, seq=1, start=P0)
    outs = [kvr.swa_sink_prefill_chunk(q, P0, 1, stage, ring, sinks, table, SCALE) for _ in range(3)]
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    k, v = raw_kv(syn, hkv, 1, P0 - 128, P0 + C)
    want = oracle.attend_seq(q, np.arange(P0, P0 + C), k, v, P0 - 128, 1e4, 0.707, SCALE, 128,
                             sinks.double().cpu().numpy())
    compare_rows_vec(outs[0], want, "band prefill, 27-tile runs")


def test_swa_band_prefill_shifted_logits(table):
    # The logit statistics of the tiny sanity workload (mean -25, sd 3; the
    # sink takes most of the mass), where the relative per-row bar binds.
    hq, hkv, P0, C = 64, 8, 260, 300
    syn = Synth(4201, dist="shifted", device=DEV)
    sinks = syn.sinks(hq).to(DEV)
    ring = _ring_for(syn, hkv, P0, table, 0.707)
    stage = _stage_for(syn, hkv, P0, C, table, 0.707)
    q = syn.q(C, hq, hkv, seq=1, start=P0)
    out = kvr.swa_sink_prefill_chunk(q, P0, 1, stage, ring, sinks, table, SCALE)
    k, v = raw_kv(syn, hkv, 1, P0 - 128, P0 + C)
    want = oracle.attend_seq(q, np.arange(P0, P0 + C), k, v, P0 - 128, 1e4, 0.707, SCALE, 128,
                             sinks.double().cpu().numpy())
    compare_rows(out, want, "band prefill, shifted logits")


@pytest.mark.parametrize("chunks", [[200, 312], [16, 16, 480], [1, 130, 381]])
def test_swa_band_chunking_invariance(chunks, table):
    # Prefill in chunks (each chunk's last min(C, 128) rows then committed to
    # the ring) equals one 512-row chunk, within the bar, against the oracle.
    hq, hkv = 64, 8
    syn = Synth(4301, dist="plain", device=DEV)
    sinks = syn.sinks(hq).to(DEV)
    ring = kvr.RingLayout.empty(2, hkv)
    outs, P0 = [], 0
    for C in chunks:
        k, v = raw_kv(syn, hkv, 1, P0, P0 + C)
        stage = kvr.LinearLayout.empty(C, hkv)
        kvr.kv_ring_append_rope(k, v, torch.arange(P0, P0 + C, device=DEV), None, table, 0.707, stage)
        q = syn.q(C, hq, hkv, seq=1, start=P0)
        outs.append(kvr.swa_sink_prefill_chunk(q, P0, 1, stage, ring, sinks, table, SCALE))
        t = min(C, 128)
        kvr.kv_ring_append_rope(k[-t:].contiguous(), v[-t:].contiguous(), torch.arange(P0 + C - t, P0 + C, device=DEV),
                                torch.ones(t, dtype=torch.int32, device=DEV), table, 0.707, ring)
        P0 += C
    out = torch.cat(outs)
    qs = torch.cat([syn.q(C, hq, hkv, seq=1, start=p) for C, p in zip(chunks, np.cumsum([0] + chunks[:-1]))])
    k, v = raw_kv(syn, hkv, 1, 0, 512)
    want = oracle.attend_seq(qs, np.arange(512), k, v, 0, 1e4, 0.707, SCALE, 128, sinks.double().cpu().numpy())
    compare(out, want, "band prefill in chunks")
    compare_rows(out, want, "band prefill in chunks")
    assert kvr.device_status() == 0
