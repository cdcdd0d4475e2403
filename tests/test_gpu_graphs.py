"""Every call of the C ABI can be captured in a CUDA graph (no host
synchronisation, no allocation inside the calls) and a replay gives the
eager result bit for bit.  Serving loops replay their decode and prefill
steps this way."""
import pytest
import torch

import sinks_kv_ring_gb300 as kvr
from sinks_kv_ring_gb300.synth import Synth

from kvr_cases import SCALE, fill_paged, fill_ring, raw_kv

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sinks_kv_ring_gb300 import build
    build.build()
    kvr.device_status(reset=True)
    yield


@pytest.fixture(scope="module")
def tables():
    return {1e4: kvr.rope_table(1e4, 8192), 1e7: kvr.rope_table(1e7, 8192)}


def _capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fn(s)
    torch.cuda.current_stream().wait_stream(s)
    return g


def _bits(t):
    return t.contiguous().view(torch.int16 if t.element_size() == 2 else torch.int32).clone()


def test_decode_and_prefill_calls_replay_bit_for_bit(tables):
    syn = Synth(7101, dist="plain", device=DEV)
    hq, hkv_s, hkv_f, vs = 16, 2, 2, 0.707
    positions = [200, 1000, 130]
    B = len(positions)
    ring = kvr.RingLayout.empty(B, hkv_s)
    fill_ring(ring, syn, list(range(B)), [p - 1 for p in positions], tables[1e4], vs)
    pool = kvr.PagedLayout.contiguous(B, hkv_f, 2048, block_size=64)
    fill_paged(pool, syn, list(range(B)), positions, tables[1e7], vs)
    q_s, q_f = syn.q(B, hq, hkv_s, seq=50), syn.q(B, hq, hkv_f, seq=51)
    k_s, v_s = syn.k(B, hkv_s, seq=52), syn.v(B, hkv_s, seq=52)
    k_f, v_f = syn.k(B, hkv_f, seq=53), syn.v(B, hkv_f, seq=53)
    pos = torch.tensor(positions, dtype=torch.int64, device=DEV)
    seq = torch.arange(B, dtype=torch.int32, device=DEV)
    sinks = syn.sinks(hq).to(DEV)
    ws = torch.empty(kvr.full_attn_decode_workspace_size(B, hq, hkv_f, 2048), dtype=torch.uint8, device=DEV)
    # a 40-token chunk of sequence 0 at P0 = 1500 for both prefill calls
    P0, C = 1500, 40
    kc, vc = raw_kv(syn, hkv_f, 0, P0, P0 + C)
    kvr.kv_ring_append_rope(kc, vc, torch.arange(P0, P0 + C, device=DEV),
                            torch.zeros(C, dtype=torch.int32, device=DEV), tables[1e7], vs, pool)
    stage = kvr.LinearLayout.empty(C, hkv_s)
    ks2, vs2 = raw_kv(syn, hkv_s, 7, P0, P0 + C)
    q_pf, q_ps = syn.q(C, hq, hkv_f, seq=0, start=P0), syn.q(C, hq, hkv_s, seq=7, start=P0)
    pos_stage = torch.arange(P0, P0 + C, device=DEV)
    outs = {n: torch.empty(*shape, 128, dtype=torch.bfloat16, device=DEV)
            for n, shape in [("swa", (B, hq)), ("full", (B, hq)), ("pf", (C, hq)), ("ps", (C, hq))]}

    def step(st):
        kvr.kv_ring_append_rope(k_s, v_s, pos, seq, tables[1e4], vs, ring, stream=st)
        kvr.kv_ring_append_rope(k_f, v_f, pos, seq, tables[1e7], vs, pool, stream=st)
        kvr.swa_sink_decode(q_s, pos, seq, ring, sinks, tables[1e4], SCALE, out=outs["swa"], stream=st)
        kvr.full_attn_decode(q_f, pos, seq, pool, tables[1e7], SCALE, 2048, workspace=ws, out=outs["full"],
                             stream=st)
        kvr.full_attn_prefill_chunk(q_pf, P0, 0, pool, tables[1e7], SCALE, out=outs["pf"], stream=st)
        kvr.kv_ring_append_rope(ks2, vs2, pos_stage, None, tables[1e4], vs, stage, stream=st)
        kvr.swa_sink_prefill_chunk(q_ps, P0, 1, stage, ring, sinks, tables[1e4], SCALE, out=outs["ps"], stream=st)

    step(torch.cuda.current_stream())
    torch.cuda.synchronize()
    want = {n: _bits(t) for n, t in outs.items()}
    assert all(torch.count_nonzero(t) > 0 for t in outs.values())
    g = _capture(step)
    for t in outs.values():
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    for n, t in outs.items():
        assert torch.equal(_bits(t), want[n]), n


def test_pool_operations_replay_bit_for_bit(tables):
    syn = Synth(7201, dist="plain", device=DEV)
    hkv, bsz, vs = 2, 16, 0.707
    ends = [300, 77, 129]
    S = len(ends)
    pool = kvr.PagedLayout.contiguous(S, hkv, 512, block_size=bsz)
    fill_paged(pool, syn, list(range(S)), ends, tables[1e4], vs)
    ring = kvr.RingLayout.empty(S, hkv)
    seqs = torch.arange(S, dtype=torch.int32, device=DEV)
    end = torch.tensor(ends, dtype=torch.int64, device=DEV)
    last = end - 1
    snap = kvr.ring_snapshot_alloc(S, hkv)
    ring2 = kvr.RingLayout.empty(S, hkv)
    table0 = pool.block_table.clone()
    free = torch.full((pool.num_blocks,), -1, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
    lo = torch.zeros(S, dtype=torch.int32, device=DEV)
    q = syn.q(S, 8, hkv, seq=9)
    sinks = syn.sinks(8).to(DEV)
    out = torch.empty(S, 8, 128, dtype=torch.bfloat16, device=DEV)

    def step(st):
        pool.block_table.copy_(table0)
        cnt.zero_()
        lo.zero_()
        kvr.swa_sink_decode(q, last, seqs, pool, sinks, tables[1e4], SCALE, out=out, stream=st)
        kvr.kv_ring_gather_pages(pool, ring, seqs, seqs, end, stream=st)
        kvr.kv_ring_snapshot(ring, seqs, snap, stream=st)
        kvr.kv_ring_restore(ring2, seqs, snap, stream=st)
        kvr.kv_pages_release_window(pool.block_table, pool.num_blocks, bsz, seqs, end, free, cnt, lo=lo, stream=st)

    step(torch.cuda.current_stream())
    torch.cuda.synchronize()
    state = lambda: [_bits(out), _bits(ring.k), ring.slot_pos.clone(), _bits(ring2.v), pool.block_table.clone(),
                     free.clone(), cnt.clone(), lo.clone()]
    want = state()
    assert int(cnt.item()) > 0
    g = _capture(step)
    for t in (out, ring.k, ring2.v):
        t.zero_()
    ring.slot_pos.fill_(-1)
    free.fill_(-1)
    g.replay()
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    for a, b in zip(state(), want):
        assert torch.equal(a, b)
