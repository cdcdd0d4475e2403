"""GPU parity at the full workload sizes, in the launch configuration bench.py
times: sampled outputs against the fp64 oracle.

* Flash-shaped decode: batch 64, 64 q heads, windowed layer (8 KV heads) and
  full layer (4 KV heads) at context 32769 -- sampled sequences, all heads.
* Chunked prefill: 8192-token chunk on 122880 cached tokens -- sampled rows
  (first, last, window and tile boundaries), all heads, both layer kinds.
* Long-context decode: batch 16 at context 524289 -- sampled sequences.
* Pro-shaped decode: 128 sequences with contexts log-uniform up to ~1M, both
  head configurations -- the shortest, a median and the longest sequence.
* Draft verification: the decode batch checking 4 tokens per sequence
  through the varlen calls -- sampled sequences, all rows and heads.

Raw K/V are regenerated from the same seeded draws the bench used (never read
back from the CUDA path).
"""
import math
import os
import sys

import numpy as np
import pytest
import torch

import oracle

from kvr_cases import compare_rows

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

pytestmark = pytest.mark.gpu
SCALE = 1.0 / math.sqrt(192.0)


@pytest.fixture(scope="module")
def kvr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sinks_kv_ring_gb300 import build
    build.build()
    import sinks_kv_ring_gb300 as k
    k.device_status(reset=True)
    return k


def _pool_raw(syn, hkv, b, n, chunk=65536):
    """Raw K/V of positions 0..n-1 as bench._fill_pool drew them."""
    ks = [syn.k(min(chunk, n - lo), hkv, seq=b, start=lo) for lo in range(0, n, chunk)]
    vs = [syn.v(min(chunk, n - lo), hkv, seq=b, start=lo) for lo in range(0, n, chunk)]
    return torch.cat(ks), torch.cat(vs)


def _decode_check(kvr, work, seqs, label):
    import bench
    from sinks_kv_ring_gb300.synth import Synth
    stream = torch.cuda.current_stream()
    work.step(stream)
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    p = work.p
    syn_f = Synth(1001, layer=1, device="cuda")
    syn_s = Synth(1001, layer=0, device="cuda")
    sk = work.sinks.double().cpu().numpy()
    lo = max(0, p - 127)
    for b in seqs:
        kf, vf = _pool_raw(syn_f, work.hkv_full, b, p)
        kf = torch.cat([kf, work.k_full[b:b + 1]])
        vf = torch.cat([vf, work.v_full[b:b + 1]])
        want = oracle.attend_seq(work.q_full[b:b + 1], [p], kf, vf, 0, 1e7, work.vscale, SCALE, 0, None)
        compare_rows(work.out_full[b:b + 1], want, f"{label} full b={b}")
        ks = torch.cat([syn_s.k(p - lo, work.hkv_swa, seq=b, start=lo), work.k_swa[b:b + 1]])
        vs = torch.cat([syn_s.v(p - lo, work.hkv_swa, seq=b, start=lo), work.v_swa[b:b + 1]])
        want = oracle.attend_seq(work.q_swa[b:b + 1], [p], ks, vs, lo, 1e4, work.vscale, SCALE, 128, sk)
        compare_rows(work.out_swa[b:b + 1], want, f"{label} swa b={b}")


def test_flash_decode_full_size_sampled(kvr):
    import bench
    work = bench.DecodeWorkload(kvr, B=64, ctx=32768, seed=1001, swa_copies=1)
    _decode_check(kvr, work, [0, 17, 63], "flash decode")
    # the no-allocation variant on the same full-size batch
    out2 = kvr.full_attn_decode_noalloc(work.q_full, work.pos, work.seq, work.pool, work.t7, SCALE, work.max_ctx)
    torch.cuda.synchronize()
    assert torch.equal(out2, work.out_full)
    del work
    torch.cuda.empty_cache()


def test_draft_verification_full_size_sampled(kvr):
    # The bench's draft-verification step: batch 64, 4 tokens per sequence at
    # positions 32768..32771, both layer kinds, through the varlen calls.
    import bench
    from sinks_kv_ring_gb300.synth import Synth
    work = bench.DecodeWorkload(kvr, B=64, ctx=32768, seed=1001, swa_copies=1)
    m = bench.MtpStep(work, q_len=4)
    m.step(torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    p = work.p
    syn_f = Synth(1001, layer=1, device="cuda")
    syn_s = Synth(1001, layer=0, device="cuda")
    sk = work.sinks.double().cpu().numpy()
    lo = p - 127
    pos = np.arange(p, p + 4)
    for b in [0, 33, 63]:
        r = slice(4 * b, 4 * b + 4)
        kf, vf = _pool_raw(syn_f, work.hkv_full, b, p)
        kf, vf = torch.cat([kf, m.kf[r]]), torch.cat([vf, m.vf[r]])
        want = oracle.attend_seq(m.qf[r], pos, kf, vf, 0, 1e7, work.vscale, SCALE, 0, None)
        compare_rows(m.out_f[r], want, f"draft full b={b}")
        ks = torch.cat([syn_s.k(p - lo, work.hkv_swa, seq=b, start=lo), m.ks[r]])
        vs = torch.cat([syn_s.v(p - lo, work.hkv_swa, seq=b, start=lo), m.vs[r]])
        want = oracle.attend_seq(m.qs[r], pos, ks, vs, lo, 1e4, work.vscale, SCALE, 128, sk)
        compare_rows(m.out_s[r], want, f"draft swa b={b}")
    del m, work
    torch.cuda.empty_cache()


def test_long_context_decode_full_size_sampled(kvr):
    import bench
    work = bench.DecodeWorkload(kvr, B=16, ctx=524288, seed=1001, swa_copies=1)
    _decode_check(kvr, work, [0, 15], "long decode")
    del work
    torch.cuda.empty_cache()


def test_chunked_prefill_full_size_sampled(kvr):
    import bench
    from sinks_kv_ring_gb300.synth import Synth
    work = bench.PrefillWorkload(kvr, P0=122880, C=8192, seed=1002)
    work.step(torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    P0, C = work.P0, work.C
    rows = [0, 1, 126, 127, 128, 255, 256, 4095, 8190, 8191]
    sf, ss = Synth(1002, layer=1, device="cuda"), Synth(1002, layer=0, device="cuda")
    # full layer: keys 0 .. P0 + C - 1
    kf, vf = _pool_raw(sf, work.hkv_full, 0, P0)
    kf, vf = torch.cat([kf, work.kf]), torch.cat([vf, work.vf])
    want = oracle.attend_seq(work.qf[rows], np.array(rows) + P0, kf, vf, 0, 1e7, work.vscale, SCALE, 0, None)
    compare_rows(work.out_f[rows], want, "prefill full")
    # windowed layer: ring positions P0-127 .. P0-1 then the chunk
    lo = P0 - 127
    ks = torch.cat([ss.k(127, work.hkv_swa, seq=0, start=lo), work.ks])
    vs = torch.cat([ss.v(127, work.hkv_swa, seq=0, start=lo), work.vs])
    want = oracle.attend_seq(work.qs[rows], np.array(rows) + P0, ks, vs, lo, 1e4, work.vscale, SCALE, 128,
                             work.sinks.double().cpu().numpy())
    compare_rows(work.out_s[rows], want, "prefill swa")
    del work
    torch.cuda.empty_cache()


@pytest.mark.parametrize("hq,hkv_full", [(64, 4), (128, 8)])
def test_pro_shaped_contexts_decode_sampled(kvr, hq, hkv_full):
    # The Pro-shaped decode step's batch: 128 sequences with contexts
    # log-uniform over [1K, 1M] (seed 1004), one full layer (paged pool of all
    # 19.6M cached tokens) and one windowed layer (8 KV heads, ring 128 +
    # sink); 64 q / 4 KV heads as the workload states, and the Pro's own 128 q
    # / 8 KV heads.  Sampled: the shortest, a median and the longest sequence.
    from sinks_kv_ring_gb300.synth import Synth, ragged_contexts
    B, vs_, bsz = 128, 0.612, 64
    ctx = ragged_contexts(B, 1024, 1 << 20, 1004)
    max_ctx = max(ctx) + 1
    t4, t7 = kvr.rope_table(1e4, max_ctx), kvr.rope_table(1e7, max_ctx)
    mb = [(c + 1 + bsz - 1) // bsz for c in ctx]
    bt = torch.zeros(B, max(mb), dtype=torch.int32)
    off = 0
    for b, m in enumerate(mb):
        bt[b, :m] = torch.arange(off, off + m, dtype=torch.int32)
        off += m
    pool = kvr.PagedLayout(torch.empty(off, hkv_full, bsz, 192, dtype=torch.bfloat16, device="cuda"),
                           torch.empty(off, hkv_full, bsz, 128, dtype=torch.bfloat16, device="cuda"), bt.cuda())
    syn_f, syn_s = Synth(1004, layer=1, device="cuda"), Synth(1004, layer=0, device="cuda")
    import bench
    bench._fill_pool(kvr, pool, syn_f, range(B), ctx, t7, vs_)
    ring = kvr.RingLayout.empty(B, 8)
    for b, c in enumerate(ctx):
        lo = c - 127
        kvr.kv_ring_append_rope(syn_s.k(127, 8, seq=b, start=lo), syn_s.v(127, 8, seq=b, start=lo),
                                torch.arange(lo, c, device="cuda"), torch.full((127,), b, dtype=torch.int32,
                                                                              device="cuda"), t4, vs_, ring)
    pos = torch.tensor(ctx, dtype=torch.int64, device="cuda")
    seq = torch.arange(B, dtype=torch.int32, device="cuda")
    kn_f, vn_f = syn_f.k(B, hkv_full, seq=60_000), syn_f.v(B, hkv_full, seq=60_000)
    kn_s, vn_s = syn_s.k(B, 8, seq=60_000), syn_s.v(B, 8, seq=60_000)
    kvr.kv_ring_append_rope(kn_f, vn_f, pos, seq, t7, vs_, pool)
    kvr.kv_ring_append_rope(kn_s, vn_s, pos, seq, t4, vs_, ring)
    qf, qs = syn_f.q(B, hq, hkv_full, seq=50_000), syn_s.q(B, hq, 8, seq=50_000)
    sinks = syn_s.sinks(hq).cuda()
    scale = 1.0 / math.sqrt(192.0)
    of = kvr.full_attn_decode(qf, pos, seq, pool, t7, scale, max_ctx)
    osw = kvr.swa_sink_decode(qs, pos, seq, ring, sinks, t4, scale)
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    order = np.argsort(ctx)
    for b in (int(order[0]), int(order[B // 2]), int(order[-1])):
        p = ctx[b]
        kf, vf = _pool_raw(syn_f, hkv_full, b, p)
        kf, vf = torch.cat([kf, kn_f[b:b + 1]]), torch.cat([vf, vn_f[b:b + 1]])
        want = oracle.attend_seq(qf[b:b + 1], [p], kf, vf, 0, 1e7, vs_, scale, 0, None)
        compare_rows(of[b:b + 1], want, f"pro full b={b} ctx={p}")
        lo = p - 127
        ks = torch.cat([syn_s.k(127, 8, seq=b, start=lo), kn_s[b:b + 1]])
        vs = torch.cat([syn_s.v(127, 8, seq=b, start=lo), vn_s[b:b + 1]])
        want = oracle.attend_seq(qs[b:b + 1], [p], ks, vs, lo, 1e4, vs_, scale, 128, sinks.double().cpu().numpy())
        compare_rows(osw[b:b + 1], want, f"pro swa b={b}")
    del pool, ring
    torch.cuda.empty_cache()


def test_pro_stack_captured_graph_sampled(kvr):
    # The Pro-shaped decode step as the bench runs it: a layer stack (layer i
    # full iff i % 7 == 6) captured as one CUDA graph, each layer a KV write
    # then its attention, on the seed-1004 batch (128 sequences, contexts
    # log-uniform over [1K, 1M]).  14 layers: 12 windowed (a ring each) and 2
    # full that share one paged pool, as the bench's full layers share pools;
    # every layer has its own q, sinks, new-token K/V and output.  Two
    # replays are bit-equal, and every layer's shortest, median and longest
    # sequences match the oracle (all heads).
    from sinks_kv_ring_gb300.synth import Synth, ragged_contexts
    import bench
    B, hq, vs_, bsz, layers = 128, 64, 0.612, 64, 14
    kinds = ["full" if i % 7 == 6 else "swa" for i in range(layers)]
    ctx = ragged_contexts(B, 1024, 1 << 20, 1004)
    max_ctx = max(ctx) + 1
    t4, t7 = kvr.rope_table(1e4, max_ctx), kvr.rope_table(1e7, max_ctx)
    mb = [(c + 1 + bsz - 1) // bsz for c in ctx]
    bt = torch.zeros(B, max(mb), dtype=torch.int32)
    off = 0
    for b, m in enumerate(mb):
        bt[b, :m] = torch.arange(off, off + m, dtype=torch.int32)
        off += m
    pool = kvr.PagedLayout(torch.empty(off, 4, bsz, 192, dtype=torch.bfloat16, device="cuda"),
                           torch.empty(off, 4, bsz, 128, dtype=torch.bfloat16, device="cuda"), bt.cuda())
    syn_pool = Synth(1004, layer=100, device="cuda")
    bench._fill_pool(kvr, pool, syn_pool, range(B), ctx, t7, vs_)
    pos = torch.tensor(ctx, dtype=torch.int64, device="cuda")
    seq = torch.arange(B, dtype=torch.int32, device="cuda")
    L = []
    for i, kind in enumerate(kinds):
        syn = Synth(1004, layer=i, device="cuda")
        hkv = 4 if kind == "full" else 8
        d = {"kind": kind, "syn": syn, "hkv": hkv, "q": syn.q(B, hq, hkv, seq=50_000),
             "kn": syn.k(B, hkv, seq=60_000), "vn": syn.v(B, hkv, seq=60_000),
             "out": torch.empty(B, hq, 128, dtype=torch.bfloat16, device="cuda")}
        if kind == "swa":
            d["sinks"] = syn.sinks(hq).cuda()
            ring = kvr.RingLayout.empty(B, 8)
            for b, c in enumerate(ctx):
                lo = c - 127
                kvr.kv_ring_append_rope(syn.k(127, 8, seq=b, start=lo), syn.v(127, 8, seq=b, start=lo),
                                        torch.arange(lo, c, device="cuda"),
                                        torch.full((127,), b, dtype=torch.int32, device="cuda"), t4, vs_, ring)
            d["ring"] = ring
        L.append(d)
    ws = torch.empty(kvr.full_attn_decode_workspace_size(B, hq, 4, max_ctx), dtype=torch.uint8, device="cuda")

    def step(st):
        for d in L:
            if d["kind"] == "full":
                kvr.kv_ring_append_rope(d["kn"], d["vn"], pos, seq, t7, vs_, pool, stream=st)
                kvr.full_attn_decode(d["q"], pos, seq, pool, t7, SCALE, max_ctx, workspace=ws, out=d["out"],
                                     stream=st)
            else:
                kvr.kv_ring_append_rope(d["kn"], d["vn"], pos, seq, t4, vs_, d["ring"], stream=st)
                kvr.swa_sink_decode(d["q"], pos, seq, d["ring"], d["sinks"], t4, SCALE, out=d["out"], stream=st)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for d in L:
        d["out"].fill_(7.0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(torch.cuda.current_stream())
    g.replay()
    torch.cuda.synchronize()
    first = [d["out"].clone() for d in L]
    g.replay()
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    for i, d in enumerate(L):
        assert torch.equal(first[i], d["out"]), f"layer {i}: replays differ"
    order = np.argsort(ctx)
    sample = (int(order[0]), int(order[B // 2]), int(order[-1]))
    raw_pool = {b: _pool_raw(syn_pool, 4, b, ctx[b]) for b in sample}
    for i, d in enumerate(L):
        for b in sample:
            p = ctx[b]
            if d["kind"] == "full":
                kf, vf = raw_pool[b]
                kf, vf = torch.cat([kf, d["kn"][b:b + 1]]), torch.cat([vf, d["vn"][b:b + 1]])
                want = oracle.attend_seq(d["q"][b:b + 1], [p], kf, vf, 0, 1e7, vs_, SCALE, 0, None)
            else:
                lo = p - 127
                ks = torch.cat([d["syn"].k(127, 8, seq=b, start=lo), d["kn"][b:b + 1]])
                vv = torch.cat([d["syn"].v(127, 8, seq=b, start=lo), d["vn"][b:b + 1]])
                want = oracle.attend_seq(d["q"][b:b + 1], [p], ks, vv, lo, 1e4, vs_, SCALE, 128,
                                         d["sinks"].double().cpu().numpy())
            compare_rows(d["out"][b:b + 1], want, f"stack layer {i} ({d['kind']}) b={b} ctx={p}")
    del g, pool, L
    torch.cuda.empty_cache()


def test_zero_length_calls_are_no_ops(kvr):
    import sinks_kv_ring_gb300 as k
    t = k.rope_table(1e7, 64)
    pool = k.PagedLayout.contiguous(1, 4, 64)
    out = torch.full((0, 64, 128), 7, dtype=torch.bfloat16, device="cuda")
    k.full_attn_prefill_chunk(torch.empty(0, 64, 192, dtype=torch.bfloat16, device="cuda"), 10, 0, pool, t, SCALE,
                              out=out)
    ring = k.RingLayout.empty(1, 8)
    stage = k.LinearLayout.empty(1, 8)
    k.swa_sink_prefill_chunk(torch.empty(0, 64, 192, dtype=torch.bfloat16, device="cuda"), 10, 0, stage, ring,
                             torch.zeros(64, device="cuda"), k.rope_table(1e4, 64), SCALE, out=out)
    k.full_attn_decode(torch.empty(0, 64, 192, dtype=torch.bfloat16, device="cuda"),
                       torch.empty(0, dtype=torch.int64, device="cuda"), torch.empty(0, dtype=torch.int32, device="cuda"),
                       pool, t, SCALE, 64, out=torch.empty(0, 64, 128, dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    assert k.device_status() == 0
