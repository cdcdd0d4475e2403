"""GPU parity: every call of the C ABI against the fp64 oracle on the same
seeded inputs.  Bar: max |err| <= 2e-2 and relative RMS <= 1e-2 for bf16
outputs (fp32 accumulation); ring-slot tags and pass-through dims bit-exact."""
import math

import numpy as np
import pytest
import torch

import oracle
import sinks_kv_ring_gb300 as kvr
from sinks_kv_ring_gb300.synth import Synth

from kvr_cases import SCALE, compare, compare_rows, compare_rows_vec, fill_paged, fill_ring, raw_kv

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
    return {1e4: kvr.rope_table(1e4, 1 << 17), 1e7: kvr.rope_table(1e7, 1 << 17)}


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _ulp_close(a_bits, b_bits, max_ulp=1):
    a = a_bits.astype(np.int32)
    b = b_bits.astype(np.int32)
    # bf16 bit patterns with equal sign are ordered like integers
    same_sign = (a & 0x8000) == (b & 0x8000)
    d = np.abs(a - b)
    return same_sign & (d <= max_ulp) | (a == b)


# --------------------------------------------------------------------------- KV write

@pytest.mark.parametrize("kind", ["ring", "paged", "linear"])
def test_append_matches_oracle_store(kind, tables):
    syn = Synth(2001, dist="shifted", device=DEV)
    hkv, T = 4, 300
    k, v = raw_kv(syn, hkv, 0, 0, T)
    pos = torch.arange(1000, 1000 + T, dtype=torch.int64, device=DEV)
    seq = torch.full((T,), 1, dtype=torch.int32, device=DEV)
    vs = 0.707
    if kind == "ring":
        dst = kvr.RingLayout.empty(3, hkv)
        # the ring holds 128 slots: write the last 128 tokens only
        k, v, pos, seq = k[-128:].contiguous(), v[-128:].contiguous(), pos[-128:].contiguous(), seq[-128:].contiguous()
    elif kind == "paged":
        dst = kvr.PagedLayout.contiguous(3, hkv, 2048, block_size=64)
        perm = torch.randperm(dst.num_blocks, generator=torch.Generator().manual_seed(5)).to(torch.int32)
        dst.block_table.copy_(perm.reshape(dst.block_table.shape).to(DEV))
    else:
        dst = kvr.LinearLayout.empty(T, hkv)
    kvr.kv_ring_append_rope(k, v, pos, seq if kind != "linear" else None, tables[1e4], vs, dst)
    torch.cuda.synchronize()
    ko, vo = oracle.kv_store_bf16(k, v, pos.cpu().numpy(), 1e4, vs)
    n = k.shape[0]
    if kind == "ring":
        slots = (pos % 128).cpu()
        gk = dst.k[1][:, slots].permute(1, 0, 2)
        gv = dst.v[1][:, slots].permute(1, 0, 2)
        sp = dst.slot_pos.cpu().numpy()
        assert np.array_equal(sp[1][slots.numpy()], pos.cpu().numpy())          # tags bit-exact
        assert np.all(sp[0] == -1) and np.all(sp[2] == -1)
    elif kind == "paged":
        p = pos.cpu()
        bt = dst.block_table.cpu()
        blk = bt[1][p // 64]
        gk = dst.k[blk, :, p % 64]
        gv = dst.v[blk, :, p % 64]
    else:
        gk, gv = dst.k, dst.v
    gk, gv = _bits(gk), _bits(gv)
    assert gk.shape == (n, hkv, 192)
    assert np.array_equal(gk[..., 64:], ko[..., 64:])        # dims 64..191 bit copy
    assert np.all(_ulp_close(gk[..., :64], ko[..., :64]))     # fp32 rotation vs fp64, one rounding each
    assert np.all(_ulp_close(gv, vo))
    assert kvr.device_status() == 0


def test_append_flags_bad_positions(tables):
    hkv = 2
    ring = kvr.RingLayout.empty(2, hkv)
    k = torch.ones(3, hkv, 192, dtype=torch.bfloat16, device=DEV)
    v = torch.ones(3, hkv, 128, dtype=torch.bfloat16, device=DEV)
    pos = torch.tensor([5, -1, 1 << 17], dtype=torch.int64, device=DEV)
    seq = torch.tensor([0, 0, 0], dtype=torch.int32, device=DEV)
    kvr.kv_ring_append_rope(k, v, pos, seq, tables[1e4], 1.0, ring)
    assert kvr.device_status() & kvr.DEV_BAD_POS
    sp = ring.slot_pos.cpu()
    assert sp[0, 5] == 5 and int((sp != -1).sum()) == 1
    seq = torch.tensor([0, 7, 0], dtype=torch.int32, device=DEV)
    pos = torch.tensor([1, 2, 3], dtype=torch.int64, device=DEV)
    kvr.kv_ring_append_rope(k, v, pos, seq, tables[1e4], 1.0, ring)
    assert kvr.device_status() == kvr.DEV_BAD_SEQ


# --------------------------------------------------------------------------- SWA decode

def _swa_decode_case(B, hq, hkv, positions, dist, seed, tables, vscale=0.707):
    syn = Synth(seed, dist=dist, device=DEV)
    ring = kvr.RingLayout.empty(B + 1, hkv)
    seqs = list(range(1, B + 1))           # sequence ids 1..B (row 0 left empty)
    fill_ring(ring, syn, seqs, positions, tables[1e4], vscale)
    q = syn.q(B, hq, hkv, seq=999)
    sinks = syn.sinks(hq).to(DEV)
    pos = torch.tensor(positions, dtype=torch.int64, device=DEV)
    seq = torch.tensor(seqs, dtype=torch.int32, device=DEV)
    out = kvr.swa_sink_decode(q, pos, seq, ring, sinks, tables[1e4], SCALE)
    torch.cuda.synchronize()
    want = np.zeros((B, hq, 128))
    for b, (s, p) in enumerate(zip(seqs, positions)):
        lo = max(0, p - 127)
        k, v = raw_kv(syn, hkv, s, lo, p + 1)
        want[b] = oracle.attend_seq(q[b:b + 1], [p], k, v, lo, 1e4, vscale, SCALE, 128,
                                    sinks.double().cpu().numpy())[0]
    return out, want


@pytest.mark.parametrize("dist", ["shifted", "plain"])
def test_swa_decode_ragged_ring_fill(dist, tables):
    positions = [0, 1, 5, 126, 127, 128, 129, 300, 1000, 4095, 4096, 70000]
    out, want = _swa_decode_case(len(positions), 64, 8, positions, dist, 2101, tables)
    compare(out, want, "swa decode")
    compare_rows(out, want, "swa decode")
    assert kvr.device_status() == 0


@pytest.mark.parametrize("B,hq", [(240, 64), (240, 128), (64, 64), (70, 64)])
def test_swa_decode_many_units_per_cta(B, hq, tables):
    """A batch of 240 sequences puts 12-13 (sequence, KV head) units on every
    CTA, so the kernel's consumer groups run many units each and can drift
    apart; 64 and 70 sequences over 8 KV heads take the layout of two CTAs of
    two groups per SM (two units per CTA): every row against the oracle, and
    three calls bit-equal."""
    hkv = 8
    positions = [(b * 977) % 5000 for b in range(B)]  # includes p < 127 (partly filled rings)
    syn = Synth(2111 + hq, dist="plain", device=DEV)
    ring = kvr.RingLayout.empty(B, hkv)
    seqs = list(range(B))
    fill_ring(ring, syn, seqs, positions, tables[1e4], 0.707)
    q = syn.q(B, hq, hkv, seq=999)
    sinks = syn.sinks(hq).to(DEV)
    pos = torch.tensor(positions, dtype=torch.int64, device=DEV)
    seq = torch.tensor(seqs, dtype=torch.int32, device=DEV)
    outs = [kvr.swa_sink_decode(q, pos, seq, ring, sinks, tables[1e4], SCALE) for _ in range(3)]
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    want = np.zeros((B, hq, 128))
    sk = sinks.double().cpu().numpy()
    for b, p in enumerate(positions):
        lo = max(0, p - 127)
        k, v = raw_kv(syn, hkv, b, lo, p + 1)
        want[b] = oracle.attend_seq(q[b:b + 1], [p], k, v, lo, 1e4, 0.707, SCALE, 128, sk)[0]
    compare_rows_vec(outs[0], want, f"swa decode B={B} hq={hq}")


def test_swa_decode_group_sizes(tables):
    for hq, hkv in [(8, 2), (16, 16), (16, 1), (24, 8)]:
        out, want = _swa_decode_case(3, hq, hkv, [200, 17, 128], "plain", 2201 + hq, tables)
        compare_rows(out, want, f"swa decode hq={hq} hkv={hkv}")


def test_swa_decode_bad_sequence_is_zeroed_and_flagged(tables):
    syn = Synth(2301, device=DEV)
    ring = kvr.RingLayout.empty(2, 2)
    fill_ring(ring, syn, [0, 1], [50, 60], tables[1e4], 0.707)
    q = syn.q(2, 8, 2)
    out = kvr.swa_sink_decode(q, torch.tensor([50, 60], device=DEV), torch.tensor([0, 5], dtype=torch.int32, device=DEV),
                              ring, syn.sinks(8).to(DEV), tables[1e4], SCALE)
    assert kvr.device_status() == kvr.DEV_BAD_SEQ
    assert torch.all(out[1] == 0) and torch.all(torch.isfinite(out[0].float()))


# --------------------------------------------------------------------------- full decode

@pytest.mark.parametrize("bsz", [16, 64, 128])
def test_full_decode_split_boundaries(bsz, tables):
    hq, hkv = 64, 4
    ctx = [1, 2, 15, 16, 17, 63, 64, 65, 1000, 3001, 7000]
    B = len(ctx)
    syn = Synth(2401 + bsz, dist="shifted", device=DEV)
    max_ctx = 8192
    pool = kvr.PagedLayout.contiguous(B, hkv, max_ctx, block_size=bsz)
    perm = torch.randperm(pool.num_blocks, generator=torch.Generator().manual_seed(bsz)).to(torch.int32)
    pool.block_table.copy_(perm.reshape(pool.block_table.shape).to(DEV))
    fill_paged(pool, syn, list(range(B)), ctx, tables[1e7], 0.707)
    q = syn.q(B, hq, hkv, seq=77)
    pos = torch.tensor([c - 1 for c in ctx], dtype=torch.int64, device=DEV)
    seq = torch.arange(B, dtype=torch.int32, device=DEV)
    out = kvr.full_attn_decode(q, pos, seq, pool, tables[1e7], SCALE, max_ctx)
    torch.cuda.synchronize()
    want = np.zeros((B, hq, 128))
    for b, c in enumerate(ctx):
        k, v = raw_kv(syn, hkv, b, 0, c)
        want[b] = oracle.attend_seq(q[b:b + 1], [c - 1], k, v, 0, 1e7, 0.707, SCALE, 0, None)[0]
    compare(out, want, "full decode")
    compare_rows(out, want, "full decode")
    assert kvr.device_status() == 0


def _ragged_pool(syn, ctx, max_ctx, hkv, bsz, table, vs, seed):
    """A paged pool with blocks for each sequence's own context only (shuffled
    ids; entries past a context are -1), filled through the library."""
    mb = (max_ctx + bsz - 1) // bsz
    need = [(b, i) for b, c in enumerate(ctx) for i in range((c + bsz - 1) // bsz)]
    ids = np.random.default_rng(seed).permutation(len(need))
    tab = np.full((len(ctx), mb), -1, dtype=np.int32)
    for (b, i), blk in zip(need, ids):
        tab[b, i] = blk
    pool = kvr.PagedLayout(torch.zeros(len(need), hkv, bsz, 192, dtype=torch.bfloat16, device=DEV),
                           torch.zeros(len(need), hkv, bsz, 128, dtype=torch.bfloat16, device=DEV),
                           torch.from_numpy(tab).to(DEV))
    fill_paged(pool, syn, list(range(len(ctx))), ctx, table, vs)
    return pool


@pytest.mark.parametrize("case", ["one_long_sequence", "many_short_sequences", "ragged_past_the_split_cap"])
def test_full_decode_split_plans(case, tables):
    # The split count follows the batch size and the longest context: one
    # sequence at 131072 (dozens of splits, the merge folds them over eight
    # warps), 400 short sequences (one split each), 128 sequences of which four
    # are far longer than the rest (splits at the length cap).
    hq, hkv, bsz, vs = 64, 4, 64, 0.707
    rng = np.random.default_rng({"one_long_sequence": 1, "many_short_sequences": 2,
                                 "ragged_past_the_split_cap": 3}[case])
    if case == "one_long_sequence":
        ctx, max_ctx = [131072], 131072
    elif case == "many_short_sequences":
        ctx, max_ctx = [int(c) for c in rng.integers(1, 1025, 400)], 1024
    else:
        ctx = [int(c) for c in rng.integers(1, 2001, 128)]
        for b in (5, 60, 61, 127):
            ctx[b] = int(rng.integers(33000, 40001))
        max_ctx = 40000
    syn = Synth(2601 + len(ctx), dist="shifted", device=DEV)
    pool = _ragged_pool(syn, ctx, max_ctx, hkv, bsz, tables[1e7], vs, len(ctx))
    B = len(ctx)
    q = syn.q(B, hq, hkv, seq=88)
    pos = torch.tensor([c - 1 for c in ctx], dtype=torch.int64, device=DEV)
    seq = torch.arange(B, dtype=torch.int32, device=DEV)
    out = kvr.full_attn_decode(q, pos, seq, pool, tables[1e7], SCALE, max_ctx)
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    longest = sorted(range(B), key=lambda b: -ctx[b])[:4]
    sample = sorted(set(longest + [0, B - 1, B // 2]))
    want = np.stack([oracle.attend_seq(q[b:b + 1], [ctx[b] - 1], *raw_kv(syn, hkv, b, 0, ctx[b]), 0, 1e7, vs,
                                       SCALE, 0, None)[0] for b in sample])
    compare_rows(out[sample], want, f"full decode, {case}")


def test_full_decode_small_groups_and_reuse_of_workspace(tables):
    syn = Synth(2501, dist="plain", device=DEV)
    for hq, hkv in [(8, 2), (4, 4)]:
        ctx = [513, 9]
        pool = kvr.PagedLayout.contiguous(2, hkv, 1024, block_size=32)
        fill_paged(pool, syn, [0, 1], ctx, tables[1e7], 0.612)
        ws = torch.full((kvr.full_attn_decode_workspace_size(2, hq, hkv, 1024),), 255, dtype=torch.uint8, device=DEV)
        q = syn.q(2, hq, hkv, seq=5)
        pos = torch.tensor([512, 8], device=DEV)
        seq = torch.tensor([0, 1], dtype=torch.int32, device=DEV)
        for _ in range(2):  # stale workspace contents must not matter
            out = kvr.full_attn_decode(q, pos, seq, pool, tables[1e7], SCALE, 1024, workspace=ws)
            want = np.stack([oracle.attend_seq(q[b:b + 1], [c - 1], *raw_kv(syn, hkv, b, 0, c), 0, 1e7, 0.612,
                                               SCALE, 0, None)[0] for b, c in enumerate(ctx)])
            compare_rows(out, want, f"full decode hq={hq}")


def test_full_decode_rejects_small_workspace(tables):
    pool = kvr.PagedLayout.contiguous(1, 4, 256, block_size=64)
    q = torch.zeros(1, 64, 192, dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(kvr.KvrError) as e:
        kvr.full_attn_decode(q, torch.tensor([3], device=DEV), torch.tensor([0], dtype=torch.int32, device=DEV), pool,
                             tables[1e7], SCALE, 256, workspace=ws)
    assert e.value.code == -3


def test_full_decode_position_past_max_ctx_is_zeroed(tables):
    pool = kvr.PagedLayout.contiguous(2, 4, 256, block_size=64)
    syn = Synth(2601, device=DEV)
    fill_paged(pool, syn, [0, 1], [100, 200], tables[1e7], 0.7)
    q = syn.q(2, 64, 4)
    out = kvr.full_attn_decode(q, torch.tensor([99, 255], device=DEV), torch.tensor([0, 1], dtype=torch.int32, device=DEV),
                               pool, tables[1e7], SCALE, 200)
    assert kvr.device_status() == kvr.DEV_BAD_POS
    assert torch.all(out[1] == 0)
    want = oracle.attend_seq(q[0:1], [99], *raw_kv(syn, 4, 0, 0, 100), 0, 1e7, 0.7, SCALE, 0, None)[0]
    compare_rows(out[0], want)


# --------------------------------------------------------------------------- prefill

def _prefill_ref(syn, hkv, q, P0, window, sinks, theta, vscale):
    C = q.shape[0]
    lo = max(0, P0 - 127) if window else 0
    k, v = raw_kv(syn, hkv, 0, lo, P0 + C)
    return oracle.attend_seq(q, np.arange(P0, P0 + C), k, v, lo, theta, vscale, SCALE, window,
                             None if sinks is None else sinks.double().cpu().numpy())


def _run_full_prefill_chunks(syn, hq, hkv, chunks, tables, vscale, bsz=64):
    total = sum(chunks)
    pool = kvr.PagedLayout.contiguous(1, hkv, total, block_size=bsz)
    outs, P0 = [], 0
    for C in chunks:
        k, v = raw_kv(syn, hkv, 0, P0, P0 + C)
        kvr.kv_ring_append_rope(k, v, torch.arange(P0, P0 + C, device=DEV), torch.zeros(C, dtype=torch.int32, device=DEV),
                                tables[1e7], vscale, pool)
        q = syn.q(C, hq, hkv, seq=0, start=P0)
        outs.append(kvr.full_attn_prefill_chunk(q, P0, 0, pool, tables[1e7], SCALE))
        P0 += C
    return torch.cat(outs), pool


def _run_swa_prefill_chunks(syn, hq, hkv, chunks, tables, vscale, sinks):
    ring = kvr.RingLayout.empty(1, hkv)
    outs, P0 = [], 0
    for C in chunks:
        k, v = raw_kv(syn, hkv, 0, P0, P0 + C)
        stage = kvr.LinearLayout.empty(C, hkv)
        kvr.kv_ring_append_rope(k, v, torch.arange(P0, P0 + C, device=DEV), None, tables[1e4], vscale, stage)
        q = syn.q(C, hq, hkv, seq=0, start=P0)
        outs.append(kvr.swa_sink_prefill_chunk(q, P0, 0, stage, ring, sinks, tables[1e4], SCALE))
        t = min(C, 128)
        kvr.kv_ring_append_rope(k[-t:].contiguous(), v[-t:].contiguous(), torch.arange(P0 + C - t, P0 + C, device=DEV),
                                torch.zeros(t, dtype=torch.int32, device=DEV), tables[1e4], vscale, ring)
        P0 += C
    return torch.cat(outs), ring


@pytest.mark.parametrize("chunks", [[512], [128, 128, 128, 128], [200, 312], [1, 63, 448]])
def test_full_prefill_tiny_config_chunking(chunks, tables):
    # Tiny sanity workload: one sequence, 8 q heads, 2 KV heads, 512 tokens.
    syn = Synth(1000, dist="shifted", device=DEV)
    out, _ = _run_full_prefill_chunks(syn, 8, 2, chunks, tables, 0.707)
    qs = torch.cat([syn.q(C, 8, 2, seq=0, start=P0) for C, P0 in zip(chunks, np.cumsum([0] + chunks[:-1]))])
    want = _prefill_ref(syn, 2, qs, 0, 0, None, 1e7, 0.707)
    compare(out, want, "full prefill")
    compare_rows(out, want, "full prefill")


@pytest.mark.parametrize("chunks", [[512], [128, 128, 128, 128], [200, 312], [1, 63, 448]])
def test_swa_prefill_tiny_config_chunking(chunks, tables):
    syn = Synth(1000, dist="shifted", device=DEV)
    sinks = syn.sinks(8).to(DEV)
    out, _ = _run_swa_prefill_chunks(syn, 8, 2, chunks, tables, 0.707, sinks)
    qs = torch.cat([syn.q(C, 8, 2, seq=0, start=P0) for C, P0 in zip(chunks, np.cumsum([0] + chunks[:-1]))])
    want = _prefill_ref(syn, 2, qs, 0, 128, sinks, 1e4, 0.707)
    compare(out, want, "swa prefill")
    compare_rows(out, want, "swa prefill")


def test_tiny_config_prefill_then_16_decode_steps(tables):
    # Tiny sanity config end to end: prefill 512 on both layer kinds, then 16
    # decode steps at p = 512..527; each decode row equals the oracle, and the
    # decode at p equals what a prefill row at p gives.
    syn = Synth(1000, dist="shifted", device=DEV)
    hq, hkv = 8, 2
    sinks = syn.sinks(hq).to(DEV)
    _, pool = _run_full_prefill_chunks(syn, hq, hkv, [512], tables, 0.707)
    big_pool = kvr.PagedLayout.contiguous(1, hkv, 528, block_size=64)
    big_pool.k[:pool.num_blocks].copy_(pool.k)
    big_pool.v[:pool.num_blocks].copy_(pool.v)
    _, ring = _run_swa_prefill_chunks(syn, hq, hkv, [512], tables, 0.707, sinks)
    seq = torch.zeros(1, dtype=torch.int32, device=DEV)
    for p in range(512, 528):
        k, v = raw_kv(syn, hkv, 0, p, p + 1)
        pos = torch.tensor([p], device=DEV)
        kvr.kv_ring_append_rope(k, v, pos, seq, tables[1e7], 0.707, big_pool)
        kvr.kv_ring_append_rope(k, v, pos, seq, tables[1e4], 0.707, ring)
        q = syn.q(1, hq, hkv, seq=0, start=p)
        of = kvr.full_attn_decode(q, pos, seq, big_pool, tables[1e7], SCALE, 528)
        osw = kvr.swa_sink_decode(q, pos, seq, ring, sinks, tables[1e4], SCALE)
        kf, vf = raw_kv(syn, hkv, 0, 0, p + 1)
        compare_rows(of, oracle.attend_seq(q, [p], kf, vf, 0, 1e7, 0.707, SCALE, 0, None), f"full decode p={p}")
        compare_rows(osw, oracle.attend_seq(q, [p], kf[p - 127:], vf[p - 127:], p - 127, 1e4, 0.707, SCALE, 128,
                                            sinks.double().cpu().numpy()), f"swa decode p={p}")
        # decode at p agrees with a one-row prefill chunk at p
        opf = kvr.full_attn_prefill_chunk(q, p, 0, big_pool, tables[1e7], SCALE)
        compare_rows(of, opf.double().cpu().numpy(), f"full decode vs prefill p={p}")
        stage = kvr.LinearLayout.empty(1, hkv)
        kvr.kv_ring_append_rope(k, v, pos, None, tables[1e4], 0.707, stage)
        ring_before = kvr.RingLayout(ring.k.clone(), ring.v.clone(), ring.slot_pos.clone())
        ring_before.slot_pos[0, p % 128] = -1    # the chunk row supplies p itself
        ops = kvr.swa_sink_prefill_chunk(q, p, 0, stage, ring_before, sinks, tables[1e4], SCALE)
        compare_rows(osw, ops.double().cpu().numpy(), f"swa decode vs prefill p={p}")
    assert kvr.device_status() == 0


def test_swa_prefill_respects_stale_ring_slots(tables):
    # A ring slot whose tag does not match the position the window wants
    # (here: the ring was never filled) contributes nothing.
    syn = Synth(2701, dist="plain", device=DEV)
    hq, hkv = 16, 8
    sinks = syn.sinks(hq).to(DEV)
    ring = kvr.RingLayout.empty(1, hkv)
    C, P0 = 100, 1000
    k, v = raw_kv(syn, hkv, 0, P0, P0 + C)
    stage = kvr.LinearLayout.empty(C, hkv)
    kvr.kv_ring_append_rope(k, v, torch.arange(P0, P0 + C, device=DEV), None, tables[1e4], 0.7, stage)
    q = syn.q(C, hq, hkv, seq=3)
    out = kvr.swa_sink_prefill_chunk(q, P0, 0, stage, ring, sinks, tables[1e4], SCALE)
    # the oracle sees only the chunk's own keys
    want = oracle.attend_seq(q, np.arange(P0, P0 + C), k, v, P0, 1e4, 0.7, SCALE, 128, sinks.double().cpu().numpy())
    compare_rows(out, want, "swa prefill, empty ring")


@pytest.mark.parametrize("hq,hkv", [(64, 4), (24, 8), (6, 2)])
def test_full_prefill_with_context_and_groups(hq, hkv, tables):
    syn = Synth(2801 + hq, dist="plain", device=DEV)
    P0, C = 3000, 333
    pool = kvr.PagedLayout.contiguous(1, hkv, P0 + C, block_size=128)
    fill_paged(pool, syn, [0], [P0 + C], tables[1e7], 0.612)
    q = syn.q(C, hq, hkv, seq=0, start=P0)
    out = kvr.full_attn_prefill_chunk(q, P0, 0, pool, tables[1e7], SCALE)
    rows = [0, 1, 127, 128, 200, 331, 332]
    k, v = raw_kv(syn, hkv, 0, 0, P0 + C)
    want = oracle.attend_seq(q[rows], np.array(rows) + P0, k, v, 0, 1e7, 0.612, SCALE, 0, None)
    compare_rows(out[rows], want, "full prefill with context")


@pytest.mark.parametrize("bsz", [16, 48, 96, 192, 256])
def test_full_prefill_block_sizes(bsz, tables):
    # Page sizes that are not 128: the key tiles are assembled from several
    # pages (or part of one), with a shuffled block table.
    syn = Synth(2901 + bsz, dist="shifted", device=DEV)
    hq, hkv, P0, C = 32, 2, 1500, 300
    pool = kvr.PagedLayout.contiguous(1, hkv, P0 + C + bsz, block_size=bsz)
    perm = torch.randperm(pool.num_blocks, generator=torch.Generator().manual_seed(bsz)).to(torch.int32)
    pool.block_table.copy_(perm.reshape(pool.block_table.shape).to(DEV))
    fill_paged(pool, syn, [0], [P0 + C], tables[1e7], 0.707)
    q = syn.q(C, hq, hkv, seq=0, start=P0)
    out = kvr.full_attn_prefill_chunk(q, P0, 0, pool, tables[1e7], SCALE)
    rows = [0, 7, 8, 150, 255, 256, 299]
    k, v = raw_kv(syn, hkv, 0, 0, P0 + C)
    want = oracle.attend_seq(q[rows], np.array(rows) + P0, k, v, 0, 1e7, 0.707, SCALE, 0, None)
    compare_rows(out[rows], want, f"full prefill bsz={bsz}")
    assert kvr.device_status() == 0


def test_full_prefill_many_tiles_all_rows(tables):
    # Several CTAs along the chunk and a few hundred key tiles; every row checked.
    syn = Synth(3001, dist="plain", device=DEV)
    hq, hkv, P0, C = 16, 1, 9000, 200
    pool = kvr.PagedLayout.contiguous(1, hkv, P0 + C, block_size=64)
    fill_paged(pool, syn, [0], [P0 + C], tables[1e7], 0.612)
    q = syn.q(C, hq, hkv, seq=0, start=P0)
    out = kvr.full_attn_prefill_chunk(q, P0, 0, pool, tables[1e7], SCALE)
    k, v = raw_kv(syn, hkv, 0, 0, P0 + C)
    want = oracle.attend_seq(q, np.arange(P0, P0 + C), k, v, 0, 1e7, 0.612, SCALE, 0, None)
    compare(out, want, "full prefill many tiles")
    compare_rows(out, want, "full prefill many tiles")


# --------------------------------------------------------------------------- Pro-true head shapes

def test_pro_true_heads_decode_both_kinds(tables):
    # The pages' MiMo-V2.6-Pro: 128 query heads and 8 KV heads on both layer
    # kinds (gaudi-cookbook "MiMo-V2.6-Pro"); value scale 0.612.
    hq, hkv = 128, 8
    positions = [5, 127, 128, 3000]
    out, want = _swa_decode_case(len(positions), hq, hkv, positions, "shifted", 3101, tables, vscale=0.612)
    compare_rows(out, want, "pro swa decode")
    syn = Synth(3102, dist="plain", device=DEV)
    ctx = [1, 130, 2049]
    pool = kvr.PagedLayout.contiguous(len(ctx), hkv, 4096, block_size=64)
    fill_paged(pool, syn, list(range(len(ctx))), ctx, tables[1e7], 0.612)
    q = syn.q(len(ctx), hq, hkv, seq=9)
    out = kvr.full_attn_decode(q, torch.tensor([c - 1 for c in ctx], device=DEV),
                               torch.arange(len(ctx), dtype=torch.int32, device=DEV), pool, tables[1e7], SCALE, 4096)
    want = np.stack([oracle.attend_seq(q[b:b + 1], [c - 1], *raw_kv(syn, hkv, b, 0, c), 0, 1e7, 0.612, SCALE, 0,
                                       None)[0] for b, c in enumerate(ctx)])
    compare_rows(out, want, "pro full decode")


def test_pro_true_heads_prefill_both_kinds(tables):
    hq, hkv, P0, C = 128, 8, 700, 200
    syn = Synth(3103, dist="shifted", device=DEV)
    sinks = syn.sinks(hq).to(DEV)
    pool = kvr.PagedLayout.contiguous(1, hkv, P0 + C, block_size=64)
    fill_paged(pool, syn, [0], [P0 + C], tables[1e7], 0.612)
    q = syn.q(C, hq, hkv, seq=0, start=P0)
    out = kvr.full_attn_prefill_chunk(q, P0, 0, pool, tables[1e7], SCALE)
    rows = [0, 1, 100, 199]
    k, v = raw_kv(syn, hkv, 0, 0, P0 + C)
    want = oracle.attend_seq(q[rows], np.array(rows) + P0, k, v, 0, 1e7, 0.612, SCALE, 0, None)
    compare_rows(out[rows], want, "pro full prefill")
    ring = kvr.RingLayout.empty(1, hkv)
    fill_ring(ring, syn, [0], [P0 - 1], tables[1e4], 0.612)
    stage = kvr.LinearLayout.empty(C, hkv)
    kc, vc = raw_kv(syn, hkv, 0, P0, P0 + C)
    kvr.kv_ring_append_rope(kc, vc, torch.arange(P0, P0 + C, device=DEV), None, tables[1e4], 0.612, stage)
    out = kvr.swa_sink_prefill_chunk(q, P0, 0, stage, ring, sinks, tables[1e4], SCALE)
    lo = P0 - 127
    k, v = raw_kv(syn, hkv, 0, lo, P0 + C)
    want = oracle.attend_seq(q[rows], np.array(rows) + P0, k, v, lo, 1e4, 0.612, SCALE, 128,
                             sinks.double().cpu().numpy())
    compare_rows(out[rows], want, "pro swa prefill")


# --------------------------------------------------------------------------- ring snapshot / restore

def test_ring_snapshot_restore_roundtrip_and_decode(tables):
    # colibri "System One mode and prompt reuse": the rings are copied into a
    # snapshot and back; a decode after the restore equals the decode the
    # snapshot's state gives, bit for bit.
    syn = Synth(3201, dist="plain", device=DEV)
    hq, hkv = 64, 8
    ring = kvr.RingLayout.empty(4, hkv)
    fill_ring(ring, syn, [0, 1, 2, 3], [300, 90, 500, 127], tables[1e4], 0.707)
    seqs = torch.tensor([2, 0], dtype=torch.int32, device=DEV)
    snap = kvr.ring_snapshot_alloc(2, hkv)
    kvr.kv_ring_snapshot(ring, seqs, snap)
    q = syn.q(2, hq, hkv, seq=4)
    sinks = syn.sinks(hq).to(DEV)
    pos = torch.tensor([500, 300], device=DEV)
    before = kvr.swa_sink_decode(q, pos, seqs, ring, sinks, tables[1e4], SCALE).clone()
    ref = (ring.k.clone(), ring.v.clone(), ring.slot_pos.clone())
    # a later prompt overwrites the rings (here: 200 more positions on each)
    fill_ring(ring, syn, [0, 2], [700, 900], tables[1e4], 0.707)
    assert not torch.equal(ring.slot_pos, ref[2])
    kvr.kv_ring_restore(ring, seqs, snap)
    torch.cuda.synchronize()
    assert torch.equal(ring.k, ref[0]) and torch.equal(ring.v, ref[1]) and torch.equal(ring.slot_pos, ref[2])
    after = kvr.swa_sink_decode(q, pos, seqs, ring, sinks, tables[1e4], SCALE)
    assert torch.equal(after, before)
    bad = torch.tensor([9], dtype=torch.int32, device=DEV)
    kvr.kv_ring_snapshot(ring, bad, snap)
    assert kvr.device_status() == kvr.DEV_BAD_SEQ
