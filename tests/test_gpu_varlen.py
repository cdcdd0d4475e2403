"""GPU parity of the varlen calls (batches of chunks of different lengths)
against the fp64 oracle: multi-token-prediction draft verification (C = 1..4
per sequence), mixed prefill + decode batches, key-split boundaries, bad
device-side inputs, and replay in a CUDA graph with new lengths."""
import numpy as np
import pytest
import torch

import oracle
import sinks_kv_ring_gb300 as kvr
from sinks_kv_ring_gb300.synth import Synth

from kvr_cases import SCALE, compare, compare_rows, compare_rows_vec, fill_paged, fill_ring, raw_kv

pytestmark = pytest.mark.gpu

DEV = "cuda"
VS = 0.707


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
    return {1e4: kvr.rope_table(1e4, 1 << 16), 1e7: kvr.rope_table(1e7, 1 << 16)}


def _batch(syn, hq, hkv, seqs, P0s, Cs):
    """q rows of the batch in chunk order, plus the device plan arrays."""
    qs = [syn.q(C, hq, hkv, seq=s, start=P0) for s, P0, C in zip(seqs, P0s, Cs)]
    q = torch.cat(qs) if qs else torch.empty(0, hq, 192, dtype=torch.bfloat16, device=DEV)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(Cs)]), dtype=torch.int32, device=DEV)
    return (q.contiguous(), cu, torch.tensor(P0s, dtype=torch.int64, device=DEV),
            torch.tensor(seqs, dtype=torch.int32, device=DEV))


def _full_case(syn, hq, hkv, seqs, P0s, Cs, tables, bsz=64, num_seqs=None):
    """Pool holding positions 0..P0+C-1 of every chunk's sequence (the drafts
    appended), the batch, and the oracle rows."""
    ns = num_seqs or (max(seqs) + 1)
    max_ctx = max(P0 + C for P0, C in zip(P0s, Cs))
    pool = kvr.PagedLayout.contiguous(ns, hkv, max_ctx, block_size=bsz)
    fill_paged(pool, syn, seqs, [P0 + C for P0, C in zip(P0s, Cs)], tables[1e7], VS)
    q, cu, P0, sq = _batch(syn, hq, hkv, seqs, P0s, Cs)
    return pool, q, cu, P0, sq, max_ctx


def _full_want(syn, hkv, q, seqs, P0s, Cs):
    rows, r = [], 0
    for s, P0, C in zip(seqs, P0s, Cs):
        if C:
            k, v = raw_kv(syn, hkv, s, 0, P0 + C)
            rows.append(oracle.attend_seq(q[r:r + C], np.arange(P0, P0 + C), k, v, 0, 1e7, VS, SCALE, 0, None))
        r += C
    return np.concatenate(rows)


@pytest.mark.parametrize("hq,hkv", [(64, 4), (64, 8), (16, 4)])
def test_full_varlen_draft_verification(hq, hkv, tables):
    # Draft lengths 1..4; contexts around split boundaries (about 1024 keys
    # per split at this batch size), from a single key to ~5000.
    syn = Synth(3101 + hq + hkv, dist="shifted", device=DEV)
    seqs = [0, 1, 2, 3, 4, 5, 6]
    P0s = [0, 129, 1021, 2047, 2044, 4999, 300]
    Cs = [1, 2, 3, 2, 4, 4, 3]
    pool, q, cu, P0, sq, max_ctx = _full_case(syn, hq, hkv, seqs, P0s, Cs, tables)
    out = kvr.full_attn_prefill_varlen(q, cu, P0, sq, pool, tables[1e7], SCALE, max_ctx)
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    compare_rows(out, _full_want(syn, hkv, q, seqs, P0s, Cs), "full varlen draft")


def test_full_varlen_mixed_prefill_and_decode(tables):
    # One prefill chunk (several 256-row tiles, no key split) beside single
    # decode tokens and an empty chunk, in one call; the ragged chunk order
    # puts sequences out of order.
    syn = Synth(3201, dist="plain", device=DEV)
    hq, hkv = 32, 4
    seqs = [3, 0, 2, 1, 4]
    P0s = [700, 5000, 33, 2500, 0]
    Cs = [300, 1, 1, 0, 1]
    pool, q, cu, P0, sq, max_ctx = _full_case(syn, hq, hkv, seqs, P0s, Cs, tables, bsz=128)
    out = kvr.full_attn_prefill_varlen(q, cu, P0, sq, pool, tables[1e7], SCALE, max_ctx)
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    want = _full_want(syn, hkv, q, seqs, P0s, Cs)
    rows = list(range(0, 300, 37)) + [299, 300, 301, 302]
    compare_rows(out[rows], want[rows], "full varlen mixed")


def test_full_varlen_one_chunk_equals_prefill_chunk(tables):
    # A chunk too long to be split runs the same arithmetic as the single-chunk
    # call: bit-identical outputs.
    syn = Synth(3301, dist="plain", device=DEV)
    hq, hkv = 64, 4
    pool, q, cu, P0, sq, max_ctx = _full_case(syn, hq, hkv, [0], [3000], [333], tables)
    a = kvr.full_attn_prefill_varlen(q, cu, P0, sq, pool, tables[1e7], SCALE, max_ctx)
    b = kvr.full_attn_prefill_chunk(q, 3000, 0, pool, tables[1e7], SCALE)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_full_varlen_many_splits_large_batch(tables):
    # 64 draft chunks of 3 tokens with contexts up to ~20K: several splits per
    # chunk at the plan's split length; sampled chunks, all rows and heads.
    syn = Synth(3401, dist="shifted", device=DEV)
    hq, hkv = 64, 4
    rng = np.random.default_rng(3401)
    n = 64
    P0s = [int(x) for x in rng.integers(1, 20000, size=n)]
    seqs = list(range(n))
    Cs = [3] * n
    pool, q, cu, P0, sq, max_ctx = _full_case(syn, hq, hkv, seqs, P0s, Cs, tables, bsz=256)
    out = kvr.full_attn_prefill_varlen(q, cu, P0, sq, pool, tables[1e7], SCALE, max_ctx)
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    for s in (0, 17, 40, 63):
        k, v = raw_kv(syn, hkv, s, 0, P0s[s] + 3)
        want = oracle.attend_seq(q[3 * s:3 * s + 3], np.arange(P0s[s], P0s[s] + 3), k, v, 0, 1e7, VS, SCALE, 0, None)
        compare_rows(out[3 * s:3 * s + 3], want, f"full varlen chunk {s}")


# --------------------------------------------------------------------------- windowed

def _swa_case(syn, hq, hkv, seqs, P0s, Cs, tables, num_seqs=None):
    """Rings holding each sequence's window before its chunk, the chunk rows
    in a LINEAR staging layout (batch order), and the batch."""
    ns = num_seqs or (max(seqs) + 1)
    ring = kvr.RingLayout.empty(ns, hkv)
    fill_ring(ring, syn, [s for s, P0 in zip(seqs, P0s) if P0 > 0], [P0 - 1 for P0 in P0s if P0 > 0], tables[1e4], VS)
    ks, vs, ps = [], [], []
    for s, P0, C in zip(seqs, P0s, Cs):
        k, v = raw_kv(syn, hkv, s, P0, P0 + C)
        ks.append(k)
        vs.append(v)
        ps.append(torch.arange(P0, P0 + C, dtype=torch.int64, device=DEV))
    T = sum(Cs)
    stage = kvr.LinearLayout.empty(max(T, 1), hkv)
    if T:
        kvr.kv_ring_append_rope(torch.cat(ks).contiguous(), torch.cat(vs).contiguous(), torch.cat(ps), None,
                                tables[1e4], VS, stage)
    q, cu, P0, sq = _batch(syn, hq, hkv, seqs, P0s, Cs)
    return ring, stage, q, cu, P0, sq


def _swa_want(syn, hkv, q, seqs, P0s, Cs, sinks):
    rows, r = [], 0
    for s, P0, C in zip(seqs, P0s, Cs):
        if C:
            lo = max(0, P0 - 127)
            k, v = raw_kv(syn, hkv, s, lo, P0 + C)
            rows.append(oracle.attend_seq(q[r:r + C], np.arange(P0, P0 + C), k, v, lo, 1e4, VS, SCALE, 128,
                                          sinks.double().cpu().numpy()))
        r += C
    return np.concatenate(rows)


@pytest.mark.parametrize("dist", ["shifted", "plain"])
@pytest.mark.parametrize("hq,hkv", [(64, 8), (16, 8), (32, 2)])
def test_swa_varlen_draft_verification(dist, hq, hkv, tables):
    # Draft lengths 1..4 with the ring before the draft: empty ring, partly
    # filled, exactly full, wrapped several times.
    syn = Synth(3501 + hq + hkv, dist=dist, device=DEV)
    sinks = syn.sinks(hq).to(DEV)
    seqs = [0, 1, 2, 3, 4, 5]
    P0s = [0, 5, 127, 128, 1000, 4093]
    Cs = [4, 1, 2, 3, 4, 2]
    ring, stage, q, cu, P0, sq = _swa_case(syn, hq, hkv, seqs, P0s, Cs, tables)
    out = kvr.swa_sink_prefill_varlen(q, cu, P0, sq, stage, ring, sinks, tables[1e4], SCALE)
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    compare_rows(out, _swa_want(syn, hkv, q, seqs, P0s, Cs, sinks), "swa varlen draft")


def test_swa_varlen_mixed_and_equal_to_single_chunks(tables):
    # A long chunk beside decode tokens: the long chunk's rows agree with the
    # single-chunk call on the same ring and rows (a different kernel for
    # this group size: the band kernel, single-pass softmax) within the bar,
    # and both with the oracle; the single tokens (short-chunk kernel) match
    # the oracle.
    syn = Synth(3601, dist="shifted", device=DEV)
    hq, hkv = 64, 8
    sinks = syn.sinks(hq).to(DEV)
    seqs = [2, 0, 1]
    P0s = [900, 77, 3000]
    Cs = [513, 1, 1]
    ring, stage, q, cu, P0, sq = _swa_case(syn, hq, hkv, seqs, P0s, Cs, tables)
    out = kvr.swa_sink_prefill_varlen(q, cu, P0, sq, stage, ring, sinks, tables[1e4], SCALE)
    st = kvr.LinearLayout(stage.k[:513].contiguous(), stage.v[:513].contiguous())
    one = kvr.swa_sink_prefill_chunk(q[:513].contiguous(), 900, 2, st, ring, sinks, tables[1e4], SCALE)
    torch.cuda.synchronize()
    compare_rows(out[:513], one.double().cpu().numpy(), "swa varlen vs single chunk")
    want = _swa_want(syn, hkv, q, seqs, P0s, Cs, sinks)
    rows = list(range(0, 513, 41)) + [512, 513, 514]
    compare_rows(out[rows], want[rows], "swa varlen mixed")
    compare_rows(one[rows[:-2]], want[rows[:-2]], "swa single chunk")
    assert kvr.device_status() == 0


@pytest.mark.parametrize("hq,hkv,Cs", [(16, 4, [8, 3, 9, 16]), (8, 8, [16, 17, 1]), (64, 8, [2, 1]),
                                       (128, 8, [2, 3, 1])])
def test_swa_varlen_short_chunk_limits(hq, hkv, Cs, tables):
    # Short chunks up to 32 query rows and 16 tokens (4 heads x 8 tokens;
    # 1 head x 16; 16 heads x 2), chunks just past either limit (4 x 9,
    # 1 x 17, 16 x 3) that fall to the tiled kernel, and a batch of fewer
    # than 16 rows.
    syn = Synth(3551 + hq + len(Cs), dist="plain", device=DEV)
    sinks = syn.sinks(hq).to(DEV)
    seqs = list(range(len(Cs)))
    P0s = [3000 + 77 * s for s in seqs]
    ring, stage, q, cu, P0, sq = _swa_case(syn, hq, hkv, seqs, P0s, Cs, tables)
    out = kvr.swa_sink_prefill_varlen(q, cu, P0, sq, stage, ring, sinks, tables[1e4], SCALE)
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    compare_rows(out, _swa_want(syn, hkv, q, seqs, P0s, Cs, sinks), "swa varlen short chunks")


def test_varlen_plan_more_than_1024_chunks(tables):
    # 2500 chunks (the plan scans 1024 at a time with a carried prefix): a
    # mix of single tokens, drafts of 2-3 tokens and empty chunks over 40
    # sequences; every 97th chunk and the last ones checked, both kinds.
    syn = Synth(3901, dist="plain", device=DEV)
    hq, hkv_f, hkv_s = 16, 4, 8
    rng = np.random.default_rng(3901)
    n, ns = 2500, 40
    Cs = [int(c) for c in rng.choice([0, 1, 1, 2, 3], size=n)]
    seqs = [int(x) for x in rng.integers(0, ns, size=n)]
    P0s = [int(x) for x in rng.integers(0, 3000, size=n)]
    T = sum(Cs)
    # full layer: every sequence's pool holds positions 0..2999 + 3 (drafts
    # of different chunks of one sequence read the same pool rows)
    pool = kvr.PagedLayout.contiguous(ns, hkv_f, 3003, block_size=128)
    fill_paged(pool, syn, list(range(ns)), [3003] * ns, tables[1e7], VS)
    q, cu, P0, sq = _batch(syn, hq, hkv_f, seqs, P0s, Cs)
    out = kvr.full_attn_prefill_varlen(q, cu, P0, sq, pool, tables[1e7], SCALE, 3003)
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    starts = np.concatenate([[0], np.cumsum(Cs)])
    pick = [i for i in range(0, n, 97) if Cs[i]] + [i for i in range(n - 5, n) if Cs[i]]
    for i in pick:
        k, v = raw_kv(syn, hkv_f, seqs[i], 0, P0s[i] + Cs[i])
        r = slice(int(starts[i]), int(starts[i + 1]))
        want = oracle.attend_seq(q[r], np.arange(P0s[i], P0s[i] + Cs[i]), k, v, 0, 1e7, VS, SCALE, 0, None)
        compare_rows(out[r], want, f"full chunk {i}")
    # windowed layer: one ring per sequence holding positions 2872..2999;
    # every chunk verifies its tokens at 3000.. (chunks of one sequence share
    # that ring state and read their own staged rows)
    sinks = syn.sinks(hq).to(DEV)
    P0w = [3000] * n
    ring = kvr.RingLayout.empty(ns, hkv_s)
    fill_ring(ring, syn, list(range(ns)), [2999] * ns, tables[1e4], VS)
    ks, vs, ps = [], [], []
    for s_, C in zip(seqs, Cs):
        k, v = raw_kv(syn, hkv_s, s_, 3000, 3000 + C)
        ks.append(k)
        vs.append(v)
        ps.append(torch.arange(3000, 3000 + C, dtype=torch.int64, device=DEV))
    stage = kvr.LinearLayout.empty(T, hkv_s)
    kvr.kv_ring_append_rope(torch.cat(ks).contiguous(), torch.cat(vs).contiguous(), torch.cat(ps), None, tables[1e4],
                            VS, stage)
    qw, cuw, P0wt, sqw = _batch(syn, hq, hkv_s, seqs, P0w, Cs)
    outw = kvr.swa_sink_prefill_varlen(qw, cuw, P0wt, sqw, stage, ring, sinks, tables[1e4], SCALE)
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    for i in pick:
        k, v = raw_kv(syn, hkv_s, seqs[i], 2873, 3000 + Cs[i])
        r = slice(int(starts[i]), int(starts[i + 1]))
        want = oracle.attend_seq(qw[r], np.arange(3000, 3000 + Cs[i]), k, v, 2873, 1e4, VS, SCALE, 128,
                                 sinks.double().cpu().numpy())
        compare_rows(outw[r], want, f"swa chunk {i}")


@pytest.mark.parametrize("hq,hkv", [(64, 8), (128, 8), (64, 4)])
def test_swa_varlen_long_chunks(hq, hkv, tables):
    # Long windowed chunks beside decode tokens and drafts with 8 or 16 q
    # heads per KV head (tiles of 128 query rows, one key band each): chunk
    # lengths that are not whole tiles, chunks near position 0 and deep in
    # their sequence, a chunk of 2048 rows; every row against the oracle.
    syn = Synth(3801 + hq + hkv, dist="plain", device=DEV)
    sinks = syn.sinks(hq).to(DEV)
    seqs = [0, 1, 2, 3, 4, 5, 6]
    P0s = [0, 1000, 300, 60, 4000, 129, 2000]
    Cs = [300, 1, 517, 130, 3, 2048, 64]
    ring, stage, q, cu, P0, sq = _swa_case(syn, hq, hkv, seqs, P0s, Cs, tables)
    out = kvr.swa_sink_prefill_varlen(q, cu, P0, sq, stage, ring, sinks, tables[1e4], SCALE)
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    want = _swa_want(syn, hkv, q, seqs, P0s, Cs, sinks)
    compare(out, want, "swa varlen long chunks")
    compare_rows_vec(out, want, "swa varlen long chunks")
    # the same call again gives the same bits (tiles of different chunks in
    # one CTA, tiles that reach before their chunk among others)
    again = kvr.swa_sink_prefill_varlen(q, cu, P0, sq, stage, ring, sinks, tables[1e4], SCALE)
    assert torch.equal(again, out)
    # a long chunk with a bad sequence id: its rows are zeros, BAD_SEQ, the
    # others unchanged
    sq_bad = sq.clone()
    sq_bad[2] = ring.num_seqs
    bad = kvr.swa_sink_prefill_varlen(q, cu, P0, sq_bad, stage, ring, sinks, tables[1e4], SCALE)
    torch.cuda.synchronize()
    assert kvr.device_status() == kvr.DEV_BAD_SEQ
    r0, r1 = sum(Cs[:2]), sum(Cs[:3])
    assert torch.count_nonzero(bad[r0:r1]) == 0
    assert torch.equal(bad[:r0], out[:r0]) and torch.equal(bad[r1:], out[r1:])


def test_swa_varlen_many_long_chunks(tables):
    # 300 chunks of 5..80 rows (none short enough for the short-chunk kernel
    # at 8 q heads per KV head) over 40 sequences, all at 3000 on rings that
    # hold 2872..2999: the tile records come from a long chunk search, most
    # chunks end in a partial tile; every 13th chunk and the last ones
    # checked row by row.
    syn = Synth(3991, dist="plain", device=DEV)
    hq, hkv = 64, 8
    rng = np.random.default_rng(3991)
    n, ns = 300, 40
    Cs = [int(c) for c in rng.integers(5, 81, size=n)]
    seqs = [int(x) for x in rng.integers(0, ns, size=n)]
    T = sum(Cs)
    sinks = syn.sinks(hq).to(DEV)
    ring = kvr.RingLayout.empty(ns, hkv)
    fill_ring(ring, syn, list(range(ns)), [2999] * ns, tables[1e4], VS)
    ks, vs, ps = [], [], []
    for s_, C in zip(seqs, Cs):
        k, v = raw_kv(syn, hkv, s_, 3000, 3000 + C)
        ks.append(k)
        vs.append(v)
        ps.append(torch.arange(3000, 3000 + C, dtype=torch.int64, device=DEV))
    stage = kvr.LinearLayout.empty(T, hkv)
    kvr.kv_ring_append_rope(torch.cat(ks).contiguous(), torch.cat(vs).contiguous(), torch.cat(ps), None, tables[1e4],
                            VS, stage)
    q, cu, P0, sq = _batch(syn, hq, hkv, seqs, [3000] * n, Cs)
    out = kvr.swa_sink_prefill_varlen(q, cu, P0, sq, stage, ring, sinks, tables[1e4], SCALE)
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    starts = np.concatenate([[0], np.cumsum(Cs)])
    for i in list(range(0, n, 13)) + [n - 2, n - 1]:
        k, v = raw_kv(syn, hkv, seqs[i], 2873, 3000 + Cs[i])
        r = slice(int(starts[i]), int(starts[i + 1]))
        want = oracle.attend_seq(q[r], np.arange(3000, 3000 + Cs[i]), k, v, 2873, 1e4, VS, SCALE, 128,
                                 sinks.double().cpu().numpy())
        compare_rows_vec(out[r], want, f"swa chunk {i}")


@pytest.mark.parametrize("hq,hkv", [(6, 2), (24, 2)])
def test_swa_prefill_odd_group_sizes(hq, hkv, tables):
    # Group sizes that do not divide the 256-row tiles (3 and 12 query heads
    # per KV head): a single long chunk on a wrapped ring, and a varlen batch
    # of short and long chunks.
    syn = Synth(3951 + hq, dist="plain", device=DEV)
    sinks = syn.sinks(hq).to(DEV)
    P0, C = 1000, 300
    ring, stage, q, cu, P0t, sq = _swa_case(syn, hq, hkv, [0], [P0], [C], tables)
    out = kvr.swa_sink_prefill_chunk(q, P0, 0, stage, ring, sinks, tables[1e4], SCALE)
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    compare_rows(out, _swa_want(syn, hkv, q, [0], [P0], [C], sinks), f"swa chunk G={hq // hkv}")
    seqs, P0s, Cs = [0, 1, 2, 3], [500, 77, 2000, 129], [3, 1, 150, 10]
    ring, stage, q, cu, P0t, sq = _swa_case(syn, hq, hkv, seqs, P0s, Cs, tables)
    out = kvr.swa_sink_prefill_varlen(q, cu, P0t, sq, stage, ring, sinks, tables[1e4], SCALE)
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    compare_rows(out, _swa_want(syn, hkv, q, seqs, P0s, Cs, sinks), f"swa varlen G={hq // hkv}")


# --------------------------------------------------------------------------- bad inputs, graphs

def test_varlen_bad_device_inputs_are_flagged(tables):
    syn = Synth(3701, dist="plain", device=DEV)
    hq, hkv = 16, 4
    seqs, P0s, Cs = [0, 1, 0, 1], [100, 200, 50, 60], [2, 3, 1, 2]
    pool, q, cu, P0, sq, max_ctx = _full_case(syn, hq, hkv, seqs, P0s, Cs, tables)
    good = kvr.full_attn_prefill_varlen(q, cu, P0, sq, pool, tables[1e7], SCALE, max_ctx)
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    # chunk 1: sequence id outside the pool -> zeros, BAD_SEQ
    sq_bad = sq.clone()
    sq_bad[1] = 9
    out = kvr.full_attn_prefill_varlen(q, cu, P0, sq_bad, pool, tables[1e7], SCALE, max_ctx)
    torch.cuda.synchronize()
    assert kvr.device_status() == kvr.DEV_BAD_SEQ
    assert torch.count_nonzero(out[2:5]) == 0
    assert torch.equal(out[:2], good[:2]) and torch.equal(out[5:], good[5:])
    # chunk 2: P0 + C past max_ctx -> zeros, BAD_POS
    P0_bad = P0.clone()
    P0_bad[2] = max_ctx
    out = kvr.full_attn_prefill_varlen(q, cu, P0_bad, sq, pool, tables[1e7], SCALE, max_ctx)
    torch.cuda.synchronize()
    assert kvr.device_status() == kvr.DEV_BAD_POS
    assert torch.count_nonzero(out[5:6]) == 0
    assert torch.equal(out[:5], good[:5]) and torch.equal(out[6:], good[6:])
    # chunk 1's rows end past T -> skipped (rows untouched), BAD_ROWS
    cu_bad = cu.clone()
    cu_bad[2] = 100
    out = torch.full_like(good, 3.0)
    kvr.full_attn_prefill_varlen(q, cu_bad, P0, sq, pool, tables[1e7], SCALE, max_ctx, out=out)
    torch.cuda.synchronize()
    assert kvr.device_status() & kvr.DEV_BAD_ROWS
    assert torch.equal(out[:2], good[:2]) and torch.equal(out[6:], good[6:])
    assert torch.all(out[2:6] == 3.0)
    # the windowed call: bad sequence id -> zeros, BAD_SEQ
    sinks = syn.sinks(hq).to(DEV)
    ring, stage, q2, cu2, P02, sq2 = _swa_case(syn, hq, hkv, seqs, P0s, Cs, tables)
    sq2[0] = -1
    out = kvr.swa_sink_prefill_varlen(q2, cu2, P02, sq2, stage, ring, sinks, tables[1e4], SCALE)
    torch.cuda.synchronize()
    assert kvr.device_status() == kvr.DEV_BAD_SEQ
    assert torch.count_nonzero(out[:2]) == 0 and torch.count_nonzero(out[2:]) > 0


def test_varlen_calls_replay_in_a_cuda_graph_with_new_lengths(tables):
    # The plan is built on the device: a captured call replays with other
    # positions / lengths written into the same device arrays.
    syn = Synth(3801, dist="plain", device=DEV)
    hq, hkv = 64, 4
    seqs, P0s, Cs = [0, 1, 2], [1500, 40, 3000], [3, 3, 3]
    pool, q, cu, P0, sq, max_ctx = _full_case(syn, hq, hkv, seqs, P0s, Cs, tables)
    ws = torch.empty(kvr.full_attn_prefill_varlen_workspace_size(3, 9, hq, hkv, max_ctx), dtype=torch.uint8,
                     device=DEV)
    out = torch.empty(9, hq, 128, dtype=torch.bfloat16, device=DEV)
    kvr.full_attn_prefill_varlen(q, cu, P0, sq, pool, tables[1e7], SCALE, max_ctx, workspace=ws, out=out)
    torch.cuda.synchronize()
    first = out.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            kvr.full_attn_prefill_varlen(q, cu, P0, sq, pool, tables[1e7], SCALE, max_ctx, workspace=ws, out=out,
                                         stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, first)
    # new lengths: chunk 0 verifies 2 tokens at 1000, chunk 1 one token, chunk 2 six
    P0.copy_(torch.tensor([1000, 40, 2990], device=DEV))
    cu.copy_(torch.tensor([0, 2, 3, 9], dtype=torch.int32, device=DEV))
    g.replay()
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    want = _full_want(syn, hkv, q, seqs, [1000, 40, 2990], [2, 1, 6])
    compare_rows(out, want, "graph replay, new lengths")
