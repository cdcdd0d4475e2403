"""GPU parity for a windowed layer kept in pages: windowed decode over a
PAGED layout against the fp64 oracle; out-of-window release and the
ring-from-pages gather bit-exact against oracle/pages.py.

Xiaomi "Full-Pipeline Inference Optimization for MiMo-V2.5 Series", section
2.1 (the SWA pool kept at window size by releasing out-of-window KV);
gaudi-cookbook "Windowed KV groups" (paged sliding-window groups whose
out-of-window blocks are freed); colibri "System One mode and prompt reuse"
(slot p mod 128, slot tags)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import pages as opages
import sinks_kv_ring_gb300 as kvr
from sinks_kv_ring_gb300.synth import Synth

from kvr_cases import SCALE, compare, compare_rows, raw_kv

pytestmark = pytest.mark.gpu

DEV = "cuda"
NAN_BITS = -1  # int16 0xFFFF: a bf16 NaN, planted where nothing may be read


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
    return {1e4: kvr.rope_table(1e4, 1 << 17)}


def _nan_pool(nblk, hkv, bsz, table):
    k = torch.full((nblk, hkv, bsz, 192), NAN_BITS, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    v = torch.full((nblk, hkv, bsz, 128), NAN_BITS, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    return kvr.PagedLayout(k, v, table)


def _append_range(pool, syn, s, lo, hi, table, vscale):
    if hi <= lo:
        return
    k, v = raw_kv(syn, pool.num_kv_heads, s, lo, hi)
    pos = torch.arange(lo, hi, dtype=torch.int64, device=DEV)
    sq = torch.full((hi - lo,), s, dtype=torch.int32, device=DEV)
    kvr.kv_ring_append_rope(k, v, pos, sq, table, vscale, pool)


def _window_pool(positions, hkv, bsz, seed):
    """A paged windowed pool holding, for sequence b+1, only the blocks that
    cover positions max(0, p-127)..p (in shuffled order); every other table
    entry is -1 and every unwritten row a NaN."""
    B = len(positions)
    mb = max(positions) // bsz + 1
    need = [(b + 1, bi) for b, p in enumerate(positions) for bi in range(max(0, p - 127) // bsz, p // bsz + 1)]
    nblk = len(need) + 3
    ids = np.random.default_rng(seed).permutation(nblk)
    tab = np.full((B + 1, mb), -1, dtype=np.int32)
    for (s, bi), i in zip(need, ids):
        tab[s, bi] = i
    return _nan_pool(nblk, hkv, bsz, torch.from_numpy(tab).to(DEV))


def _oracle_swa(q, syn, hkv, seqs, positions, sinks, vscale):
    want = np.zeros((len(positions), q.shape[1], 128))
    for b, (s, p) in enumerate(zip(seqs, positions)):
        lo = max(0, p - 127)
        k, v = raw_kv(syn, hkv, s, lo, p + 1)
        want[b] = oracle.attend_seq(q[b:b + 1], [p], k, v, lo, 1e4, vscale, SCALE, 128,
                                    sinks.double().cpu().numpy())[0]
    return want


# --------------------------------------------------------------------------- windowed decode over pages

@pytest.mark.parametrize("dist", ["shifted", "plain"])
@pytest.mark.parametrize("bsz", [16, 32, 64, 128, 256])
def test_swa_decode_paged_matches_oracle(dist, bsz, tables):
    positions = [0, 1, 5, 15, 16, 126, 127, 128, 129, 143, 144, 300, 1000, 4095, 4096, 70000]
    hq, hkv, vs = 64, 8, 0.707
    syn = Synth(6101 + bsz, dist=dist, device=DEV)
    pool = _window_pool(positions, hkv, bsz, 61 + bsz)
    seqs = list(range(1, len(positions) + 1))
    for s, p in zip(seqs, positions):
        _append_range(pool, syn, s, max(0, p - 127), p + 1, tables[1e4], vs)
    q = syn.q(len(positions), hq, hkv, seq=999)
    sinks = syn.sinks(hq).to(DEV)
    pos = torch.tensor(positions, dtype=torch.int64, device=DEV)
    out = kvr.swa_sink_decode(q, pos, torch.tensor(seqs, dtype=torch.int32, device=DEV), pool, sinks,
                              tables[1e4], SCALE)
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    want = _oracle_swa(q, syn, hkv, seqs, positions, sinks, vs)
    compare(out, want, "paged swa decode")
    compare_rows(out, want, "paged swa decode")


@pytest.mark.parametrize("bsz", [16, 64])
@pytest.mark.parametrize("hq", [64, 128])
@pytest.mark.parametrize("B", [64, 200])
def test_swa_decode_paged_many_items_per_cta(bsz, hq, B, tables):
    """More (sequence, KV head) items than CTAs: at 8 q heads per KV head
    each CTA streams the subtiles of its items through its ring of eight
    places (at B = 200 five or more windows, every place reused many times,
    its barriers' parities alternating; at B = 64 one or two, the first
    prefetched before the wait on the kernel ahead), at 16 through the split
    kernel's window mode (the next item's ids carried, its window
    prefetched); positions mixed: short sequences, windows on and off 16-key
    boundaries.  Two calls must agree bit for bit, and every row must match
    the oracle."""
    rng = np.random.default_rng(6401 + bsz + B)
    positions = [int(x) for x in rng.integers(0, 5000, size=B)]
    positions[:6] = [0, 5, 127, 128, 143, 144]
    hkv, vs = 8, 0.707
    syn = Synth(6501 + bsz, dist="shifted", device=DEV)
    pool = _window_pool(positions, hkv, bsz, 71 + bsz)
    seqs = list(range(1, B + 1))
    for s, p in zip(seqs, positions):
        _append_range(pool, syn, s, max(0, p - 127), p + 1, tables[1e4], vs)
    q = syn.q(B, hq, hkv, seq=77)
    sinks = syn.sinks(hq).to(DEV)
    pos = torch.tensor(positions, dtype=torch.int64, device=DEV)
    sq = torch.tensor(seqs, dtype=torch.int32, device=DEV)
    out1 = kvr.swa_sink_decode(q, pos, sq, pool, sinks, tables[1e4], SCALE).clone()
    out2 = kvr.swa_sink_decode(q, pos, sq, pool, sinks, tables[1e4], SCALE)
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    assert torch.equal(out1, out2)
    want = _oracle_swa(q, syn, hkv, seqs, positions, sinks, vs)
    compare(out1, want, "paged swa decode, many items per CTA")
    compare_rows(out1, want, "paged swa decode, many items per CTA")


def test_swa_decode_paged_group_sizes(tables):
    positions = [200, 17, 128, 3000]
    for hq, hkv in [(8, 2), (16, 16), (16, 1), (24, 8), (128, 8)]:
        syn = Synth(6201 + hq + hkv, dist="plain", device=DEV)
        pool = _window_pool(positions, hkv, 32, hq)
        seqs = list(range(1, len(positions) + 1))
        for s, p in zip(seqs, positions):
            _append_range(pool, syn, s, max(0, p - 127), p + 1, tables[1e4], 0.612)
        q = syn.q(len(positions), hq, hkv, seq=5)
        sinks = syn.sinks(hq).to(DEV)
        out = kvr.swa_sink_decode(q, torch.tensor(positions, device=DEV), torch.tensor(seqs, dtype=torch.int32,
                                  device=DEV), pool, sinks, tables[1e4], SCALE)
        want = _oracle_swa(q, syn, hkv, seqs, positions, sinks, 0.612)
        compare_rows(out, want, f"paged swa decode hq={hq} hkv={hkv}")
    assert kvr.device_status() == 0


def test_swa_decode_paged_bad_inputs_are_zeroed_and_flagged(tables):
    syn = Synth(6301, device=DEV)
    pool = _window_pool([50, 60, 70], 2, 16, 3)
    for s, p in zip([1, 2, 3], [50, 60, 70]):
        _append_range(pool, syn, s, 0, p + 1, tables[1e4], 0.707)
    q = syn.q(4, 8, 2)
    sinks = syn.sinks(8).to(DEV)
    # row 1: sequence id outside the table; row 2: position past the table
    # (max_blocks * block_size = 80); row 3: its block entry is -1
    pool.block_table[3, 70 // 16] = -1
    pos = torch.tensor([50, 60, 80, 70], device=DEV)
    seq = torch.tensor([1, 9, 2, 3], dtype=torch.int32, device=DEV)
    out = kvr.swa_sink_decode(q, pos, seq, pool, sinks, tables[1e4], SCALE)
    st = kvr.device_status()
    assert st == kvr.DEV_BAD_SEQ | kvr.DEV_BAD_POS | kvr.DEV_BAD_BLOCK, st
    assert torch.all(out[1] == 0) and torch.all(out[2] == 0)
    assert torch.all(torch.isfinite(out[0].float())) and torch.all(torch.isfinite(out[3].float()))


# --------------------------------------------------------------------------- out-of-window release

def _release_gpu(table_np, nblk, bsz, seqs, nxt, window, lo, free_np, count, cap_override=None):
    tab = torch.from_numpy(table_np.copy()).to(DEV)
    free = torch.from_numpy(free_np.copy()).to(DEV)
    if cap_override is not None:
        free = free[:cap_override]
    cnt = torch.tensor([count], dtype=torch.int32, device=DEV)
    lo_t = None if lo is None else torch.tensor(lo, dtype=torch.int32, device=DEV)
    kvr.kv_pages_release_window(tab, nblk, bsz, torch.tensor(seqs, dtype=torch.int32, device=DEV),
                                torch.tensor(nxt, dtype=torch.int64, device=DEV), free, cnt, lo=lo_t, window=window)
    st = kvr.device_status()
    return (tab.cpu().numpy(), None if lo_t is None else lo_t.cpu().tolist(), free.cpu().numpy(),
            int(cnt.item()), st)


def _check_release(table_np, nblk, bsz, seqs, nxt, window, lo, free_np, count, cap=None):
    cap = len(free_np) if cap is None else cap
    got = _release_gpu(table_np, nblk, bsz, seqs, nxt, window, lo, free_np, count, cap_override=cap)
    w_tab, w_lo, w_ids, w_cnt, w_flags = opages.release_window(
        table_np.tolist(), nblk, bsz, seqs, nxt, window, lo=lo, free_ids=free_np[:cap].tolist(), free_count=count,
        free_cap=cap)
    g_tab, g_lo, g_ids, g_cnt, g_flags = got
    assert g_flags == w_flags, (g_flags, w_flags)
    assert g_cnt == w_cnt
    assert np.array_equal(g_tab, np.array(w_tab, dtype=np.int32))
    assert g_lo == w_lo
    assert g_ids.tolist() == w_ids
    return np.array(w_tab, dtype=np.int32), w_lo, np.array(w_ids + free_np[cap:].tolist(), dtype=np.int32), w_cnt


def test_release_matches_oracle_over_several_calls():
    rng = np.random.default_rng(71)
    S, mb, bsz, W = 45, 300, 16, 128          # 45 sequences: more than one round of 32 warps
    nblk = S * mb + 10
    tab = rng.permutation(nblk)[: S * mb].reshape(S, mb).astype(np.int32)
    tab[rng.random(tab.shape) < 0.1] = -1
    lo = [int(x) for x in rng.integers(0, 5, S)]
    free = rng.integers(0, 1000, nblk + 10).astype(np.int32)
    count = 5
    nxt = rng.integers(0, mb * bsz // 2, S)
    for step in range(3):
        seqs = [int(x) for x in rng.permutation(S)[:40]]
        nxt = nxt + rng.integers(0, 1500, S)
        tab, lo, free, count = _check_release(tab, nblk, bsz, seqs, [int(nxt[s]) for s in seqs], W, lo, free, count)
    assert count > 5
    # lo = NULL: every entry from block 0 is looked at again (the released ones hold -1)
    seqs = list(range(S))
    _check_release(tab, nblk, bsz, seqs, [int(x) + 4000 for x in nxt], W, None, free, count)


def test_release_long_range_and_window_sizes():
    # one sequence releasing ~20000 entries at once (the first release after a
    # long prefill), several windows and block sizes
    rng = np.random.default_rng(72)
    for bsz, W in [(16, 128), (64, 128), (64, 1), (256, 4096)]:
        S, mb = 3, 20000
        nblk = S * mb
        tab = rng.permutation(nblk).reshape(S, mb).astype(np.int32)
        free = np.zeros(nblk, dtype=np.int32)
        _check_release(tab, nblk, bsz, [2, 0], [mb * bsz - 7, 12345], W, [0, 0, 0], free, 0)


def test_release_flags_and_all_or_nothing():
    rng = np.random.default_rng(73)
    S, mb, bsz = 6, 40, 16
    nblk = S * mb
    tab = rng.permutation(nblk).reshape(S, mb).astype(np.int32)
    tab[1, 2] = nblk + 5                      # not a block id of the pool: left in place, flagged
    free = np.full(nblk, 7, dtype=np.int32)
    # bad sequence ids are skipped and flagged, the rest released
    _check_release(tab, nblk, bsz, [1, -1, 3, 6], [400, 500, 600, 700], 128, [0] * S, free, 0)
    # a free list that cannot take everything: nothing changes
    _check_release(tab, nblk, bsz, [0, 2], [639, 639], 128, [0] * S, free, 3, cap=10)


def test_paged_decode_unchanged_by_release(tables):
    # releasing with next_pos = p frees the blocks below the window and the
    # decode at p reads nothing from them: bit-identical output
    hq, hkv, bsz, vs = 64, 8, 16, 0.707
    positions = [140, 1000, 2047, 3000]
    syn = Synth(6401, device=DEV)
    B = len(positions)
    mb = max(positions) // bsz + 1
    nblk = B * mb
    tab = torch.from_numpy(np.random.default_rng(9).permutation(nblk).reshape(B, mb).astype(np.int32)).to(DEV)
    pool = _nan_pool(nblk, hkv, bsz, tab)
    for s, p in enumerate(positions):
        _append_range(pool, syn, s, 0, p + 1, tables[1e4], vs)
    q = syn.q(B, hq, hkv, seq=42)
    sinks = syn.sinks(hq).to(DEV)
    pos = torch.tensor(positions, dtype=torch.int64, device=DEV)
    seq = torch.arange(B, dtype=torch.int32, device=DEV)
    before = kvr.swa_sink_decode(q, pos, seq, pool, sinks, tables[1e4], SCALE).clone()
    free = torch.full((nblk,), -1, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
    lo = torch.zeros(B, dtype=torch.int32, device=DEV)
    kvr.kv_pages_release_window(pool.block_table, pool.num_blocks, bsz, seq, pos, free, cnt, lo=lo)
    # poison every released block: a read of one would show
    freed = free[: int(cnt.item())].long()
    pool.k.view(torch.int16)[freed] = NAN_BITS
    pool.v.view(torch.int16)[freed] = NAN_BITS
    after = kvr.swa_sink_decode(q, pos, seq, pool, sinks, tables[1e4], SCALE)
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    assert int(cnt.item()) == sum((p - 127) // bsz for p in positions)
    assert torch.equal(after.view(torch.int16), before.view(torch.int16))
    compare_rows(after, _oracle_swa(q, syn, hkv, list(range(B)), positions, sinks, vs), "after release")


# --------------------------------------------------------------------------- ring from pages

def test_ring_gather_matches_oracle_and_appends(tables):
    hkv, bsz, vs = 8, 32, 0.707
    ends = [0, 1, 77, 128, 129, 300, 1000]
    syn = Synth(6501, dist="shifted", device=DEV)
    S = len(ends)
    mb = max(ends) // bsz + 1
    nblk = S * mb
    tab = torch.from_numpy(np.random.default_rng(11).permutation(nblk).reshape(S, mb).astype(np.int32)).to(DEV)
    pool = _nan_pool(nblk, hkv, bsz, tab)
    for s, e in enumerate(ends):
        _append_range(pool, syn, s, 0, e, tables[1e4], vs)
    # ring rows 2..S+1 receive sequences 0..S-1; rows start with other data
    ring = kvr.RingLayout.empty(S + 2, hkv)
    ring.k.normal_()
    ring.v.normal_()
    ring.slot_pos.fill_(12345)
    k0, v0, t0 = ring.k.clone(), ring.v.clone(), ring.slot_pos.clone()
    src = torch.arange(S, dtype=torch.int32, device=DEV)
    dst = src + 2
    kvr.kv_ring_gather_pages(pool, ring, src, dst, torch.tensor(ends, dtype=torch.int64, device=DEV))
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    pk = pool.k.view(torch.int16).cpu().numpy().view(np.uint16)
    pv = pool.v.view(torch.int16).cpu().numpy().view(np.uint16)
    tb = tab.cpu().numpy()
    rk = ring.k.view(torch.int16).cpu().numpy().view(np.uint16)
    rv = ring.v.view(torch.int16).cpu().numpy().view(np.uint16)
    rt = ring.slot_pos.cpu().numpy()
    k0n = k0.view(torch.int16).cpu().numpy().view(np.uint16)
    v0n = v0.view(torch.int16).cpu().numpy().view(np.uint16)
    for s, e in enumerate(ends):
        wk, wv, wt, fl = opages.ring_from_pages(pk, pv, tb, bsz, s, e, k0n[s + 2], v0n[s + 2], t0[s + 2].cpu().numpy())
        assert fl == 0
        assert np.array_equal(rt[s + 2], wt) and np.array_equal(rk[s + 2], wk) and np.array_equal(rv[s + 2], wv)
    # rows 0 and 1 untouched
    assert torch.equal(ring.k[:2], k0[:2]) and torch.equal(ring.slot_pos[:2], t0[:2])
    # the same as a ring that received the positions by appends
    ring2 = kvr.RingLayout.empty(S + 2, hkv)
    for s, e in enumerate(ends):
        lo = max(0, e - 128)
        if e > lo:
            k, v = raw_kv(syn, hkv, s, lo, e)
            kvr.kv_ring_append_rope(k, v, torch.arange(lo, e, device=DEV),
                                    torch.full((e - lo,), s + 2, dtype=torch.int32, device=DEV), tables[1e4], vs, ring2)
    valid = ring2.slot_pos[2:] >= 0
    assert torch.equal(ring.slot_pos[2:][valid], ring2.slot_pos[2:][valid])
    assert torch.equal((ring.slot_pos[2:] >= 0), valid)
    for h in range(hkv):
        assert torch.equal(ring.k[2:, h][valid].view(torch.int16), ring2.k[2:, h][valid].view(torch.int16))
        assert torch.equal(ring.v[2:, h][valid].view(torch.int16), ring2.v[2:, h][valid].view(torch.int16))


@pytest.mark.parametrize("bsz", [16, 64, 256])
def test_ring_gather_runs_across_adjacent_blocks(bsz, tables):
    # One KV head and a block table of consecutive ids: the pool rows of
    # neighbouring blocks are adjacent in memory, so a window's slots form
    # runs longer than a block (split only at the ring's wrap, at a missing
    # block and where the ids stop being consecutive).  Bit-exact against the
    # oracle's ring_from_pages.
    hkv, vs = 1, 0.707
    ends = [1, 128, 129, 200, 1000, 1000, 777]
    syn = Synth(6701, dist="shifted", device=DEV)
    S = len(ends)
    mb = max(ends) // bsz + 1
    nblk = S * mb
    tab = torch.arange(nblk, dtype=torch.int32, device=DEV).reshape(S, mb)
    tab[5] = torch.flip(tab[5], [0])           # sequence 5: descending ids, runs end at every block edge
    pool = _nan_pool(nblk, hkv, bsz, tab)
    for s, e in enumerate(ends):
        _append_range(pool, syn, s, 0, e, tables[1e4], vs)
    miss = (777 - 60) // bsz
    pool.block_table[6, miss] = -1            # sequence 6: a hole inside its window
    ring = kvr.RingLayout.empty(S, hkv)
    ring.k.normal_()
    ring.v.normal_()
    ring.slot_pos.fill_(-7)
    k0, v0, t0 = ring.k.clone(), ring.v.clone(), ring.slot_pos.clone()
    src = torch.arange(S, dtype=torch.int32, device=DEV)
    assert kvr.device_status() == 0          # (and cleared)
    kvr.kv_ring_gather_pages(pool, ring, src, src, torch.tensor(ends, dtype=torch.int64, device=DEV))
    torch.cuda.synchronize()
    assert kvr.device_status() == kvr.DEV_BAD_BLOCK
    pk = pool.k.view(torch.int16).cpu().numpy().view(np.uint16)
    pv = pool.v.view(torch.int16).cpu().numpy().view(np.uint16)
    tb = pool.block_table.cpu().numpy()
    rk = ring.k.view(torch.int16).cpu().numpy().view(np.uint16)
    rv = ring.v.view(torch.int16).cpu().numpy().view(np.uint16)
    rt = ring.slot_pos.cpu().numpy()
    k0n = k0.view(torch.int16).cpu().numpy().view(np.uint16)
    v0n = v0.view(torch.int16).cpu().numpy().view(np.uint16)
    for s, e in enumerate(ends):
        wk, wv, wt, fl = opages.ring_from_pages(pk, pv, tb, bsz, s, e, k0n[s], v0n[s], t0[s].cpu().numpy())
        assert fl == (opages.BAD_BLOCK if s == 6 else 0), s
        assert np.array_equal(rt[s], wt), s
        assert np.array_equal(rk[s], wk) and np.array_equal(rv[s], wv), s


def test_ring_gather_flags_missing_blocks(tables):
    hkv, bsz = 2, 16
    syn = Synth(6601, device=DEV)
    tab = torch.arange(40, dtype=torch.int32, device=DEV).reshape(2, 20)
    pool = _nan_pool(40, hkv, bsz, tab)
    _append_range(pool, syn, 0, 0, 300, tables[1e4], 0.707)
    pool.block_table[0, 12] = -1               # positions 192..207: inside the window of end = 300
    ring = kvr.RingLayout.empty(3, hkv)
    kvr.kv_ring_gather_pages(pool, ring, torch.tensor([0, 5], dtype=torch.int32, device=DEV),
                             torch.tensor([1, 2], dtype=torch.int32, device=DEV),
                             torch.tensor([300, 10], dtype=torch.int64, device=DEV))
    assert kvr.device_status() == kvr.DEV_BAD_BLOCK | kvr.DEV_BAD_SEQ
    tags = ring.slot_pos[1].cpu().numpy()
    for c in range(128):
        p = opages.ring_slot_position(300, c)
        assert tags[c] == (-1 if 192 <= p < 208 else p)
    assert torch.all(ring.slot_pos[2] == -1)   # the bad entry was skipped


def test_gather_then_windowed_prefill_chunk(tables):
    # a sequence kept in pages continues through the ring-based chunked
    # prefill: gather the window before P0, then swa_sink_prefill_chunk
    hq, hkv, bsz, vs = 64, 8, 64, 0.707
    P0, C = 500, 300
    syn = Synth(6701, dist="plain", device=DEV)
    tab = torch.arange(16, dtype=torch.int32, device=DEV).reshape(1, 16)
    pool = _nan_pool(16, hkv, bsz, tab)
    _append_range(pool, syn, 0, 0, P0, tables[1e4], vs)
    ring = kvr.RingLayout.empty(1, hkv)
    kvr.kv_ring_gather_pages(pool, ring, torch.tensor([0], dtype=torch.int32, device=DEV),
                             torch.tensor([0], dtype=torch.int32, device=DEV),
                             torch.tensor([P0], dtype=torch.int64, device=DEV))
    k, v = raw_kv(syn, hkv, 0, P0, P0 + C)
    stage = kvr.LinearLayout.empty(C, hkv)
    kvr.kv_ring_append_rope(k, v, torch.arange(P0, P0 + C, device=DEV), None, tables[1e4], vs, stage)
    q = syn.q(C, hq, hkv, seq=0, start=P0)
    sinks = syn.sinks(hq).to(DEV)
    out = kvr.swa_sink_prefill_chunk(q, P0, 0, stage, ring, sinks, tables[1e4], SCALE)
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    lo = P0 - 127
    kk, vv = raw_kv(syn, hkv, 0, lo, P0 + C)
    want = oracle.attend_seq(q, np.arange(P0, P0 + C), kk, vv, lo, 1e4, vs, SCALE, 128, sinks.double().cpu().numpy())
    compare(out, want, "gather + windowed prefill")
    compare_rows(out, want, "gather + windowed prefill")
