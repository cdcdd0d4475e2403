"""The bounded-wait exit of the pipelined kernels, made to run on purpose.

Every wait of the windowed decode kernels (over rings and over pages), of the
short-chunk windowed kernel, of the tensor-core prefill kernel and of the
bulk-copy kernels (ring from pages, ring snapshot / restore) has a time
limit; when one runs out the kernel sets an abort flag, its other warps
leave their loops, the loads and products already issued finish, tensor
memory is freed and the kernel returns with KVR_DEV_TIMEOUT set.  The test
hook kvr_debug_stall_next makes one launch wait on a barrier that nothing
completes, with a short limit, once its loads are in flight: the call must
return promptly, report the timeout, and leave the device usable -- the next
normal call on it matches the oracle.  No fault, trap or endless wait is
involved: the stalled wait ends by its own limit.
"""
import math
import time

import numpy as np
import pytest
import torch

import oracle
import sinks_kv_ring_gb300 as kvr
from sinks_kv_ring_gb300.synth import Synth

from kvr_cases import SCALE, compare_rows, fill_paged, fill_ring, raw_kv

pytestmark = pytest.mark.gpu
DEV = "cuda"
LIMIT_NS = 200_000  # the stalled wait's limit: 0.2 ms


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sinks_kv_ring_gb300 import build
    build.build()
    kvr.device_status(reset=True)
    yield
    kvr.debug_stall_next(0, 1000)


def _stalled(call):
    """Run call() with the next launch stalled; returns the seconds it took."""
    kvr.device_status(reset=True)
    kvr.debug_stall_next(1, LIMIT_NS)
    try:
        t0 = time.perf_counter()
        call()
        torch.cuda.synchronize()
        return time.perf_counter() - t0
    finally:
        kvr.debug_stall_next(0, 1000)


# 16 x 8 KV heads: one unit per CTA of one group; 40: CTAs of four groups;
# 64: two CTAs of two groups per SM
@pytest.mark.parametrize("B", [16, 40, 64])
def test_windowed_decode_stall_takes_the_bounded_exit(B):
    hq, hkv = 64, 8
    positions = [300 + 7 * b for b in range(B)]
    t4 = kvr.rope_table(1e4, 4096)
    syn = Synth(2601, dist="plain", device=DEV)
    ring = kvr.RingLayout.empty(B, hkv)
    fill_ring(ring, syn, list(range(B)), positions, t4, 0.707)
    q = syn.q(B, hq, hkv, seq=999)
    sinks = syn.sinks(hq).to(DEV)
    pos = torch.tensor(positions, dtype=torch.int64, device=DEV)
    seq = torch.arange(B, dtype=torch.int32, device=DEV)
    out = torch.empty(B, hq, 128, dtype=torch.bfloat16, device=DEV)
    dt = _stalled(lambda: kvr.swa_sink_decode(q, pos, seq, ring, sinks, t4, SCALE, out=out))
    assert kvr.device_status() & kvr.DEV_TIMEOUT
    assert dt < 5.0, f"the stalled call took {dt:.2f} s"
    # the device is still usable: the same call, not stalled
    out = kvr.swa_sink_decode(q, pos, seq, ring, sinks, t4, SCALE)
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    want = np.zeros((B, hq, 128))
    sk = sinks.double().cpu().numpy()
    for b, p in enumerate(positions):
        k, v = raw_kv(syn, hkv, b, p - 127, p + 1)
        want[b] = oracle.attend_seq(q[b:b + 1], [p], k, v, p - 127, 1e4, 0.707, SCALE, 128, sk)[0]
    compare_rows(out, want, "windowed decode after a stalled launch")


def test_prefill_stall_takes_the_bounded_exit():
    # The tensor-core kernel stalls in its MMA warp with TMEM allocated and
    # its first K/V loads issued; 20 CTAs (10 tiles of 256 rows x 2 KV heads).
    hq, hkv, P0, C = 16, 2, 700, 300
    t7 = kvr.rope_table(1e7, 2048)
    syn = Synth(2602, dist="plain", device=DEV)
    pool = kvr.PagedLayout.contiguous(1, hkv, 2048, block_size=64)
    fill_paged(pool, syn, [0], [P0 + C], t7, 0.707)
    q = syn.q(C, hq, hkv, seq=5, start=P0)
    out = torch.empty(C, hq, 128, dtype=torch.bfloat16, device=DEV)
    dt = _stalled(lambda: kvr.full_attn_prefill_chunk(q, P0, 0, pool, t7, SCALE, out=out))
    assert kvr.device_status() & kvr.DEV_TIMEOUT
    assert dt < 5.0, f"the stalled call took {dt:.2f} s"
    out = kvr.full_attn_prefill_chunk(q, P0, 0, pool, t7, SCALE)
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    k, v = raw_kv(syn, hkv, 0, 0, P0 + C)
    want = oracle.attend_seq(q, np.arange(P0, P0 + C), k, v, 0, 1e7, 0.707, SCALE, 0, None)
    compare_rows(out, want, "prefill after a stalled launch")


def test_paged_windowed_decode_stall_takes_the_bounded_exit():
    # The windowed decode over pages (8 q heads per KV head): 40 sequences x 8
    # KV heads = 320 windows, two or three per CTA, its producers and both
    # consumer groups in flight when group 0 stalls.
    B, hq, hkv = 40, 64, 8
    positions = [300 + 7 * b for b in range(B)]
    t4 = kvr.rope_table(1e4, 4096)
    syn = Synth(2603, dist="plain", device=DEV)
    pool = kvr.PagedLayout.contiguous(B, hkv, max(positions) + 1, block_size=64)
    fill_paged(pool, syn, list(range(B)), [p + 1 for p in positions], t4, 0.707)
    q = syn.q(B, hq, hkv, seq=998)
    sinks = syn.sinks(hq).to(DEV)
    pos = torch.tensor(positions, dtype=torch.int64, device=DEV)
    seq = torch.arange(B, dtype=torch.int32, device=DEV)
    out = torch.empty(B, hq, 128, dtype=torch.bfloat16, device=DEV)
    dt = _stalled(lambda: kvr.swa_sink_decode(q, pos, seq, pool, sinks, t4, SCALE, out=out))
    assert kvr.device_status() & kvr.DEV_TIMEOUT
    assert dt < 5.0, f"the stalled call took {dt:.2f} s"
    out = kvr.swa_sink_decode(q, pos, seq, pool, sinks, t4, SCALE)
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    want = np.zeros((B, hq, 128))
    sk = sinks.double().cpu().numpy()
    for b, p in enumerate(positions):
        k, v = raw_kv(syn, hkv, b, p - 127, p + 1)
        want[b] = oracle.attend_seq(q[b:b + 1], [p], k, v, p - 127, 1e4, 0.707, SCALE, 128, sk)[0]
    compare_rows(out, want, "paged windowed decode after a stalled launch")


def test_short_chunk_windowed_stall_takes_the_bounded_exit():
    # Draft verification of a windowed layer: 48 sequences x 3 tokens x 8 KV
    # heads = 384 units through the short-chunk kernel, group 0 stalled.
    n, C, hq, hkv = 48, 3, 64, 8
    P0s = [500 + 11 * s for s in range(n)]
    t4 = kvr.rope_table(1e4, 4096)
    syn = Synth(2604, dist="plain", device=DEV)
    sinks = syn.sinks(hq).to(DEV)
    ring = kvr.RingLayout.empty(n, hkv)
    fill_ring(ring, syn, list(range(n)), [P0 - 1 for P0 in P0s], t4, 0.707)
    ks, vs, ps = [], [], []
    for s, P0 in enumerate(P0s):
        k, v = raw_kv(syn, hkv, s, P0, P0 + C)
        ks.append(k)
        vs.append(v)
        ps.append(torch.arange(P0, P0 + C, dtype=torch.int64, device=DEV))
    stage = kvr.LinearLayout.empty(n * C, hkv)
    kvr.kv_ring_append_rope(torch.cat(ks).contiguous(), torch.cat(vs).contiguous(), torch.cat(ps), None, t4, 0.707,
                            stage)
    q = torch.cat([syn.q(C, hq, hkv, seq=s, start=P0) for s, P0 in enumerate(P0s)]).contiguous()
    cu = torch.arange(0, n * C + 1, C, dtype=torch.int32, device=DEV)
    P0 = torch.tensor(P0s, dtype=torch.int64, device=DEV)
    sq = torch.arange(n, dtype=torch.int32, device=DEV)
    out = torch.empty(n * C, hq, 128, dtype=torch.bfloat16, device=DEV)
    call = lambda o=None: kvr.swa_sink_prefill_varlen(q, cu, P0, sq, stage, ring, sinks, t4, SCALE, out=o)
    dt = _stalled(lambda: call(out))
    assert kvr.device_status() & kvr.DEV_TIMEOUT
    assert dt < 5.0, f"the stalled call took {dt:.2f} s"
    out = call()
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    sk = sinks.double().cpu().numpy()
    want = np.concatenate([
        oracle.attend_seq(q[s * C:(s + 1) * C], np.arange(P0, P0 + C), *raw_kv(syn, hkv, s, P0 - 127, P0 + C),
                          P0 - 127, 1e4, 0.707, SCALE, 128, sk) for s, P0 in enumerate(P0s)])
    compare_rows(out, want, "short-chunk windowed attention after a stalled launch")


def test_ring_gather_stall_takes_the_bounded_exit():
    # Ring from pages, 12 sequences x 8 KV heads (K and V CTAs): the first
    # CTA's copies are in flight when it stalls; it stores nothing.
    import oracle.pages as opages
    hkv, bsz, S = 8, 32, 12
    ends = [200 + 37 * s for s in range(S)]
    t4 = kvr.rope_table(1e4, 4096)
    syn = Synth(2605, dist="plain", device=DEV)
    pool = kvr.PagedLayout.contiguous(S, hkv, max(ends), block_size=bsz)
    fill_paged(pool, syn, list(range(S)), ends, t4, 0.707)
    ring = kvr.RingLayout.empty(S, hkv)
    seq = torch.arange(S, dtype=torch.int32, device=DEV)
    end = torch.tensor(ends, dtype=torch.int64, device=DEV)
    dt = _stalled(lambda: kvr.kv_ring_gather_pages(pool, ring, seq, seq, end))
    assert kvr.device_status() & kvr.DEV_TIMEOUT
    assert dt < 5.0, f"the stalled call took {dt:.2f} s"
    kvr.kv_ring_gather_pages(pool, ring, seq, seq, end)
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    pk = pool.k.view(torch.int16).cpu().numpy().view(np.uint16)
    pv = pool.v.view(torch.int16).cpu().numpy().view(np.uint16)
    tb = pool.block_table.cpu().numpy()
    rk = ring.k.view(torch.int16).cpu().numpy().view(np.uint16)
    rv = ring.v.view(torch.int16).cpu().numpy().view(np.uint16)
    rt = ring.slot_pos.cpu().numpy()
    for s, e in enumerate(ends):  # every slot holds a position (end >= 128): the base rows do not matter
        wk, wv, wt, fl = opages.ring_from_pages(pk, pv, tb, bsz, s, e, rk[s], rv[s], rt[s])
        assert fl == 0 and np.array_equal(rt[s], wt), s
        assert np.array_equal(rk[s], wk) and np.array_equal(rv[s], wv), s


@pytest.mark.parametrize("restore", [False, True])
def test_ring_snapshot_stall_takes_the_bounded_exit(restore):
    # Snapshot (or restore) of 12 sequences x 8 KV heads in 16 KB pieces: the
    # first piece's copy is in flight when its CTA stalls; it stores nothing.
    S, hkv = 12, 8
    ring = kvr.RingLayout.empty(S, hkv)
    ring.k.normal_()
    ring.v.normal_()
    ring.slot_pos.copy_(torch.arange(S * 128, dtype=torch.int32, device=DEV).reshape(S, 128))
    seq = torch.arange(S, dtype=torch.int32, device=DEV)
    snap = kvr.ring_snapshot_alloc(S, hkv, device=DEV)
    if restore:
        kvr.kv_ring_snapshot(ring, seq, snap)
        k0, v0, t0 = ring.k.clone(), ring.v.clone(), ring.slot_pos.clone()
        ring.k.zero_()
        ring.v.zero_()
        call = lambda: kvr.kv_ring_restore(ring, seq, snap)
    else:
        call = lambda: kvr.kv_ring_snapshot(ring, seq, snap)
    dt = _stalled(call)
    assert kvr.device_status() & kvr.DEV_TIMEOUT
    assert dt < 5.0, f"the stalled call took {dt:.2f} s"
    call()
    torch.cuda.synchronize()
    assert kvr.device_status() == 0
    if restore:
        assert torch.equal(ring.k.view(torch.int16), k0.view(torch.int16))
        assert torch.equal(ring.v.view(torch.int16), v0.view(torch.int16))
        assert torch.equal(ring.slot_pos, t0)
    else:
        back = kvr.RingLayout.empty(S, hkv)
        kvr.kv_ring_restore(back, seq, snap)
        torch.cuda.synchronize()
        assert torch.equal(back.k.view(torch.int16), ring.k.view(torch.int16))
        assert torch.equal(back.v.view(torch.int16), ring.v.view(torch.int16))
        assert torch.equal(back.slot_pos, ring.slot_pos)
