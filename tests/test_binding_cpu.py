"""Host logic of the Python binding, without a GPU.  The C ABI takes bare
pointers, so the binding checks every size the kernels index by, and that a
call's tensors share the current device, before it reaches the library.  Here
the library is a recorder that only logs the calls it gets (nothing computes)
and the tensors live on the CPU."""
import pytest
import torch

import sinks_kv_ring_gb300 as kvr

B, HQ, HKV = 3, 16, 2


class _Recorder:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def call(*args):
            self.calls.append((name, args))
            return 4096 if name.endswith("workspace_size") else 0
        return call


@pytest.fixture
def rec(monkeypatch):
    r = _Recorder()
    want = kvr._want
    monkeypatch.setattr(kvr, "lib", lambda: r)
    monkeypatch.setattr(kvr, "_want", lambda t, name, dtype, dim=None, cuda=True: want(t, name, dtype, dim, cuda=False))
    monkeypatch.setattr(kvr, "_stream", lambda s: None)
    monkeypatch.setattr(torch.cuda, "current_device", lambda: None)  # a CPU tensor's device index
    return r


def _bf(*shape):
    return torch.zeros(*shape, dtype=torch.bfloat16)


def _i32(*shape):
    return torch.zeros(*shape, dtype=torch.int32)


def _i64(*shape):
    return torch.zeros(*shape, dtype=torch.int64)


def _f32(*shape):
    return torch.zeros(*shape, dtype=torch.float32)


def _layouts():
    ring = kvr.RingLayout.empty(4, HKV, device="cpu")
    pool = kvr.PagedLayout.contiguous(4, HKV, 256, block_size=64, device="cpu")
    stage = kvr.LinearLayout.empty(8, HKV, device="cpu")
    return ring, pool, stage


def _decode_args():
    return _bf(B, HQ, 192), _i64(B), _i32(B)


def test_matching_shapes_reach_the_library(rec):
    ring, pool, stage = _layouts()
    q, pos, seq = _decode_args()
    table, sinks = _f32(300, 32, 2), _f32(HQ)
    out = kvr.swa_sink_decode(q, pos, seq, ring, sinks, table, 0.1)
    assert tuple(out.shape) == (B, HQ, 128)
    kvr.full_attn_decode(q, pos, seq, pool, table, 0.1, 256)
    kvr.full_attn_decode_noalloc(q, pos, seq, pool, table, 0.1, 256, out=_bf(B, HQ, 128))
    qc = _bf(8, HQ, 192)
    kvr.swa_sink_prefill_chunk(qc, 100, 1, stage, ring, sinks, table, 0.1)
    kvr.full_attn_prefill_chunk(qc, 100, 1, pool, table, 0.1)
    cu, P0, sq = torch.tensor([0, 5, 8], dtype=torch.int32), _i64(2), _i32(2)
    kvr.full_attn_prefill_varlen(qc, cu, P0, sq, pool, table, 0.1, 256)
    kvr.swa_sink_prefill_varlen(qc, cu, P0, sq, stage, ring, sinks, table, 0.1)
    kvr.kv_ring_append_rope(_bf(8, HKV, 192), _bf(8, HKV, 128), _i64(8), None, table, 0.7, stage)
    names = [n for n, _ in rec.calls if not n.endswith("workspace_size")]
    assert names == ["swa_sink_decode", "full_attn_decode", "full_attn_decode_noalloc", "swa_sink_prefill_chunk",
                     "full_attn_prefill_chunk", "full_attn_prefill_varlen", "swa_sink_prefill_varlen",
                     "kv_ring_append_rope"]
    args = dict(rec.calls)["swa_sink_decode"]
    assert (args[3], args[4], args[8]) == (B, HQ, 300)  # B, Hq, the table's positions


@pytest.mark.parametrize("bad", ["out_rows", "out_heads", "out_width", "sinks", "pos", "seq", "q_width",
                                 "table", "device", "current_device"])
def test_swa_decode_refuses_before_the_library(rec, monkeypatch, bad):
    ring, _, _ = _layouts()
    q, pos, seq = _decode_args()
    table, sinks, out = _f32(300, 32, 2), _f32(HQ), _bf(B, HQ, 128)
    if bad == "out_rows":
        out = _bf(B - 1, HQ, 128)
    elif bad == "out_heads":
        out = _bf(B, HQ // 2, 128)
    elif bad == "out_width":
        out = _bf(B, HQ, 64)
    elif bad == "sinks":
        sinks = _f32(HQ - 1)
    elif bad == "pos":
        pos = _i64(B - 1)
    elif bad == "seq":
        seq = _i32(B + 1)
    elif bad == "q_width":
        q = _bf(B, HQ, 128)
    elif bad == "table":
        table = _f32(300, 64)[:, :, None].contiguous()
    elif bad == "device":
        sinks = torch.empty(HQ, dtype=torch.float32, device="meta")
    elif bad == "current_device":
        monkeypatch.setattr(torch.cuda, "current_device", lambda: 1)
    with pytest.raises(ValueError):
        kvr.swa_sink_decode(q, pos, seq, ring, sinks, table, 0.1, out=out)
    assert rec.calls == []


def test_other_calls_refuse_mismatched_sizes(rec):
    ring, pool, stage = _layouts()
    q, pos, seq = _decode_args()
    table, sinks = _f32(300, 32, 2), _f32(HQ)
    qc = _bf(8, HQ, 192)
    cu, P0, sq = torch.tensor([0, 5, 8], dtype=torch.int32), _i64(2), _i32(2)
    cases = [
        lambda: kvr.full_attn_decode(q, pos[:2], seq, pool, table, 0.1, 256),
        lambda: kvr.full_attn_decode(q, pos, seq, pool, table, 0.1, 256, out=_bf(B + 1, HQ, 128)),
        lambda: kvr.full_attn_decode_noalloc(q, pos, seq[:1], pool, table, 0.1, 256),
        lambda: kvr.swa_sink_prefill_chunk(qc, 100, 1, stage, ring, _f32(HQ + 1), table, 0.1),
        lambda: kvr.swa_sink_prefill_chunk(qc, 100, 1, stage, ring, sinks, table, 0.1, out=_bf(7, HQ, 128)),
        lambda: kvr.full_attn_prefill_chunk(_bf(8, HQ, 191), 100, 1, pool, table, 0.1),
        lambda: kvr.full_attn_prefill_varlen(qc, cu, P0, sq, pool, _f32(300, 16, 2), 0.1, 256),
        lambda: kvr.swa_sink_prefill_varlen(qc, cu, P0, sq, stage, ring, sinks, table, 0.1, out=_bf(8, HQ, 192)),
        lambda: kvr.swa_sink_prefill_varlen(qc, cu[:2], P0, sq, stage, ring, sinks, table, 0.1),
        lambda: kvr.kv_ring_append_rope(_bf(8, HKV, 192), _bf(8, HKV, 128), _i64(8), None, _f32(300, 32, 3), 0.7,
                                        stage),
        lambda: kvr.full_attn_prefill_chunk(qc, 100, 1, pool, table.to("meta"), 0.1),
    ]
    for i, case in enumerate(cases):
        with pytest.raises(ValueError):
            case()
        assert [n for n, _ in rec.calls if not n.endswith("workspace_size")] == [], i


def test_pool_calls_check_devices_and_reach_the_library(rec):
    ring, pool, _ = _layouts()
    seqs, end = _i32(2), _i64(2)
    snap = kvr.ring_snapshot_alloc(2, HKV, device="cpu")
    kvr.kv_ring_snapshot(ring, seqs, snap)
    kvr.kv_ring_restore(ring, seqs, snap)
    kvr.kv_ring_gather_pages(pool, ring, seqs, seqs, end)
    kvr.kv_pages_release_window(pool.block_table, pool.num_blocks, 64, seqs, end, _i32(16), _i32(1))
    assert [n for n, _ in rec.calls] == ["kv_ring_snapshot", "kv_ring_restore", "kv_ring_gather_pages",
                                         "kv_pages_release_window"]
    rec.calls.clear()
    meta = lambda t: torch.empty(t.shape, dtype=t.dtype, device="meta")
    cases = [
        lambda: kvr.kv_ring_snapshot(ring, seqs, (snap[0], meta(snap[1]), snap[2])),
        lambda: kvr.kv_ring_gather_pages(pool, ring, seqs, seqs, meta(end)),
        lambda: kvr.kv_pages_release_window(pool.block_table, pool.num_blocks, 64, seqs, end, _i32(16), _i32(1),
                                            lo=meta(_i32(4))),
    ]
    for i, case in enumerate(cases):
        with pytest.raises(ValueError):
            case()
        assert rec.calls == [], i
