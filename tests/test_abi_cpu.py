"""CPU-side checks of the C-ABI library: it loads, exports every function
include/kvring.h declares, rejects bad arguments on the host before touching
a GPU, and its host-built fp64 RoPE table matches the oracle."""
import ctypes
import os
import re

import numpy as np
import pytest

import sinks_kv_ring_gb300 as kvr
from sinks_kv_ring_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvring.h")


@pytest.fixture(scope="module")
def L():
    kbuild.build()
    return kvr.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    src = re.sub(r"^\s*#[^\n]*", "", src, flags=re.M)
    names = re.findall(r"\b([A-Za-z_]\w*)\s*\([^;{}]*\)\s*;", src)
    return sorted(set(names))


def test_header_declares_the_five_calls():
    names = declared_functions()
    for n in ("kv_ring_append_rope", "swa_sink_decode", "full_attn_decode", "swa_sink_prefill_chunk",
              "full_attn_prefill_chunk", "full_attn_decode_workspace_size", "kvr_rope_table_build",
              "kvr_last_error", "kvr_device_status"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for n in declared_functions():
        assert hasattr(L, n), n


FAKE = 0x10000  # aligned, never dereferenced: every call below fails validation first


def _ring(**kw):
    d = dict(kind=1, num_kv_heads=8, k=FAKE, v=FAKE, slot_pos=FAKE, block_table=None, num_seqs=4,
             max_blocks=0, block_size=0, num_blocks=0, num_rows=0)
    d.update(kw)
    return kvr._Layout(**d)


def _paged(**kw):
    d = dict(kind=2, num_kv_heads=4, k=FAKE, v=FAKE, slot_pos=None, block_table=FAKE, num_seqs=4,
             max_blocks=16, block_size=64, num_blocks=64, num_rows=0)
    d.update(kw)
    return kvr._Layout(**d)


def test_host_validation_codes(L):
    P = ctypes.c_void_p(FAKE)
    ring = _ring()
    # wrong layout kind (RING or PAGED are taken)
    lin = _paged(kind=3, num_rows=16)
    assert L.swa_sink_decode(P, P, P, 2, 64, ctypes.byref(lin), P, P, 1000, 0.1, P, None) == -1
    # a PAGED windowed layer: still at most 16 query heads per KV head
    assert L.swa_sink_decode(P, P, P, 2, 128, ctypes.byref(_paged()), P, P, 1000, 0.1, P, None) == -4
    # Hq not a multiple of Hkv
    assert L.swa_sink_decode(P, P, P, 2, 60, ctypes.byref(ring), P, P, 1000, 0.1, P, None) == -1
    # more than 16 query heads per KV head
    assert L.swa_sink_decode(P, P, P, 2, 256, ctypes.byref(ring), P, P, 1000, 0.1, P, None) == -4
    assert b"at most 16" in L.kvr_last_error()
    # null layout
    assert L.swa_sink_decode(P, P, P, 2, 64, None, P, P, 1000, 0.1, P, None) == -1
    # unaligned q
    assert L.swa_sink_decode(ctypes.c_void_p(FAKE + 2), P, P, 2, 64, ctypes.byref(ring), P, P, 1000, 0.1, P,
                             None) == -1
    pool = _paged()
    need = L.full_attn_decode_workspace_size(2, 64, 4, 1000)
    assert need > 0
    # workspace too small
    assert L.full_attn_decode(P, P, P, 2, 64, ctypes.byref(pool), P, 1000, 0.1, 1000, P, need - 1, P, None) == -3
    # max_ctx past the table / past the block table
    assert L.full_attn_decode(P, P, P, 2, 64, ctypes.byref(pool), P, 1000, 0.1, 1001, P, 1 << 40, P, None) == -2
    assert L.full_attn_decode(P, P, P, 2, 64, ctypes.byref(pool), P, 5000, 0.1, 1025, P, 1 << 40, P, None) == -2
    # block size not a multiple of 16
    assert L.full_attn_decode(P, P, P, 2, 64, ctypes.byref(_paged(block_size=24)), P, 1000, 0.1, 100, P, 1 << 40,
                              P, None) == -4
    # prefill past the table, bad sequence id
    assert L.full_attn_prefill_chunk(P, 900, 200, 0, 64, ctypes.byref(pool), P, 1000, 0.1, P, None) == -2
    assert L.full_attn_prefill_chunk(P, 0, 200, 9, 64, ctypes.byref(pool), P, 1000, 0.1, P, None) == -1
    lin = kvr._Layout(kind=3, num_kv_heads=8, k=FAKE, v=FAKE, slot_pos=None, block_table=None, num_seqs=0,
                      max_blocks=0, block_size=0, num_blocks=0, num_rows=100)
    assert L.swa_sink_prefill_chunk(P, 0, 200, 0, 64, ctypes.byref(lin), ctypes.byref(ring), P, P, 1000, 0.1,
                                    P, None) == -1          # chunk rows < C
    # append: Hkv disagrees with the layout; LINEAR too short
    assert L.kv_ring_append_rope(P, P, P, P, 10, 4, P, 1000, 0.7, ctypes.byref(ring), None) == -1
    assert L.kv_ring_append_rope(P, P, P, None, 200, 8, P, 1000, 0.7, ctypes.byref(lin), None) == -1
    # zero-sized calls are no-ops that succeed without a GPU
    assert L.kv_ring_append_rope(P, P, P, P, 0, 8, P, 1000, 0.7, ctypes.byref(ring), None) == 0
    assert L.swa_sink_decode(P, P, P, 0, 64, ctypes.byref(ring), P, P, 1000, 0.1, P, None) == 0


def test_varlen_host_validation_codes(L):
    P = ctypes.c_void_p(FAKE)
    ring, pool = _ring(), _paged()
    lin = kvr._Layout(kind=3, num_kv_heads=8, k=FAKE, v=FAKE, slot_pos=None, block_table=None, num_seqs=0,
                      max_blocks=0, block_size=0, num_blocks=0, num_rows=100)
    need = L.full_attn_prefill_varlen_workspace_size(4, 16, 64, 4, 1000)
    assert need > 0
    assert L.full_attn_prefill_varlen_workspace_size(4, 16, 62, 4, 1000) == 0  # Hq % Hkv
    # workspace too small; max_ctx past the table; null cu_rows; wrong layout kind
    assert L.full_attn_prefill_varlen(P, P, P, P, 4, 16, 64, ctypes.byref(pool), P, 1000, 0.1, 1000, P, need - 1,
                                      P, None) == -3
    assert L.full_attn_prefill_varlen(P, P, P, P, 4, 16, 64, ctypes.byref(pool), P, 1000, 0.1, 1001, P, 1 << 40,
                                      P, None) == -2
    assert L.full_attn_prefill_varlen(P, None, P, P, 4, 16, 64, ctypes.byref(pool), P, 1000, 0.1, 1000, P,
                                      1 << 40, P, None) == -1
    assert L.full_attn_prefill_varlen(P, P, P, P, 4, 16, 64, ctypes.byref(ring), P, 1000, 0.1, 1000, P, 1 << 40,
                                      P, None) == -1
    # empty batches succeed without a GPU
    assert L.full_attn_prefill_varlen(P, P, P, P, 0, 16, 64, ctypes.byref(pool), P, 1000, 0.1, 1000, None, 0, P,
                                      None) == 0
    wsn = L.swa_sink_prefill_varlen_workspace_size(4)
    assert wsn >= 4 * 3 * 4
    # chunk rows < T; workspace too small; unaligned out
    assert L.swa_sink_prefill_varlen(P, P, P, P, 4, 200, 64, ctypes.byref(lin), ctypes.byref(ring), P, P, 1000, 0.1,
                                     P, 1 << 30, P, None) == -1
    assert L.swa_sink_prefill_varlen(P, P, P, P, 4, 16, 64, ctypes.byref(lin), ctypes.byref(ring), P, P, 1000, 0.1,
                                     P, wsn - 1, P, None) == -3
    assert L.swa_sink_prefill_varlen(P, P, P, P, 4, 16, 64, ctypes.byref(lin), ctypes.byref(ring), P, P, 1000, 0.1,
                                     P, 1 << 30, ctypes.c_void_p(FAKE + 2), None) == -1
    assert L.swa_sink_prefill_varlen(P, P, P, P, 4, 0, 64, ctypes.byref(lin), ctypes.byref(ring), P, P, 1000, 0.1,
                                     None, 0, P, None) == 0


def test_stall_hook_host_validation(L):
    assert L.kvr_debug_stall_next(-1, 100000) == -1
    assert L.kvr_debug_stall_next(1, 999) == -1
    assert L.kvr_debug_stall_next(1, 2_000_000_000) == -1
    assert L.kvr_debug_stall_next(0, 1000) == 0


def test_workspace_size_grows_with_context(L):
    a = L.full_attn_decode_workspace_size(64, 64, 4, 32769)
    b = L.full_attn_decode_workspace_size(64, 64, 4, 2 * 32769)
    assert 0 < a <= b
    assert L.full_attn_decode_workspace_size(64, 60, 8, 100) == 0


def test_rope_table_matches_oracle_fp64():
    import oracle
    for theta in (1e4, 1e7):
        for base in (0, 131000, 199990, 524280, 1048560):
            tab = kvr.rope_table(theta, base + 16, device="cpu").numpy()
            for p in range(base, base + 16):
                want = oracle.rope_cos_sin(theta, p)
                # fp64 value rounded once to fp32: within half an fp32 ulp
                assert np.all(np.abs(tab[p] - want) <= np.abs(want) * 2.0 ** -24 + 1e-45)


def test_layout_byte_counts_match_the_pages():
    # colibri "System One mode and prompt reuse": a Flash ring snapshot is
    # 39 layers x 128 slots x 8 heads x (192 + 128) floats, "about 50 MB".
    snap = 39 * kvr.RingLayout.bytes_per_layer(1, 8, elem_bytes=4)
    assert 48e6 < snap < 53e6
    # gaudi-cookbook "Windowed KV groups": 6,912 B per token per card for the
    # 9 global layers (bf16, V padded to 192, one KV head per card at TP8)
    # against 36,864 B when all 48 layers keep full-length KV.
    assert 9 * kvr.PagedLayout.bytes_per_token(1, v_width=192) == 6912
    assert 48 * kvr.PagedLayout.bytes_per_token(1, v_width=192) == 36864
    # colibri "Pro": 0.78 GiB of f32 KV for 10 full layers at 8k context
    # (8 KV heads there) -- same per-token arithmetic.
    gib = 10 * 8192 * kvr.PagedLayout.bytes_per_token(8, elem_bytes=4) / 2 ** 30
    assert abs(gib - 0.78) < 0.01


def test_pages_management_host_validation(L):
    P = ctypes.c_void_p(FAKE)
    rel = L.kv_pages_release_window
    # n < 0, empty pool shapes, window < 1, negative capacity, NULL table / counter
    assert rel(P, 4, 16, 64, 64, P, P, None, -1, 128, P, P, 8, None) == -1
    assert rel(P, 0, 16, 64, 64, P, P, None, 1, 128, P, P, 8, None) == -1
    assert rel(P, 4, 16, 64, 64, P, P, None, 1, 0, P, P, 8, None) == -1
    assert rel(P, 4, 16, 64, 64, P, P, None, 1, 128, P, P, -1, None) == -1
    assert rel(None, 4, 16, 64, 64, P, P, None, 1, 128, P, P, 8, None) == -1
    assert rel(P, 4, 16, 64, 64, P, P, None, 1, 128, P, None, 8, None) == -1
    # NULL seqs / next_pos / free_ids (with a capacity)
    assert rel(P, 4, 16, 64, 64, None, P, None, 1, 128, P, P, 8, None) == -1
    assert rel(P, 4, 16, 64, 64, P, P, None, 1, 128, None, P, 8, None) == -1
    # n = 0 launches nothing
    assert rel(P, 4, 16, 64, 64, None, None, None, 0, 128, None, P, 0, None) == 0
    gat = L.kv_ring_gather_pages
    ring8 = _ring()
    # pages must be PAGED, ring must be RING, and their KV head counts agree
    assert gat(ctypes.byref(ring8), ctypes.byref(ring8), P, P, P, 1, None) == -1
    assert gat(ctypes.byref(_paged(num_kv_heads=8)), ctypes.byref(_paged(num_kv_heads=8)), P, P, P, 1, None) == -1
    assert gat(ctypes.byref(_paged()), ctypes.byref(ring8), P, P, P, 1, None) == -1
    pg8 = _paged(num_kv_heads=8)
    assert gat(ctypes.byref(pg8), ctypes.byref(ring8), P, P, P, -1, None) == -1
    assert gat(ctypes.byref(pg8), ctypes.byref(ring8), None, P, P, 1, None) == -1
    assert gat(ctypes.byref(pg8), ctypes.byref(ring8), None, None, None, 0, None) == 0


def _items_cap(B, hkv, max_ctx, sms=152):
    """The most items the decode split plan can give: a candidate of about k
    items per resident CTA (two per SM, k <= 8) gives at most 8 x 2 x SMs plus
    one partial split per (sequence, KV head); a split length capped at 8448
    keys at most ceil(max_ctx / 8448) splits per sequence."""
    units = B * hkv
    return max(8 * 2 * sms + units, units * -(-max_ctx // 8448))


@pytest.mark.parametrize("B,max_ctx", [(64, 32769), (1, 131073), (4, 32769), (16, 524289), (128, 1 << 20),
                                        (700, 2048), (64, 8193)])
def test_decode_workspace_follows_the_split_plan(L, B, max_ctx):
    # workspace = the plan (split length, item count, per-sequence item prefix
    # after 64 header words), then fp32 (m, l) and 128 numerators per (item, q
    # head of the group), each part rounded up to 256 bytes; no GPU here, so
    # the library plans for 152 SMs
    hq, hkv = 64, 4
    items = _items_cap(B, hkv, max_ctx)
    G = hq // hkv
    up = lambda x: -(-x // 256) * 256
    want = up((64 + B + 1) * 4) + up(items * G * 2 * 4) + up(items * G * 128 * 4)
    assert L.full_attn_decode_workspace_size(B, hq, hkv, max_ctx) == want
