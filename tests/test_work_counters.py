"""The bench's algorithmic work counters (the numerators of every roofline
fraction) against what the pages and plain arithmetic fix.

Xiaomi "Full-Pipeline Inference Optimization for MiMo-V2.5 Series",
section 1.1: with 10 full-attention and 60 windowed layers (window 128), the
attention compute of the hybrid stack is about 1/7 of an all-full stack at
long context; section 2.1: the KV cache shrinks by about the same factor."""
import pytest

import bench


@pytest.mark.parametrize("ctx", [131072, 1 << 20])

def test_hybrid_decode_bytes_are_one_seventh_of_full_at_long_context(ctx):
    # decode: K/V bytes read per step by 10 full + 60 windowed layers vs 70 full
    hyb = 10 * bench.layer_kv_bytes([ctx], 4) + 60 * bench.layer_kv_bytes([ctx], 4, window=128)
    full = 70 * bench.layer_kv_bytes([ctx], 4)
    assert hyb / full == pytest.approx(1 / 7, rel=128 * 6 / ctx + 1e-12)
    assert hyb / full > 1 / 7


def test_hybrid_prefill_flops_are_one_seventh_of_full_at_long_context():
    P0, C = 1 << 20, 8192
    hyb = 10 * bench.prefill_pairs(P0, C) + 60 * bench.prefill_pairs(P0, C, window=128)
    full = 70 * bench.prefill_pairs(P0, C)
    assert hyb / full == pytest.approx(1 / 7, rel=1e-3)


def test_prefill_pairs_brute_force():
    # every (row, key) pair counted one by one on small chunks
    for P0, C, w in [(0, 5, None), (7, 9, None), (0, 200, 128), (130, 20, 128), (3, 300, 128)]:
        brute = sum(1 for i in range(C) for j in range(P0 + i + 1) if w is None or j > P0 + i - w)
        assert bench.prefill_pairs(P0, C, w) == brute


def test_workload_numbers_of_the_configs():
    # the bench's prefill work (8192-token chunk on 122880 cached, 64 q heads)
    assert bench.attn_flops(bench.prefill_pairs(122880, 8192), 64) == 42606243348480
    assert bench.attn_flops(bench.prefill_pairs(122880, 8192, 128), 64) == 64 * 8192 * 128 * 2 * 320
    # flash decode: 64 sequences x 32769 positions x 4 KV heads x 640 B = 5.37 GB
    assert bench.layer_kv_bytes([32769] * 64, 4) == 64 * 32769 * 4 * 640
    # a windowed layer reads at most 128 positions per (sequence, KV head)
    assert bench.layer_kv_bytes([100, 5000], 8, window=128) == (100 + 128) * 8 * 640
    # the windowed share of a 60:10 stack at 1M context is under 0.1% of the full layers' bytes
    w = 60 * bench.layer_kv_bytes([1 << 20], 8, window=128)
    f = 10 * bench.layer_kv_bytes([1 << 20], 4)
    assert w / f < 2e-3
