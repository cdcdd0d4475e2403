"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Each test names what fixes the expected value: a number the pages print, a
closed form, a textbook reduction (the sink as a zero-valued extra key; no
sink = library SDPA), brute force on tiny inputs, or an invariant the pages
state (the window is exactly the last 128 positions; V zero-padded to 192
changes nothing; n blocks with sink - log(n) add up to one sink term).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import dense

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SCALE = 1.0 / math.sqrt(192.0)


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _rand_bf16(shape, seed, scale=1.0, shift=None):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(shape, generator=g) * scale
    if shift is not None:
        x = x + shift
    return x.to(torch.bfloat16)


def _case(nq, hq, nk, hkv, seed, k0=0, qpos=None):
    q = _rand_bf16((nq, hq, 192), seed)
    k = _rand_bf16((nk, hkv, 192), seed + 1)
    v = _rand_bf16((nk, hkv, 128), seed + 2)
    if qpos is None:
        qpos = np.arange(k0 + nk - nq, k0 + nk, dtype=np.int64)
    sinks = (1.0 + 0.5 * torch.randn(hq, generator=torch.Generator().manual_seed(seed + 3))).double().numpy()
    return _bits(q), np.asarray(qpos, dtype=np.int64), _bits(k), _bits(v), sinks


# ---------------------------------------------------------------- rounding

def test_round_bf16_matches_torch_on_fp32_values():
    # torch's float32 -> bfloat16 cast is round-to-nearest-even; on values that
    # are exactly float32 no double rounding is involved.
    g = torch.Generator().manual_seed(7)
    x = (torch.randn(20000, generator=g) * torch.exp(torch.randn(20000, generator=g) * 4)).float()
    want = _bits(x.to(torch.bfloat16))
    got = np.array([oracle.round_bf16(float(v)) for v in x.tolist()], dtype=np.uint16)
    assert np.array_equal(got, want)


def test_round_bf16_ties_to_even():
    assert oracle.round_bf16(1.0 + 2.0 ** -8) == 0x3F80          # tie -> even (1.0)
    assert oracle.round_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82      # tie -> even (1 + 2^-6)
    assert oracle.round_bf16(-(1.0 + 2.0 ** -8 + 2.0 ** -30)) == 0xBF81  # above tie -> up


# ---------------------------------------------------------------- RoPE

def test_rope_rotate_half_pairs_dim_i_with_i_plus_32():
    # colibri "What the engine implements": rotate-half on the first 64 dims.
    # A unit vector on dim i rotates into dim i+32 (not i+1, as an interleaved
    # layout would).  theta=1e4, i=16: inv_freq = 1e4^(-1/2) = 0.01 exactly in
    # real arithmetic, so position 100 has angle 1 rad.
    x = np.zeros((2, 192), dtype=np.uint16)
    x[0, 16] = 0x3F80   # e_16
    x[1, 48] = 0x3F80   # e_48
    out = oracle.rope_heads(x, np.array([100, 100]), 1e4)
    c, s = math.cos(1.0), math.sin(1.0)
    assert abs(out[0, 16] - c) < 1e-14 and abs(out[0, 48] - s) < 1e-14
    assert abs(out[1, 16] + s) < 1e-14 and abs(out[1, 48] - c) < 1e-14
    assert np.count_nonzero(out[0]) == 2 and np.count_nonzero(out[1]) == 2


def test_rope_fastest_frequency_angle_is_position():
    # gaudi-cookbook "The RoPE fix": the fastest frequency's angle equals the
    # position in radians.  Both thetas of the hybrid layers.
    for theta in (1e4, 1e7):
        for p in (0, 1, 7, 131071, 524288):
            cs = oracle.rope_cos_sin(theta, p)
            assert cs[0, 0] == math.cos(float(p)) and cs[0, 1] == math.sin(float(p))


def test_rope_slowest_frequency_closed_form():
    # inv_freq_31 = theta^(-62/64): for theta = 1e4 that is 10^(-3.875).
    cs = oracle.rope_cos_sin(1e4, 1000)
    assert abs(cs[31, 0] - math.cos(1000 * 10 ** -3.875)) < 1e-12
    cs = oracle.rope_cos_sin(1e7, 1000)
    assert abs(cs[31, 0] - math.cos(1000 * 10 ** (-7 * 62 / 64))) < 1e-12


def test_rope_golden_cos_200000():
    with open(os.path.join(GOLDEN, "rope_cos_200000.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    for pos, i, val, tol in rows:
        cs = oracle.rope_cos_sin(1e4, int(pos))
        assert abs(cs[int(i), 0] - float(val)) <= float(tol)


def test_rope_identity_at_zero_and_passthrough_dims():
    x = _bits(_rand_bf16((5, 192), 11))
    out = oracle.rope_heads(x, np.zeros(5, dtype=np.int64), 1e7)
    assert np.array_equal(out, dense.bf16_bits_to_f64(x))
    out = oracle.rope_heads(x, np.array([3, 99, 1000, 70000, 524287]), 1e4)
    assert np.array_equal(out[:, 64:], dense.bf16_bits_to_f64(x)[:, 64:])


def test_rope_norm_and_relative_position():
    x = _bits(_rand_bf16((2, 192), 12))
    a = oracle.rope_heads(x[:1], np.array([37]), 1e4)[0]
    b = oracle.rope_heads(x[1:], np.array([5]), 1e4)[0]
    a2 = oracle.rope_heads(x[:1], np.array([37 + 9001]), 1e4)[0]
    b2 = oracle.rope_heads(x[1:], np.array([5 + 9001]), 1e4)[0]
    raw = dense.bf16_bits_to_f64(x)
    for i in range(32):   # each (i, i+32) pair keeps its norm
        assert abs(math.hypot(a[i], a[i + 32]) - math.hypot(raw[0, i], raw[0, i + 32])) < 1e-12
    assert abs(a @ b - a2 @ b2) < 1e-10


# ---------------------------------------------------------------- KV store

def test_kv_store_bf16_value_scale_and_passthrough():
    k = _bits(_rand_bf16((9, 2, 192), 21))
    v = _bits(_rand_bf16((9, 2, 128), 22))
    pos = np.arange(100, 109)
    ko, vo = oracle.kv_store_bf16(k, v, pos, 1e4, 0.5)
    assert np.array_equal(ko[..., 64:], k[..., 64:])       # dims 64..191 stored bit-exact
    # scale 0.5 is exact in binary: v' must equal v/2 bit for bit
    half = _bits((torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).float() * 0.5).to(torch.bfloat16))
    assert np.array_equal(vo, half)
    # rotated dims: round-to-nearest of the fp64 rotation
    ref = oracle.rope_heads(k.reshape(-1, 192), np.repeat(pos, 2), 1e4).reshape(9, 2, 192)
    got = dense.bf16_bits_to_f64(ko)
    assert np.all(np.abs(got[..., :64] - ref[..., :64]) <= np.abs(ref[..., :64]) * 2.0 ** -8 + 1e-38)


# ---------------------------------------------------------------- attention

@pytest.mark.parametrize("window,use_sink", [(0, False), (128, True), (128, False), (16, True)])
def test_c_oracle_matches_dense_formulation(window, use_sink):
    q, qpos, k, v, sinks = _case(nq=40, hq=8, nk=300, hkv=2, seed=31)
    s = sinks if use_sink else None
    a = oracle.attend_seq(q, qpos, k, v, 0, 1e4, 0.707, SCALE, window, s)
    b = dense.attend(q, qpos, k, v, 0, 1e4, 0.707, SCALE, window, s)
    assert np.max(np.abs(a - b)) <= 1e-12 * max(1.0, np.max(np.abs(b)))


def test_no_sink_equals_torch_sdpa_with_band_mask():
    # Textbook reduction: without a sink, windowed attention is SDPA with a
    # band mask; with window 0 it is causal SDPA.  Library routine in fp64.
    q, qpos, k, v, _ = _case(nq=64, hq=4, nk=256, hkv=2, seed=41)
    qr = oracle.rope_heads(q.reshape(-1, 192), np.repeat(qpos, 4), 1e7).reshape(64, 4, 192)
    kr = oracle.rope_heads(k.reshape(-1, 192), np.repeat(np.arange(256), 2), 1e7).reshape(256, 2, 192)
    vr = dense.bf16_bits_to_f64(v) * 0.612
    for window in (0, 128, 7):
        allowed = np.arange(256)[None, :] <= qpos[:, None]
        if window:
            allowed &= np.arange(256)[None, :] > qpos[:, None] - window
        Q = torch.from_numpy(qr).permute(1, 0, 2)
        K = torch.from_numpy(kr).permute(1, 0, 2).repeat_interleave(2, dim=0)
        V = torch.from_numpy(vr).permute(1, 0, 2).repeat_interleave(2, dim=0)
        want = torch.nn.functional.scaled_dot_product_attention(
            Q, K, V, attn_mask=torch.from_numpy(allowed), scale=SCALE).permute(1, 0, 2).numpy()
        got = oracle.attend_seq(q, qpos, k, v, 0, 1e7, 0.612, SCALE, window, None)
        assert np.max(np.abs(got - want)) < 1e-12


def test_brute_force_tiny_by_hand():
    # One query at position 2, keys at 0..2, all mass on dims >= 64 so RoPE
    # leaves them alone.  Logits by hand: q.k_j / sqrt(192).
    q = np.zeros((1, 1, 192), dtype=np.uint16)
    k = np.zeros((3, 1, 192), dtype=np.uint16)
    v = np.zeros((3, 1, 128), dtype=np.uint16)
    q[0, 0, 100] = 0x4000          # 2.0
    k[0, 0, 100] = 0x3F80          # 1.0   -> raw 2
    k[1, 0, 100] = 0xBF80          # -1.0  -> raw -2
    k[2, 0, 100] = 0x4040          # 3.0   -> raw 6
    for j in range(3):
        v[j, 0, 0] = [0x3F80, 0x4000, 0x4040][j]   # 1, 2, 3
    sink = 0.25
    e = [math.exp(r / math.sqrt(192)) for r in (2.0, -2.0, 6.0)]
    want = 0.5 * (1 * e[0] + 2 * e[1] + 3 * e[2]) / (math.exp(sink) + sum(e))
    got = oracle.attend_seq(q, [2], k, v, 0, 1e4, 0.5, SCALE, 128, [sink])
    assert abs(got[0, 0, 0] - want) < 1e-15 and np.count_nonzero(got) == 1
    got = oracle.attend_seq(q, [2], k, v, 0, 1e4, 0.5, SCALE, 0, None)
    assert abs(got[0, 0, 0] - 0.5 * (e[0] + 2 * e[1] + 3 * e[2]) / sum(e)) < 1e-15


def test_sink_joins_denominator_only():
    # colibri "What the engine implements": with the sink, o is the no-sink
    # output times Z/(Z + e^sink) -- nothing else changes.
    q, qpos, k, v, sinks = _case(nq=20, hq=4, nk=200, hkv=1, seed=51)
    a, sa = oracle.attend_seq(q, qpos, k, v, 0, 1e4, 0.707, SCALE, 128, None, with_stats=True)
    b = oracle.attend_seq(q, qpos, k, v, 0, 1e4, 0.707, SCALE, 128, sinks)
    z = sa[..., 1] * np.exp(sa[..., 0])                    # sum_j e^{s_j}
    factor = z / (z + np.exp(sinks)[None, :])
    assert np.max(np.abs(b - a * factor[..., None])) < 1e-13


def test_sink_limits():
    q, qpos, k, v, _ = _case(nq=5, hq=2, nk=64, hkv=1, seed=61)
    big = oracle.attend_seq(q, qpos, k, v, 0, 1e4, 0.707, SCALE, 128, [800.0, 800.0])
    assert np.max(np.abs(big)) < 1e-300
    neg = oracle.attend_seq(q, qpos, k, v, 0, 1e4, 0.707, SCALE, 128, [-800.0, -800.0])
    none = oracle.attend_seq(q, qpos, k, v, 0, 1e4, 0.707, SCALE, 128, None)
    assert np.max(np.abs(neg - none)) < 1e-13


def test_window_is_exactly_the_last_128_positions():
    # gaudi-cookbook "What was built": exactly the last 128 positions.  The
    # query at p sees p-127..p: the key at p-128 must not matter, p-127 must.
    nk, p = 400, 399
    q, _, k, v, sinks = _case(nq=1, hq=2, nk=nk, hkv=1, seed=71)
    base = oracle.attend_seq(q, [p], k, v, 0, 1e4, 0.707, SCALE, 128, sinks)
    k2 = k.copy(); k2[p - 128] ^= 0x0040; v2 = v.copy(); v2[p - 128] ^= 0x0040
    assert np.array_equal(oracle.attend_seq(q, [p], k2, v2, 0, 1e4, 0.707, SCALE, 128, sinks), base)
    k3 = k.copy(); k3[p - 127] ^= 0x0040; v3 = v.copy(); v3[p - 127] ^= 0x0040
    assert not np.array_equal(oracle.attend_seq(q, [p], k3, v3, 0, 1e4, 0.707, SCALE, 128, sinks), base)
    # a window of 128 with fewer than 128 keys before it is causal attention
    q, qpos, k, v, _ = _case(nq=100, hq=2, nk=100, hkv=1, seed=72)
    assert np.array_equal(oracle.attend_seq(q, qpos, k, v, 0, 1e4, 0.707, SCALE, 128, None),
                          oracle.attend_seq(q, qpos, k, v, 0, 1e4, 0.707, SCALE, 0, None))


def test_zero_padding_v_to_192_changes_nothing():
    # gaudi-cookbook "What was built": V zero-padded to 192, extra output
    # columns dropped -- exact.  Checked on the dense formulation, bit for bit.
    q, qpos, k, v, sinks = _case(nq=30, hq=4, nk=150, hkv=2, seed=81)
    a = dense.attend(q, qpos, k, v, 0, 1e4, 0.707, SCALE, 128, sinks)
    b = dense.attend(q, qpos, k, v, 0, 1e4, 0.707, SCALE, 128, sinks, pad_v_to=192)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("n", [1, 2, 3, 7])
def test_sink_minus_log_n_per_block_is_one_sink(n):
    # gaudi-cookbook "What was built": each of a sequence's n blocks gets
    # sink - log(n) so the n copies add up to one sink term.  Merge the blocks
    # by log-sum-exp and compare with the one-block result.
    p = 127 + 90
    q, _, k, v, sinks = _case(nq=1, hq=4, nk=p + 1, hkv=1, seed=91)
    want = oracle.attend_seq(q, [p], k, v, 0, 1e4, 0.707, SCALE, 128, sinks)
    edges = np.linspace(p - 127, p + 1, n + 1).astype(int)
    outs, stats = [], []
    for a, b in zip(edges[:-1], edges[1:]):
        o, s = oracle.attend_seq(q, [p], k[a:b], v[a:b], a, 1e4, 0.707, SCALE, 128,
                                 sinks - math.log(n), with_stats=True)
        outs.append(o); stats.append(s)
    M = np.max([s[..., 0] for s in stats], axis=0)
    w = [s[..., 1] * np.exp(s[..., 0] - M) for s in stats]
    got = sum(o * wi[..., None] for o, wi in zip(outs, w)) / sum(w)[..., None]
    assert np.max(np.abs(got - want)) < 1e-13


def test_split_k_merge_of_a_full_layer():
    # Full layer, no sink: splitting the keys and merging by log-sum-exp
    # gives the unsplit result.
    p = 999
    q, _, k, v, _ = _case(nq=1, hq=4, nk=p + 1, hkv=2, seed=95)
    want = oracle.attend_seq(q, [p], k, v, 0, 1e7, 0.707, SCALE, 0, None)
    edges = [0, 1, 250, 256, 700, 1000]
    outs, stats = [], []
    for a, b in zip(edges[:-1], edges[1:]):
        o, s = oracle.attend_seq(q, [p], k[a:b], v[a:b], a, 1e7, 0.707, SCALE, 0, None, with_stats=True)
        outs.append(o); stats.append(s)
    M = np.max([s[..., 0] for s in stats], axis=0)
    w = [s[..., 1] * np.exp(s[..., 0] - M) for s in stats]
    got = sum(o * wi[..., None] for o, wi in zip(outs, w)) / sum(w)[..., None]
    assert np.max(np.abs(got - want)) < 1e-13


def test_value_scale_is_linear():
    q, qpos, k, v, sinks = _case(nq=10, hq=2, nk=140, hkv=1, seed=101)
    a = oracle.attend_seq(q, qpos, k, v, 0, 1e4, 1.0, SCALE, 128, sinks)
    b = oracle.attend_seq(q, qpos, k, v, 0, 1e4, 0.612, SCALE, 128, sinks)
    assert np.max(np.abs(b - 0.612 * a)) < 1e-14


def test_gqa_head_h_reads_kv_head_h_over_group():
    q, qpos, k, v, sinks = _case(nq=6, hq=8, nk=60, hkv=2, seed=111)
    full = oracle.attend_seq(q, qpos, k, v, 0, 1e4, 0.707, SCALE, 128, sinks)
    for h in range(8):
        one = oracle.attend_seq(q[:, h:h + 1], qpos, k[:, h // 4:h // 4 + 1], v[:, h // 4:h // 4 + 1],
                                0, 1e4, 0.707, SCALE, 128, sinks[h:h + 1])
        assert np.array_equal(one[:, 0], full[:, h])


def test_shifted_inputs_have_the_stated_logit_statistics():
    # The workload: scaled q.k logits near -25 with std 3, sinks ~ N(1, 0.5).
    from sinks_kv_ring_gb300.synth import Synth
    s = Synth(1000, dist="shifted")
    q = s.q(64, 8, 2)
    k = s.k(256, 2)
    qr = oracle.rope_heads(q.reshape(-1, 192), np.full(64 * 8, 300), 1e4).reshape(64, 8, 192)
    kr = oracle.rope_heads(k.reshape(-1, 192), np.arange(256).repeat(2), 1e4).reshape(256, 2, 192)
    logits = np.einsum("qgd,kd->qgk", qr[:, :4], kr[:, 0]) * SCALE
    assert abs(logits.mean() + 25.0) < 0.5 and abs(logits.std() - 3.0) < 0.3
    sk = Synth(1000).sinks(20000).numpy()
    assert abs(sk.mean() - 1.0) < 0.02 and abs(sk.std() - 0.5) < 0.02


# --------------------------------------------------------------------------- paged windowed pool

def _read_release_example():
    cfg, table, calls, final = {}, {}, [], {}
    for line in open(os.path.join(GOLDEN, "pages_release_example.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("table ") or line.startswith("final "):
            head, vals = line.split(":")
            (table if line.startswith("table") else final)[int(head.split()[1])] = [int(x) for x in vals.split()]
        elif line.startswith("call "):
            f = dict(kv.split("=") for kv in line[5:].split())
            ints = lambda s: [int(x) for x in s.split(",")] if s else []
            calls.append((ints(f["seqs"]), ints(f["next_pos"]), ints(f["released"]), ints(f["lo"]), int(f["flags"])))
        else:
            k, v = line.split()
            cfg[k] = int(v)
    return cfg, [table[s] for s in sorted(table)], calls, [final[s] for s in sorted(final)]


def test_release_window_worked_example():
    from oracle import pages
    cfg, table, calls, final = _read_release_example()
    lo, ids, count = [0] * len(table), [], 0
    for seqs, nxt, want_rel, want_lo, want_flags in calls:
        table, lo, ids, new_count, flags = pages.release_window(
            table, cfg["num_blocks"], cfg["block_size"], seqs, nxt, cfg["window"], lo=lo,
            free_ids=ids, free_count=count, free_cap=cfg["free_cap"])
        assert ids[count:new_count] == want_rel
        assert lo == want_lo and flags == want_flags
        count = new_count
    assert table == final


def _attended_by_later_query(block_index, bs, next_pos, window):
    """Brute force: does any query at q >= next_pos read a position of the block?"""
    first, last = block_index * bs, block_index * bs + bs - 1
    for q in range(next_pos, max(next_pos, last) + 1):
        for p in range(max(0, q - window + 1), q + 1):
            if first <= p <= last:
                return True
    return False


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_release_window_against_brute_force_windows(seed):
    # every released block is read by no later query; every kept valid block
    # at or past lo is read by one (so nothing that could go stays)
    from oracle import pages
    rng = np.random.default_rng(seed)
    S, mb, bs, W = 5, 12, 4, 8
    nblk = S * mb
    ids = rng.permutation(nblk)[: S * mb].reshape(S, mb).tolist()
    for s in range(S):
        for b in range(mb):
            if rng.random() < 0.15:
                ids[s][b] = -1
    lo = [int(x) for x in rng.integers(0, 3, S)]
    nxt = [int(x) for x in rng.integers(0, mb * bs + 10, S)]
    table, lo2, free, cnt, flags = pages.release_window(ids, nblk, bs, list(range(S)), nxt, W, lo=lo)
    assert flags == 0 and cnt == len(free)
    freed = set(free)
    for s in range(S):
        for b in range(mb):
            before, after = ids[s][b], table[s][b]
            if before < 0:
                assert after == before
            elif b < lo[s]:
                assert after == before and before not in freed
            elif _attended_by_later_query(b, bs, nxt[s], W):
                assert after == before and before not in freed
            else:
                assert after == -1 and before in freed
        assert lo2[s] >= lo[s]
    # released ids come in (sequence, block index) order
    order = [ids[s][b] for s in range(S) for b in range(mb) if ids[s][b] >= 0 and table[s][b] == -1]
    assert free == order


def test_ring_from_pages_equals_appending_in_order():
    # colibri "System One mode and prompt reuse": the ring after appending
    # positions 0..E-1 one by one, slot p mod 128 <- row p, tag p
    from oracle import pages
    rng = np.random.default_rng(7)
    hkv, bs, mb = 2, 16, 24
    nblk = 2 * mb
    pk = rng.integers(0, 1 << 16, (nblk, hkv, bs, 192), dtype=np.uint16)
    pv = rng.integers(0, 1 << 16, (nblk, hkv, bs, 128), dtype=np.uint16)
    table = rng.permutation(nblk).reshape(2, mb).tolist()
    for end in [0, 1, 77, 128, 129, 300, 383]:
        k0 = rng.integers(0, 1 << 16, (hkv, 128, 192), dtype=np.uint16)
        v0 = rng.integers(0, 1 << 16, (hkv, 128, 128), dtype=np.uint16)
        t0 = np.full(128, -1, dtype=np.int32)
        wk, wv, wt = k0.copy(), v0.copy(), t0.copy()
        for p in range(end):
            b = table[1][p // bs]
            wk[:, p % 128] = pk[b, :, p % bs]
            wv[:, p % 128] = pv[b, :, p % bs]
            wt[p % 128] = p
        k, v, t, flags = pages.ring_from_pages(pk, pv, table, bs, 1, end, k0, v0, t0)
        assert flags == 0
        assert np.array_equal(t, wt) and np.array_equal(k, wk) and np.array_equal(v, wv)
