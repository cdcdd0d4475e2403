"""Benchmark of the hybrid-SWA attention hot path on GB300.

Default workload (--workload flash_decode): Flash-shaped decode, batch 64,
64 q heads; one windowed layer (8 KV heads, 128-slot ring, sink) and one
full-attention layer (4 KV heads, 32768 cached tokens + the new one).  One
step = the KV write of the new token into both layers (RoPE + value scale)
+ swa_sink_decode + full_attn_decode, for the whole batch.  The JSON line
also carries a chunked-prefill measurement (8192-token chunk on 122880
cached tokens, one full + one windowed layer) under "prefill".

The line also carries "mtp": the same batch verifying a 4-token draft per
sequence (multi-token prediction) through the varlen calls.

Other workloads: prefill, long_decode (batch 16 at 524288 tokens), mtp_decode,
pro_true (pro_mixed with the Pro's own head counts: 128 q heads, 8 KV heads on both kinds),
long_stack (batch 16 at 524288 tokens through a 48-layer stack, 9 full : 39 windowed),
pro_mixed (128 ragged sequences through a 70-layer stack, 10 full : 60
windowed), tiny (1 sequence, 512 tokens).

All inputs are synthetic (seeded), drawn on the device.  Timing: CUDA events
on the launching stream; inputs larger than L2 (the full pool is GBs; the
windowed layer rotates over enough distinct rings to exceed L2).  Prints one
JSON line on rank 0.  `--impl reference` times the fp64 CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

SCALE = 1.0 / math.sqrt(192.0)
METRIC = "decode attn tokens/s + HBM GB/s; prefill attn TFLOP/s; % of GB300 roofline"
MTP_MAX = 4
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# --------------------------------------------------------------------------- helpers

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


NOMINAL = {"hbm": 7900.0, "tensor": 2250.0}  # GB300 data-sheet HBM3e GB/s and dense bf16 TFLOP/s


def with_nominal(roof: dict) -> dict:
    """Add the fraction of the nominal (data-sheet) peak beside the measured one."""
    roof["nominal_peak"] = NOMINAL[roof["bound"]]
    roof["frac_of_nominal"] = round(roof["achieved"] / NOMINAL[roof["bound"]], 4)
    return roof


def kernel_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if the
    kernel's source has not changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f).get(kernel)
    if not d:
        return None
    src = os.path.join(ROOT, "sinks_kv_ring_gb300", "csrc", d["source"])
    if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != d["sha256_16"]:
        return None
    return d["bytes_per_launch"]


class Clocks:
    """nvidia-smi sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 9:
                rows.append(f)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def rank_seed(base: int, rank: int) -> int:
    """Each rank draws its own batch (weak scaling: per-GPU work is fixed)."""
    return base + rank


def max_over_ranks(vals, world: int, device):
    """Element-wise max over ranks (timings); the only collective of the bench,
    outside the attention data path."""
    if world <= 1:
        return [float(v) for v in vals]
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_throughput(units_per_rank: float, world: int, ms_max: float) -> float:
    """Whole-job units per second: all ranks' units over the slowest rank's time."""
    return world * units_per_rank / (ms_max / 1e3)


def flush_l2(buf):
    buf.add_(1)


class EventTimer:
    """Per-call durations of one kind of launch, from CUDA events recorded on
    the launching stream."""

    def __init__(self):
        self.pairs = []

    def start(self, stream):
        a = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        return a

    def stop(self, a, stream):
        b = torch.cuda.Event(enable_timing=True)
        b.record(stream)
        self.pairs.append((a, b))

    def mean_ms(self):
        if not self.pairs:
            return None
        return sum(a.elapsed_time(b) for a, b in self.pairs) / len(self.pairs)


# --------------------------------------------------------------------------- work counters

KV_BYTES = (192 + 128) * 2   # K and V of one position and KV head, bf16


def layer_kv_bytes(contexts, hkv: int, window: int | None = None) -> int:
    """K/V bytes one decode step must read from one layer: every context
    position (full layer) or the last `window` ones (windowed layer)."""
    return sum(min(window, c) if window else c for c in contexts) * hkv * KV_BYTES


def prefill_pairs(P0: int, C: int, window: int | None = None) -> int:
    """(query, key) pairs of a C-row chunk on P0 cached positions (causal; the
    last `window` keys of each row for a windowed layer)."""
    if window is None:
        return C * P0 + C * (C + 1) // 2
    return sum(min(window, P0 + i + 1) for i in range(C))


def attn_flops(pairs: int, hq: int) -> int:
    """Multiply-adds x 2 of S = QK^T (192) and O = PV (128) over the pairs."""
    return hq * pairs * 2 * (192 + 128)


# --------------------------------------------------------------------------- workloads

def _fill_pool(kvr, pool, syn, seqs, ctx, table, vscale, chunk=65536):
    dev = pool.k.device
    hkv = pool.num_kv_heads
    for s, n in zip(seqs, ctx):
        for lo in range(0, n, chunk):
            hi = min(n, lo + chunk)
            k = syn.k(hi - lo, hkv, seq=s, start=lo)
            v = syn.v(hi - lo, hkv, seq=s, start=lo)
            pos = torch.arange(lo, hi, device=dev)
            sq = torch.full((hi - lo,), s, dtype=torch.int32, device=dev)
            kvr.kv_ring_append_rope(k, v, pos, sq, table, vscale, pool)


def _fill_rings(kvr, ring, syn, B, p, table, vscale):
    dev = ring.k.device
    hkv = ring.num_kv_heads
    lo = max(0, p - 127)
    n = p - lo
    if n <= 0:
        return
    for s in range(B):
        k = syn.k(n, hkv, seq=s, start=lo)
        v = syn.v(n, hkv, seq=s, start=lo)
        kvr.kv_ring_append_rope(k, v, torch.arange(lo, p, device=dev), torch.full((n,), s, dtype=torch.int32, device=dev),
                                table, vscale, ring)


class DecodeWorkload:
    """One decode step over one windowed + one full-attention layer."""

    def __init__(self, kvr, B=64, hq=64, hkv_swa=8, hkv_full=4, ctx=32768, vscale=0.707, seed=1001,
                 swa_copies=None, device="cuda"):
        from sinks_kv_ring_gb300.synth import Synth
        self.kvr, self.B, self.hq, self.ctx = kvr, B, hq, ctx
        self.hkv_swa, self.hkv_full, self.vscale = hkv_swa, hkv_full, vscale
        self.p = ctx                      # the new token's position; context = ctx + 1
        self.max_ctx = ctx + 1
        dev = device
        # tables (and pool capacity) also cover a draft of up to MTP_MAX tokens at p
        self.t4 = kvr.rope_table(1e4, ctx + MTP_MAX, device=dev)
        self.t7 = kvr.rope_table(1e7, ctx + MTP_MAX, device=dev)
        syn = Synth(seed, dist="shifted", device=dev)
        self.pool = kvr.PagedLayout.contiguous(B, hkv_full, ctx + MTP_MAX, block_size=64, device=dev, zero=False)
        _fill_pool(kvr, self.pool, Synth(seed, layer=1, device=dev), range(B), [ctx] * B, self.t7, vscale)
        ring_bytes = kvr.RingLayout.bytes_per_layer(B, hkv_swa)
        if swa_copies is None:
            swa_copies = max(1, min(64, math.ceil(4 * 129e6 / ring_bytes)))
        self.rings = []
        base = kvr.RingLayout.empty(B, hkv_swa, device=dev)
        _fill_rings(kvr, base, syn, B, self.p, self.t4, vscale)
        for i in range(swa_copies):
            self.rings.append(base if i == 0 else kvr.RingLayout(base.k.clone(), base.v.clone(), base.slot_pos.clone()))
        # per-step inputs: q of both layers, the new token's k/v in both layers
        self.q_swa = syn.q(B, hq, hkv_swa, seq=10_000)
        self.q_full = Synth(seed, layer=1, device=dev).q(B, hq, hkv_full, seq=10_000)
        self.k_swa, self.v_swa = syn.k(B, hkv_swa, seq=20_000), syn.v(B, hkv_swa, seq=20_000)
        self.k_full = Synth(seed, layer=1, device=dev).k(B, hkv_full, seq=20_000)
        self.v_full = Synth(seed, layer=1, device=dev).v(B, hkv_full, seq=20_000)
        self.pos = torch.full((B,), self.p, dtype=torch.int64, device=dev)
        self.seq = torch.arange(B, dtype=torch.int32, device=dev)
        self.sinks = syn.sinks(hq).to(dev)
        self.ws = torch.empty(kvr.full_attn_decode_workspace_size(B, hq, hkv_full, self.max_ctx), dtype=torch.uint8,
                              device=dev)
        self.out_swa = torch.empty(B, hq, 128, dtype=torch.bfloat16, device=dev)
        self.out_full = torch.empty(B, hq, 128, dtype=torch.bfloat16, device=dev)
        self.step_i = 0
        self.t_full = EventTimer()
        self.t_swa = EventTimer()
        self.launches_per_step = 5

    def bytes_full(self):
        # K/V bytes the full layer must read (every cached position, every KV head)
        return layer_kv_bytes([self.p + 1] * self.B, self.hkv_full)

    def bytes_swa(self):
        return layer_kv_bytes([self.p + 1] * self.B, self.hkv_swa, window=128)

    def step(self, stream, timed=False):
        kvr = self.kvr
        ring = self.rings[self.step_i % len(self.rings)]
        self.step_i += 1
        kvr.kv_ring_append_rope(self.k_swa, self.v_swa, self.pos, self.seq, self.t4, self.vscale, ring, stream=stream)
        kvr.kv_ring_append_rope(self.k_full, self.v_full, self.pos, self.seq, self.t7, self.vscale, self.pool,
                                stream=stream)
        a = self.t_swa.start(stream) if timed else None
        kvr.swa_sink_decode(self.q_swa, self.pos, self.seq, ring, self.sinks, self.t4, SCALE, out=self.out_swa,
                            stream=stream)
        if timed:
            self.t_swa.stop(a, stream)
            a = self.t_full.start(stream)
        kvr.full_attn_decode(self.q_full, self.pos, self.seq, self.pool, self.t7, SCALE, self.max_ctx,
                             workspace=self.ws, out=self.out_full, stream=stream)
        if timed:
            self.t_full.stop(a, stream)


class MtpStep:
    """Draft verification (multi-token prediction) on a decode workload's
    pool and rings: each of the B sequences checks q_len tokens at positions
    p .. p+q_len-1 in one pass per layer.  Step = KV write of the draft into
    the full pool and into the windowed staging rows + full_attn_prefill_varlen
    + swa_sink_prefill_varlen.  (Committing the accepted tokens to the ring is
    the decode step's ring append.)"""

    def __init__(self, work, q_len=4, seed=1005):
        from sinks_kv_ring_gb300.synth import Synth
        kvr, B, dev = work.kvr, work.B, work.pool.k.device
        assert 1 <= q_len <= MTP_MAX
        self.work, self.kvr, self.B, self.q_len = work, kvr, B, q_len
        T = B * q_len
        sf, ss = Synth(seed, layer=1, device=dev), Synth(seed, layer=0, device=dev)
        self.qf, self.qs = sf.q(T, work.hq, work.hkv_full, seq=30_000), ss.q(T, work.hq, work.hkv_swa, seq=30_000)
        self.kf, self.vf = sf.k(T, work.hkv_full, seq=40_000), sf.v(T, work.hkv_full, seq=40_000)
        self.ks, self.vs = ss.k(T, work.hkv_swa, seq=40_000), ss.v(T, work.hkv_swa, seq=40_000)
        self.pos = (work.p + torch.arange(q_len, device=dev)).repeat(B)
        self.seq_rows = torch.arange(B, dtype=torch.int32, device=dev).repeat_interleave(q_len)
        self.cu = torch.arange(0, T + 1, q_len, dtype=torch.int32, device=dev)
        self.P0 = torch.full((B,), work.p, dtype=torch.int64, device=dev)
        self.seq = torch.arange(B, dtype=torch.int32, device=dev)
        self.max_ctx = work.p + q_len
        self.stage = kvr.LinearLayout.empty(T, work.hkv_swa, device=dev)
        self.ws_f = torch.empty(kvr.full_attn_prefill_varlen_workspace_size(B, T, work.hq, work.hkv_full, self.max_ctx),
                                dtype=torch.uint8, device=dev)
        self.ws_s = torch.empty(kvr.swa_sink_prefill_varlen_workspace_size(B), dtype=torch.uint8, device=dev)
        self.out_f = torch.empty(T, work.hq, 128, dtype=torch.bfloat16, device=dev)
        self.out_s = torch.empty(T, work.hq, 128, dtype=torch.bfloat16, device=dev)
        self.t_full, self.t_swa = EventTimer(), EventTimer()
        self.step_i = 0
        self.launches_per_step = 2 + 3 + 2   # two appends, varlen full (plan, attention, merge), varlen windowed

    def bytes_full(self):
        w = self.work
        return self.B * w.hkv_full * self.max_ctx * (192 + 128) * 2

    def bytes_swa(self):
        w = self.work
        return self.B * w.hkv_swa * (min(128, w.p) + self.q_len) * (192 + 128) * 2

    def step(self, stream, timed=False):
        kvr, w = self.kvr, self.work
        ring = w.rings[self.step_i % len(w.rings)]
        self.step_i += 1
        kvr.kv_ring_append_rope(self.kf, self.vf, self.pos, self.seq_rows, w.t7, w.vscale, w.pool, stream=stream)
        kvr.kv_ring_append_rope(self.ks, self.vs, self.pos, None, w.t4, w.vscale, self.stage, stream=stream)
        a = self.t_full.start(stream) if timed else None
        kvr.full_attn_prefill_varlen(self.qf, self.cu, self.P0, self.seq, w.pool, w.t7, SCALE, self.max_ctx,
                                     workspace=self.ws_f, out=self.out_f, stream=stream)
        if timed:
            self.t_full.stop(a, stream)
            a = self.t_swa.start(stream)
        kvr.swa_sink_prefill_varlen(self.qs, self.cu, self.P0, self.seq, self.stage, ring, w.sinks, w.t4, SCALE,
                                    workspace=self.ws_s, out=self.out_s, stream=stream)
        if timed:
            self.t_swa.stop(a, stream)


def run_mtp(work, steps, warmup, q_len=4):
    stream = torch.cuda.current_stream()
    m = MtpStep(work, q_len=q_len)
    with Clocks(torch.cuda.current_device()) as ck:
        ms = timed_run(m, steps, warmup, stream, label="mtp")
    timed_run(m, steps, 0, stream, label="mtp_kernels", kernel_events=True)  # the per-call durations
    full = [(lambda st: m.kvr.full_attn_prefill_varlen(m.qf, m.cu, m.P0, m.seq, work.pool, work.t7, SCALE, m.max_ctx,
                                                       workspace=m.ws_f, out=m.out_f, stream=st))] * 10
    return m, ms, ck.summary(), graph_time_ms(full)


def mtp_result(m, ms, clocks, graph_full, hbm, world):
    ms_f, ms_s = m.t_full.mean_ms(), m.t_swa.mean_ms()
    gbs = m.bytes_full() / (ms_f / 1e3) / 1e9
    ggbs = m.bytes_full() / (graph_full / 1e3) / 1e9
    return {"workload": f"draft verification: batch {m.B}, {m.q_len} tokens per sequence at positions "
                        f"{m.work.p}..{m.work.p + m.q_len - 1}; same layers and pools as the decode step",
            "ms_per_step": round(ms, 4), "verified_tokens_per_s": round(job_throughput(m.B * m.q_len, world, ms), 1),
            "full_attn_prefill_varlen": {"ms": round(ms_f, 4), "GB/s": round(gbs, 1), "hbm_frac": round(gbs / hbm, 4),
                                         "bytes": m.bytes_full(), "graph_ms": round(graph_full, 4),
                                         "graph_GB/s": round(ggbs, 1), "graph_hbm_frac": round(ggbs / hbm, 4),
                                         "traffic": kernel_traffic("full_prefill_tc_kernel_varlen")},
            "swa_sink_prefill_varlen": {"ms": round(ms_s, 5), "bytes": m.bytes_swa(),
                                        "GB/s": round(m.bytes_swa() / (ms_s / 1e3) / 1e9, 1)},
            "clocks": clocks}


class PrefillWorkload:
    """One 8192-token chunk on top of 122880 cached tokens, one full + one windowed layer."""

    def __init__(self, kvr, P0=122880, C=8192, hq=64, hkv_full=4, hkv_swa=8, vscale=0.707, seed=1002, device="cuda"):
        from sinks_kv_ring_gb300.synth import Synth
        self.kvr, self.P0, self.C, self.hq = kvr, P0, C, hq
        self.hkv_full, self.hkv_swa, self.vscale = hkv_full, hkv_swa, vscale
        dev = device
        n = P0 + C
        self.t4 = kvr.rope_table(1e4, n, device=dev)
        self.t7 = kvr.rope_table(1e7, n, device=dev)
        sf, ss = Synth(seed, layer=1, device=dev), Synth(seed, layer=0, device=dev)
        self.pool = kvr.PagedLayout.contiguous(1, hkv_full, n, block_size=64, device=dev, zero=False)
        _fill_pool(kvr, self.pool, sf, [0], [P0], self.t7, vscale)
        self.ring = kvr.RingLayout.empty(1, hkv_swa, device=dev)
        _fill_rings(kvr, self.ring, ss, 1, P0, self.t4, vscale)
        self.ring0 = (self.ring.k.clone(), self.ring.v.clone(), self.ring.slot_pos.clone())
        self.stage = kvr.LinearLayout.empty(C, hkv_swa, device=dev)
        self.kf, self.vf = sf.k(C, hkv_full, seq=0, start=P0), sf.v(C, hkv_full, seq=0, start=P0)
        self.ks, self.vs = ss.k(C, hkv_swa, seq=0, start=P0), ss.v(C, hkv_swa, seq=0, start=P0)
        self.qf = sf.q(C, hq, hkv_full, seq=0, start=P0)
        self.qs = ss.q(C, hq, hkv_swa, seq=0, start=P0)
        self.sinks = ss.sinks(hq).to(dev)
        self.pos = torch.arange(P0, P0 + C, device=dev)
        self.seq = torch.zeros(C, dtype=torch.int32, device=dev)
        self.tail = min(C, 128)
        self.out_f = torch.empty(C, hq, 128, dtype=torch.bfloat16, device=dev)
        self.out_s = torch.empty(C, hq, 128, dtype=torch.bfloat16, device=dev)
        self.t_full = EventTimer()
        self.t_swa = EventTimer()
        self.launches_per_step = 5

    def flops_full(self):
        return attn_flops(prefill_pairs(self.P0, self.C), self.hq)

    def flops_swa(self):
        return attn_flops(prefill_pairs(self.P0, self.C, window=128), self.hq)

    def bytes_swa(self):
        """Bytes the windowed prefill must move at least: q read, out written,
        the staged chunk K/V and the ring rows before the chunk read once,
        the ring tags and the fp32 RoPE rows of the chunk's positions."""
        C, hq, hkv = self.C, self.hq, self.hkv_swa
        ring_rows = min(self.P0, 127)
        return (C * hq * (192 + 128) * 2 + C * hkv * (192 + 128) * 2 + ring_rows * hkv * (192 + 128) * 2
                + 128 * 4 + C * 64 * 4)


    def step(self, stream, timed=False):
        kvr = self.kvr
        # restore the ring's pre-chunk state (the previous step committed the chunk's tail)
        self.ring.k.copy_(self.ring0[0]); self.ring.v.copy_(self.ring0[1]); self.ring.slot_pos.copy_(self.ring0[2])
        kvr.kv_ring_append_rope(self.kf, self.vf, self.pos, self.seq, self.t7, self.vscale, self.pool, stream=stream)
        a = self.t_full.start(stream) if timed else None
        kvr.full_attn_prefill_chunk(self.qf, self.P0, 0, self.pool, self.t7, SCALE, out=self.out_f, stream=stream)
        if timed:
            self.t_full.stop(a, stream)
        kvr.kv_ring_append_rope(self.ks, self.vs, self.pos, None, self.t4, self.vscale, self.stage, stream=stream)
        a = self.t_swa.start(stream) if timed else None
        kvr.swa_sink_prefill_chunk(self.qs, self.P0, 0, self.stage, self.ring, self.sinks, self.t4, SCALE, out=self.out_s,
                                   stream=stream)
        if timed:
            self.t_swa.stop(a, stream)
        t = self.tail
        kvr.kv_ring_append_rope(self.ks[-t:], self.vs[-t:], self.pos[-t:], self.seq[-t:], self.t4, self.vscale,
                                self.ring, stream=stream)


# --------------------------------------------------------------------------- runs

def timed_run(work, steps, warmup, stream, flush=None, label="timed", kernel_events=False):
    """Mean step time (ms) of `steps` steps after `warmup` untimed ones.  With
    kernel_events the step also records CUDA events around its attention calls
    (the per-kernel durations); events between two launches break their
    programmatic overlap, so the step time of such a pass is a little longer
    and a headline step time is taken without them."""
    for _ in range(warmup):
        work.step(stream)
    torch.cuda.synchronize()
    ev = []
    torch.cuda.nvtx.range_push(label)
    for _ in range(steps):
        if flush is not None:
            flush_l2(flush)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        work.step(stream, timed=kernel_events)
        b.record(stream)
        ev.append((a, b))
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    return sum(a.elapsed_time(b) for a, b in ev) / len(ev)


def graph_time_ms(calls, reps=5):
    """Per-call GPU time of a list of launches replayed as one CUDA graph
    (no host launch gaps); each call takes the capture stream."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for c in calls[:3]:
            c(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cs = torch.cuda.current_stream()
        for c in calls:
            c(cs)
    g.replay()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        g.replay()
    b.record()
    b.synchronize()
    return a.elapsed_time(b) / (reps * len(calls))


def decode_kernel_graph_times(work):
    """The two decode kernels alone, each as a graph of launches (windowed:
    rotating over the ring copies, so every launch reads from HBM)."""
    kvr = work.kvr
    swa = [(lambda st, r=r: kvr.swa_sink_decode(work.q_swa, work.pos, work.seq, r, work.sinks, work.t4, SCALE,
                                                out=work.out_swa, stream=st)) for r in work.rings] * 4
    full = [(lambda st: kvr.full_attn_decode(work.q_full, work.pos, work.seq, work.pool, work.t7, SCALE, work.max_ctx,
                                             workspace=work.ws, out=work.out_full, stream=st))] * 10
    return graph_time_ms(swa), graph_time_ms(full)


def pool_ops_times(work, hbm, peaks_src, copies=None):
    """Ring snapshot and restore of the decode batch; and the decode workload's windowed layer kept in pages (block size 64; the
    block table holds only the blocks of each sequence's window): windowed
    decode over the pages and the ring-from-pages gather, each a graph of
    launches rotating over copies larger than L2 together; and the
    out-of-window release at decode cadence (one block per sequence)."""
    kvr = work.kvr
    from sinks_kv_ring_gb300.synth import Synth
    dev = work.pos.device
    B, hkv, p, bs = work.B, work.hkv_swa, work.p, 64
    lo = max(0, p - 127)
    b0, b1 = lo // bs, p // bs
    nper = b1 - b0 + 1
    tab = torch.full((B, b1 + 1), -1, dtype=torch.int32, device=dev)
    tab[:, b0:] = torch.arange(B * nper, dtype=torch.int32, device=dev).reshape(B, nper)
    base = kvr.PagedLayout(torch.zeros(B * nper, hkv, bs, 192, dtype=torch.bfloat16, device=dev),
                           torch.zeros(B * nper, hkv, bs, 128, dtype=torch.bfloat16, device=dev), tab)
    syn = Synth(1001, dist="shifted", device=dev)
    for s in range(B):
        kvr.kv_ring_append_rope(syn.k(p + 1 - lo, hkv, seq=s, start=lo), syn.v(p + 1 - lo, hkv, seq=s, start=lo),
                                torch.arange(lo, p + 1, device=dev), torch.full((p + 1 - lo,), s, dtype=torch.int32,
                                                                                 device=dev), work.t4, work.vscale, base)
    one = (base.k.numel() + base.v.numel()) * 2
    if copies is None:
        copies = max(1, min(64, math.ceil(4 * 129e6 / one)))
    pools = [base] + [kvr.PagedLayout(base.k.clone(), base.v.clone(), tab) for _ in range(copies - 1)]
    dec = [(lambda st, pl=pl: kvr.swa_sink_decode(work.q_swa, work.pos, work.seq, pl, work.sinks, work.t4, SCALE,
                                                  out=work.out_swa, stream=st)) for pl in pools] * 4
    ms_dec = graph_time_ms(dec)
    # each launch writes its own destination ring too, so that the written
    # rows leave L2 for HBM as they would in use (one ring fits in L2)
    rings_g = [kvr.RingLayout.empty(B, hkv, device=dev) for _ in pools]
    end = torch.full((B,), p + 1, dtype=torch.int64, device=dev)
    gat = [(lambda st, pl=pl, rg=rg: kvr.kv_ring_gather_pages(pl, rg, work.seq, work.seq, end, stream=st))
           for pl, rg in zip(pools, rings_g)] * 4
    ms_gat = graph_time_ms(gat)
    gat_bytes = 2 * layer_kv_bytes([p + 1] * B, hkv, window=128) + B * 128 * 4
    # release: every sequence has a full table (ids 0..B*mb-1); each call frees
    # the one block that the next query's window has just left
    mb = b1 + 1
    rtab0 = torch.arange(B * mb, dtype=torch.int32, device=dev).reshape(B, mb)
    rtab, rlo0 = rtab0.clone(), torch.full((B,), max(0, b0 - 1), dtype=torch.int32, device=dev)
    rlo = rlo0.clone()
    free = torch.empty(B * mb, dtype=torch.int32, device=dev)
    cnt = torch.zeros(1, dtype=torch.int32, device=dev)
    nxt = torch.full((B,), b0 * bs + 127, dtype=torch.int64, device=dev)
    reset = lambda st: (rtab.copy_(rtab0), rlo.copy_(rlo0), cnt.zero_())
    rel = lambda st: kvr.kv_pages_release_window(rtab, B * mb, bs, work.seq, nxt, free, cnt, lo=rlo, stream=st)
    ms_reset = graph_time_ms([reset] * 20)
    ms_both = graph_time_ms([lambda st: (reset(st), rel(st))] * 20)
    released = int(cnt.item())
    dec_gbs = work.bytes_swa() / (ms_dec / 1e3) / 1e9
    gat_gbs = gat_bytes / (ms_gat / 1e3) / 1e9
    # ring snapshot / restore of the whole batch, rotating over the decode workload's ring copies
    # and as many snapshot buffers (one buffer would stay in L2 from launch to launch)
    del rings_g
    snaps = [kvr.ring_snapshot_alloc(B, hkv, device=dev) for _ in work.rings]
    sn = [(lambda st, r=r, sb=sb: kvr.kv_ring_snapshot(r, work.seq, sb, stream=st)) for r, sb in zip(work.rings, snaps)] * 4
    rs = [(lambda st, r=r, sb=sb: kvr.kv_ring_restore(r, work.seq, sb, stream=st)) for r, sb in zip(work.rings, snaps)] * 4
    ms_sn, ms_rs = graph_time_ms(sn), graph_time_ms(rs)
    copy_bytes = 2 * (kvr.RingLayout.bytes_per_layer(B, hkv) + B * 128 * 4)
    copy = lambda ms: {"graph_ms": round(ms, 5), "bytes": copy_bytes, "GB/s": round(copy_bytes / ms / 1e6, 1),
                       "roofline": with_nominal({"bound": "hbm", "achieved": round(copy_bytes / ms / 1e6, 1),
                                                 "peak": hbm, "unit": "GB/s",
                                                 "frac": round(copy_bytes / ms / 1e6 / hbm, 4),
                                                 "peak_source": peaks_src})}
    return {
        "kv_ring_snapshot": dict(workload=f"{B} sequences x {hkv} KV heads: rings (slots + tags) to a snapshot, "
                                          f"rotating over {len(work.rings)} ring copies and as many snapshot buffers",
                                 **copy(ms_sn)),
        "kv_ring_restore": dict(workload=f"{B} sequences x {hkv} KV heads: snapshots back into the rings (the same "
                                         f"rotation)", **copy(ms_rs)),
        "swa_sink_decode_paged": {
            "workload": f"batch {B}, windowed layer kept in pages of {bs} (block table holds the window's {nper} "
                        f"blocks per sequence), graph rotating over {copies} copies", "graph_ms": round(ms_dec, 5),
            "bytes": work.bytes_swa(), "GB/s": round(dec_gbs, 1),
            "roofline": with_nominal({"bound": "hbm", "achieved": round(dec_gbs, 1), "peak": hbm, "unit": "GB/s",
                                      "frac": round(dec_gbs / hbm, 4), "peak_source": peaks_src,
                                      "kernel": "swa_paged_kernel",
                                      "traffic": kernel_traffic("swa_paged_kernel")})},
        "kv_ring_gather_pages": {
            "workload": f"{B} sequences x {hkv} KV heads: the 128-position window from pages into rings, "
                        f"rotating over {copies} pools and as many destination rings",
            "graph_ms": round(ms_gat, 5), "bytes": gat_bytes, "GB/s": round(gat_gbs, 1),
            "roofline": with_nominal({"bound": "hbm", "achieved": round(gat_gbs, 1), "peak": hbm, "unit": "GB/s",
                                      "frac": round(gat_gbs / hbm, 4), "peak_source": peaks_src})},
        "kv_pages_release_window": {
            "workload": f"{B} sequences, one out-of-window block each (decode cadence)",
            "us_per_call": round((ms_both - ms_reset) * 1e3, 2), "released_per_call": released,
            "note": "one-CTA bookkeeping kernel; latency, no roofline"},
    }


def e2e_decode(work, steps, warmup, stream):
    """The same decode step with each step's inputs copied in from pinned host
    memory and its outputs copied back, all inside the timed region.  As in a
    serving loop the copies run on their own streams with two device buffer
    sets: step i+1's inputs upload while step i computes, and step i's outputs
    download while step i+1 computes.  The region runs from the first upload
    to the end of the last download."""
    names_in = ["q_swa", "q_full", "k_swa", "v_swa", "k_full", "v_full", "pos"]
    names_out = ["out_swa", "out_full"]
    orig = {n: getattr(work, n) for n in names_in + names_out}
    pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    host_in = {n: pin(orig[n]).copy_(orig[n]) for n in names_in}
    host_out = [{n: pin(orig[n]) for n in names_out} for _ in range(2)]
    sets = [orig, {n: torch.empty_like(orig[n]) for n in names_in + names_out}]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    fetched = [torch.cuda.Event() for _ in range(2)]

    def upload(i):
        k = i % 2
        up.wait_event(done[k])         # step i-2 (same buffer set) has finished computing
        with torch.cuda.stream(up):
            for n in names_in:
                sets[k][n].copy_(host_in[n], non_blocking=True)
        ready[k].record(up)

    def compute(i):
        k = i % 2
        stream.wait_event(ready[k])
        stream.wait_event(fetched[k])  # step i-2's outputs (same buffer set) are on the host
        for n in names_in + names_out:
            setattr(work, n, sets[k][n])
        with torch.cuda.stream(stream):
            work.step(stream)
        done[k].record(stream)

    def download(i):
        k = i % 2
        down.wait_event(done[k])
        with torch.cuda.stream(down):
            for n in names_out:
                host_out[k][n].copy_(sets[k][n], non_blocking=True)
        fetched[k].record(down)

    def run(n, a=None, b=None):
        torch.cuda.synchronize()
        for k in range(2):                 # events start out "already happened"
            done[k].record(stream)
            fetched[k].record(down)
        if a is not None:
            a.record(up)
            down.wait_event(a)
            stream.wait_event(a)
        upload(0)
        for i in range(n):
            if i + 1 < n:
                upload(i + 1)
            compute(i)
            download(i)
        if b is not None:
            b.record(down)
        torch.cuda.synchronize()

    run(warmup)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    run(steps, a, b)
    for n, t in orig.items():
        setattr(work, n, t)
    # the last step's outputs came back intact
    last = host_out[(steps - 1) % 2]
    assert all(torch.equal(last[n], sets[(steps - 1) % 2][n].cpu()) for n in names_out)
    return a.elapsed_time(b) / steps, h2d, d2h


def cpu_baseline_decode(work, budget_s=12.0, max_seqs=16):
    """The fp64 oracle on sampled sequences of the decode workload (both layers,
    all heads), on all host cores; tokens/s.  Sequences are taken in turn
    (cycling over the first max_seqs) until budget_s of oracle time is spent."""
    import oracle
    from sinks_kv_ring_gb300.synth import Synth
    cores = os.cpu_count() or 1
    syn_s, syn_f = Synth(1001, layer=0, device="cuda"), Synth(1001, layer=1, device="cuda")
    q_s, q_f = work.q_swa.cpu(), work.q_full.cpu()
    sk = work.sinks.double().cpu().numpy()
    p = work.p
    lo = max(0, p - 127)
    cache = {}

    def inputs(b):
        if b not in cache:
            kf = torch.cat([syn_f.k(min(65536, p - s0), work.hkv_full, seq=b, start=s0) for s0 in range(0, p, 65536)]
                           + [work.k_full[b:b + 1]]).cpu()
            vf = torch.cat([syn_f.v(min(65536, p - s0), work.hkv_full, seq=b, start=s0) for s0 in range(0, p, 65536)]
                           + [work.v_full[b:b + 1]]).cpu()
            ks = torch.cat([syn_s.k(p - lo, work.hkv_swa, seq=b, start=lo), work.k_swa[b:b + 1]]).cpu()
            vs = torch.cat([syn_s.v(p - lo, work.hkv_swa, seq=b, start=lo), work.v_swa[b:b + 1]]).cpu()
            cache[b] = (kf, vf, ks, vs)
        return cache[b]

    nseq = min(max_seqs, work.B)
    elapsed, done = 0.0, 0
    while elapsed < budget_s:
        b = done % nseq
        kf, vf, ks, vs = inputs(b)
        t0 = time.perf_counter()
        oracle.attend_seq(q_f[b:b + 1], [p], kf, vf, 0, 1e7, work.vscale, SCALE, 0, None, nthreads=cores)
        oracle.attend_seq(q_s[b:b + 1], [p], ks, vs, lo, 1e4, work.vscale, SCALE, 128, sk, nthreads=cores)
        elapsed += time.perf_counter() - t0
        done += 1
    # the same on one thread, one sequence-step
    kf, vf, ks, vs = inputs(0)
    t0 = time.perf_counter()
    oracle.attend_seq(q_f[0:1], [p], kf, vf, 0, 1e7, work.vscale, SCALE, 0, None, nthreads=1)
    oracle.attend_seq(q_s[0:1], [p], ks, vs, lo, 1e4, work.vscale, SCALE, 128, sk, nthreads=1)
    one = time.perf_counter() - t0
    return {"value": round(done / elapsed, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} sequence-steps (cycling over {nseq} of the {work.B} sequences), all 64 heads, one "
                      f"windowed + one full layer at context {p + 1}; {elapsed:.1f} s of fp64 oracle on {cores} threads",
            "single_thread": {"value": round(1.0 / one, 3), "unit": "tokens/s",
                              "sample": f"1 sequence-step on 1 thread, {one:.2f} s"}}


def run_decode(args, kvr, rank):
    stream = torch.cuda.current_stream()
    work = DecodeWorkload(kvr, B=args.batch, ctx=args.ctx, seed=rank_seed(1001, rank))
    torch.cuda.synchronize()
    with Clocks(torch.cuda.current_device()) as ck:
        ms = timed_run(work, args.steps, args.warmup, stream)
    clocks = ck.summary()
    # the per-kernel durations: a second timed pass of the same steps with
    # events around the two attention calls
    timed_run(work, args.steps, 0, stream, label="kernels", kernel_events=True)
    ms_full = work.t_full.mean_ms()
    ms_swa = work.t_swa.mean_ms()
    e2e_ms, h2d, d2h = e2e_decode(work, max(3, args.steps // 2), 2, stream)
    work.graph_ms = decode_kernel_graph_times(work)
    return work, ms, ms_full, ms_swa, clocks, (e2e_ms, h2d, d2h)


def append_bulk_time(pw, ntok=65536):
    """The KV write at prefill size: ntok tokens (RoPE + value scale) into the
    full layer's paged pool, replayed as a CUDA graph; returns (ms per call,
    algorithmic bytes per call).  Bytes: read k, v and write them (640 B each
    way per token and KV head) + one 256-byte table row per token."""
    kvr = pw.kvr
    from sinks_kv_ring_gb300.synth import Synth
    syn = Synth(1002, layer=1, device=pw.pool.k.device)
    k, v = syn.k(ntok, pw.hkv_full, seq=0, start=0), syn.v(ntok, pw.hkv_full, seq=0, start=0)
    pos = torch.arange(ntok, device=k.device)
    seq = torch.zeros(ntok, dtype=torch.int32, device=k.device)
    calls = [(lambda st: kvr.kv_ring_append_rope(k, v, pos, seq, pw.t7, pw.vscale, pw.pool, stream=st))] * 10
    ms = graph_time_ms(calls)
    return ms, ntok * (pw.hkv_full * KV_BYTES * 2 + 256)

def swa_prefill_entry(pw, ms, hbm, peaks_src):
    """The windowed chunked prefill: TFLOP/s and, as it is bound by memory
    (few flops per byte of q and out), its HBM roofline.  `ms` is the call
    timed by CUDA events inside the prefill step (it includes the launch gap
    after the KV write before it); `graph_ms` the call alone, replayed back to
    back in a CUDA graph over two copies of its query rows and staged K/V
    (each launch reads them from HBM: 2 x 243 MB between two uses), which is
    what the roofline object reports, as for the decode kernels."""
    kvr = pw.kvr
    # the ring's pre-chunk state (the step after the call commits the chunk's tail)
    pw.ring.k.copy_(pw.ring0[0]); pw.ring.v.copy_(pw.ring0[1]); pw.ring.slot_pos.copy_(pw.ring0[2])
    copies = [(pw.qs, pw.stage), (pw.qs.clone(), kvr.LinearLayout(pw.stage.k.clone(), pw.stage.v.clone()))]
    calls = [(lambda st, qq=qq, sg=sg: kvr.swa_sink_prefill_chunk(qq, pw.P0, 0, sg, pw.ring, pw.sinks, pw.t4, SCALE,
                                                                 out=pw.out_s, stream=st)) for qq, sg in copies] * 5
    g_ms = graph_time_ms(calls)
    del copies, calls
    gbs = pw.bytes_swa() / (ms / 1e3) / 1e9
    g_gbs = pw.bytes_swa() / (g_ms / 1e3) / 1e9
    return {"ms": round(ms, 4), "TFLOP/s": round(pw.flops_swa() / (ms / 1e3) / 1e12, 1), "flop": pw.flops_swa(),
            "bytes": pw.bytes_swa(), "GB/s": round(gbs, 1), "hbm_frac": round(gbs / hbm, 4),
            "graph_ms": round(g_ms, 4), "graph_GB/s": round(g_gbs, 1),
            "graph_TFLOP/s": round(pw.flops_swa() / (g_ms / 1e3) / 1e12, 1),
            "note": "ms: CUDA events around the call inside the timed prefill step (include its launch gap); "
                    "graph_*: the call replayed back to back in a CUDA graph, query rows and staged K/V rotated "
                    "over two copies; the roofline object uses graph_ms",
            "roofline": with_nominal({"bound": "hbm", "achieved": round(g_gbs, 1), "peak": hbm, "unit": "GB/s",
                                      "frac": round(g_gbs / hbm, 4), "peak_source": peaks_src,
                                      "kernel": "swa_band_kernel", "traffic": kernel_traffic("swa_band_kernel")})}



def mixed_window_batch(kvr, hbm, peaks_src, device="cuda"):
    """A mixed prefill / decode batch on a windowed layer through the varlen
    call: 8 chunks of 2048 rows beside 64 decode tokens (64 q / 8 KV heads,
    every sequence 32768 tokens in), two such batches alternated in one CUDA
    graph.  Bytes: q and out, the staged rows, each chunk's 127 ring rows
    and slot tags, the fp32 RoPE rows."""
    from sinks_kv_ring_gb300.synth import Synth
    hq, hkv, vs, P = 64, 8, 0.707, 32768
    Cs = [2048] * 8 + [1] * 64
    n, T = len(Cs), sum(Cs)
    t4 = kvr.rope_table(1e4, P + max(Cs), device=device)
    syn = Synth(1005, device=device)
    ring = kvr.RingLayout.empty(n, hkv, device=device)
    _fill_rings(kvr, ring, syn, n, P, t4, vs)
    cu = torch.zeros(n + 1, dtype=torch.int32, device=device)
    cu[1:] = torch.cumsum(torch.tensor(Cs, dtype=torch.int32, device=device), 0)
    P0 = torch.full((n,), P, dtype=torch.int64, device=device)
    seq = torch.arange(n, dtype=torch.int32, device=device)
    pos = torch.cat([torch.arange(P, P + C, device=device) for C in Cs])
    sinks = syn.sinks(hq).to(device)
    ws = torch.empty(kvr.swa_sink_prefill_varlen_workspace_size(n), dtype=torch.uint8, device=device)
    batches = []
    for b in range(2):
        stage = kvr.LinearLayout.empty(T, hkv, device=device)
        kvr.kv_ring_append_rope(syn.k(T, hkv, seq=100 + b, start=P), syn.v(T, hkv, seq=100 + b, start=P), pos, None, t4,
                                vs, stage)
        batches.append((syn.q(T, hq, hkv, seq=200 + b, start=P), stage,
                        torch.empty(T, hq, 128, dtype=torch.bfloat16, device=device)))
    calls = [(lambda st, bt=bt: kvr.swa_sink_prefill_varlen(bt[0], cu, P0, seq, bt[1], ring, sinks, t4, SCALE,
                                                             workspace=ws, out=bt[2], stream=st)) for bt in batches] * 2
    ms = graph_time_ms(calls)
    nbytes = T * hq * (192 + 128) * 2 + T * hkv * (192 + 128) * 2 + n * (127 * hkv * (192 + 128) * 2 + 128 * 4) + T * 256
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"workload": "mixed batch on a windowed layer: 8 chunks of 2048 rows + 64 decode tokens, 64 q / 8 KV heads, "
                        "32768 tokens in; varlen call, CUDA graph over 2 batches",
            "graph_ms": round(ms, 4), "bytes": nbytes, "GB/s": round(gbs, 1),
            "roofline": with_nominal({"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                                      "frac": round(gbs / hbm, 4), "peak_source": peaks_src,
                                      "kernel": "swa_band_kernel (+ varlen_plan_kernel, swa_short_kernel)",
                                      "traffic": None})}


def long_decode_entry(kvr, hbm, peaks_src, world, rank, min_s=0.5):
    """Long-context decode as a sub-measurement of the default line: batch
    16, each sequence at 524288 cached tokens; the step is the decode step of
    DecodeWorkload (two KV writes, windowed decode, full decode with its
    merge).  Timed over at least min_s seconds; the pool fill is timed apart."""
    t0 = time.perf_counter()
    work = DecodeWorkload(kvr, B=16, ctx=524288, seed=rank_seed(1003, rank))
    torch.cuda.synchronize()
    fill_s = time.perf_counter() - t0
    stream = torch.cuda.current_stream()
    probe = timed_run(work, 3, 3, stream)
    steps = max(20, math.ceil(min_s * 1e3 / probe))
    work.t_full, work.t_swa = EventTimer(), EventTimer()
    with Clocks(torch.cuda.current_device()) as ck:
        ms = timed_run(work, steps, 3, stream)
    ms = max_over_ranks([ms], world, "cuda")[0]
    timed_run(work, min(steps, 50), 0, stream, label="kernels", kernel_events=True)  # the per-call durations
    ms_full, ms_swa = work.t_full.mean_ms(), work.t_swa.mean_ms()
    g_swa, g_full = decode_kernel_graph_times(work)
    gbs_full = work.bytes_full() / (ms_full / 1e3) / 1e9
    step_bytes = work.bytes_full() + work.bytes_swa()
    out = {
        "workload": f"batch {work.B}, each at {work.p + 1} tokens of context; full layer 4 KV heads (theta 1e7), "
                    "windowed layer 8 KV heads ring 128 + sink (theta 1e4); 64 q heads; value scale 0.707; "
                    "step = 2 KV writes + windowed decode + full decode",
        "pool_fill_s": round(fill_s, 1), "steps": steps, "timed_s": round(steps * ms / 1e3, 2),
        "ms_per_step": round(ms, 4), "tokens/s": round(job_throughput(work.B, world, ms), 1),
        "bytes_per_step": step_bytes, "step_GB/s": round(step_bytes / (ms / 1e3) / 1e9, 1),
        "full_attn_decode": {"ms": round(ms_full, 4), "GB/s": round(gbs_full, 1), "bytes": work.bytes_full(),
                             "graph_ms": round(g_full, 4)},
        "swa_sink_decode": {"ms": round(ms_swa, 5), "bytes": work.bytes_swa(), "graph_ms": round(g_swa, 5),
                            "graph_hbm_frac": round(work.bytes_swa() / g_swa / 1e6 / hbm, 4)},
        "roofline": with_nominal({"bound": "hbm", "achieved": round(gbs_full, 1), "peak": hbm, "unit": "GB/s",
                                  "frac": round(gbs_full / hbm, 4), "peak_source": peaks_src,
                                  "kernel": "full_attn_decode (split kernel + combine)", "traffic": None}),
        "clocks": ck.summary(),
        "gpu_launches": work.launches_per_step * steps,
    }
    del work
    torch.cuda.empty_cache()
    return out


def small_batch_decode_entry(kvr, hbm, peaks_src, cases=((1, 8192), (1, 32768), (4, 32768))):
    """The full-attention decode of one layer (4 KV heads, 64 q heads) at a
    few sequences: the interactive single-stream shape, where the fixed costs
    of a launch (plan, first loads, merge) weigh most.  Each case is a CUDA
    graph of launches rotating over copies of its pool (together > 4x L2), so
    every launch reads its K/V from HBM; the roofline object is batch 1 at
    32769 tokens."""
    from sinks_kv_ring_gb300.synth import Synth
    dev = "cuda"
    hq, hkv = 64, 4
    t7 = kvr.rope_table(1e7, max(c for _, c in cases) + 8, device=dev)
    out, roof = {}, None
    for B, ctx in cases:
        n = ctx + 1
        pool = kvr.PagedLayout.contiguous(B, hkv, n, block_size=64, device=dev, zero=False)
        _fill_pool(kvr, pool, Synth(1006, layer=1, device=dev), range(B), [n] * B, t7, 0.707)
        q = Synth(1006, layer=1, device=dev).q(B, hq, hkv, seq=10_000)
        pos = torch.full((B,), ctx, dtype=torch.int64, device=dev)
        seq = torch.arange(B, dtype=torch.int32, device=dev)
        ws = torch.empty(kvr.full_attn_decode_workspace_size(B, hq, hkv, n), dtype=torch.uint8, device=dev)
        o = torch.empty(B, hq, 128, dtype=torch.bfloat16, device=dev)
        nbytes = layer_kv_bytes([n] * B, hkv)
        copies = max(1, min(32, math.ceil(4 * 129e6 / nbytes)))
        pools = [pool] + [kvr.PagedLayout(pool.k.clone(), pool.v.clone(), pool.block_table) for _ in range(copies - 1)]
        calls = [(lambda st, pl=pl: kvr.full_attn_decode(q, pos, seq, pl, t7, SCALE, n, workspace=ws, out=o,
                                                           stream=st)) for pl in pools] * max(2, 16 // copies)
        ms = graph_time_ms(calls)
        gbs = nbytes / (ms / 1e3) / 1e9
        out[f"batch{B}_ctx{n}"] = {"us": round(ms * 1e3, 2), "bytes": nbytes, "GB/s": round(gbs, 1),
                                   "hbm_frac": round(gbs / hbm, 4), "pool_copies": copies}
        if (B, ctx) == (1, 32768):
            roof = with_nominal({"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                                 "frac": round(gbs / hbm, 4), "peak_source": peaks_src,
                                 "kernel": "full_attn_decode (split kernel + combine), batch 1 at 32769 tokens",
                                 "traffic": None})
        del pools, pool
        torch.cuda.empty_cache()
    out["workload"] = ("full-attention layer, 4 KV heads (theta 1e7), 64 q heads, one decode token per sequence; "
                       "CUDA graph of launches rotating over pool copies")
    if roof is not None:
        out["roofline"] = roof
    return out


def pro_mixed_entry(kvr, hbm, peaks_src, world, rank, min_s=0.5):
    """The Pro-shaped mixed batch as a sub-measurement of the default line:
    one decode step over the 70-layer stack (ProMixedWorkload) as one CUDA
    graph.  Every full layer streams the same pool: at ~50 GB it is far
    larger than L2, so each layer reads its bytes from HBM as a distinct
    pool would (the --workload pro_mixed run keeps up to 10 distinct pools).
    Timed over at least min_s seconds; pool fill and capture timed apart."""
    t0 = time.perf_counter()
    work = ProMixedWorkload(kvr, seed=rank_seed(1004, rank), n_pools=1)
    work.capture()
    torch.cuda.synchronize()
    fill_s = time.perf_counter() - t0
    stream = torch.cuda.current_stream()
    probe = timed_run(work, 1, 3, stream)
    steps = max(5, math.ceil(min_s * 1e3 / probe))
    with Clocks(torch.cuda.current_device()) as ck:
        ms = timed_run(work, steps, 1, stream)
    ms = max_over_ranks([ms], world, "cuda")[0]
    nbytes = work.bytes_per_step()
    gbs = nbytes / (ms / 1e3) / 1e9
    out = {
        "workload": f"{work.B} sequences, contexts log-uniform 1K-1M (seed 1004, {int(sum(work.ctx))} tokens); "
                    f"{len(work.kinds)} layers (i % 7 == 6 full: {work.kinds.count('full')} full, "
                    f"{work.kinds.count('swa')} windowed); 64 q heads, windowed 8 KV heads, full 4 KV heads; value "
                    "scale 0.612; one decode step (KV write + attention per layer) as one CUDA graph",
        "buckets": work.buckets(), "distinct_full_pools": work.n_pools,
        "pool_fill_s": round(fill_s, 1), "steps": steps, "timed_s": round(steps * ms / 1e3, 2),
        "ms_per_step": round(ms, 3), "tokens/s": round(job_throughput(work.B, world, ms), 1),
        "bytes_per_step": nbytes,
        "roofline": with_nominal({"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                                  "frac": round(gbs / hbm, 4), "peak_source": peaks_src,
                                  "kernel": f"whole {len(work.kinds)}-layer step", "traffic": None}),
        "clocks": ck.summary(),
        "gpu_launches": work.launches_per_step * steps,
    }
    del work
    torch.cuda.empty_cache()
    return out


def run_prefill(kvr, steps, warmup, P0=122880, C=8192):
    stream = torch.cuda.current_stream()
    work = PrefillWorkload(kvr, P0=P0, C=C)
    torch.cuda.synchronize()
    ms = timed_run(work, steps, warmup, stream, label="timed", kernel_events=True)
    return work, ms


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="flash_decode",
                    choices=["flash_decode", "long_decode", "prefill", "pro_mixed", "pro_true", "long_stack",
                             "mtp_decode"])
    ap.add_argument("--mtp-len", type=int, default=4, help="draft tokens verified per sequence (mtp_decode)")
    ap.add_argument("--no-prefill", action="store_true", help="skip the prefill sub-measurement")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-long", action="store_true",
                    help="skip the long-context and Pro-shaped sub-measurements of the default line")
    ap.add_argument("--batch", type=int, default=None, help="decode batch per GPU (default: the workload's)")
    ap.add_argument("--ctx", type=int, default=None, help="cached tokens per sequence (default: the workload's)")
    ap.add_argument("--prefill-p0", type=int, default=122880, help="cached tokens before the prefill chunk")
    ap.add_argument("--prefill-c", type=int, default=8192, help="prefill chunk length")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.workload == "long_decode":
        args.batch = args.batch or 16
        args.ctx = args.ctx or 524288
        if "--steps" not in sys.argv:
            args.steps = 200
    else:
        args.batch = args.batch or 64
        args.ctx = args.ctx or 32768

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return run_reference(args, rank, world)

    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import __graft_entry__
    __graft_entry__.build() if rank == 0 else None
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    import sinks_kv_ring_gb300 as kvr
    peaks_d, peaks_src = peaks()
    if args.workload == "prefill":
        return prefill_only(args, kvr, peaks_d, peaks_src, rank, world)
    if args.workload in ("pro_mixed", "pro_true", "long_stack"):
        return pro_mixed(args, kvr, peaks_d, peaks_src, rank, world)
    if args.workload == "mtp_decode":
        return mtp_only(args, kvr, peaks_d, peaks_src, rank, world)

    work, ms, ms_full, ms_swa, clocks, (e2e_ms, h2d, d2h) = run_decode(args, kvr, rank)
    ms, e2e_ms = max_over_ranks([ms, e2e_ms], world, "cuda")
    B = work.B
    value = job_throughput(B, world, ms)
    hbm = peaks_d["hbm_gbs"]
    gbs_full = work.bytes_full() / (ms_full / 1e3) / 1e9
    gbs_swa = work.bytes_swa() / (ms_swa / 1e3) / 1e9
    res = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{args.workload}: batch {B}, 64 q heads; windowed layer 8 KV heads ring 128 + sink; "
                               f"full layer 4 KV heads at context {work.p + 1}; dims 192/192/128; value scale 0.707",
                   "global_batch": B * world, "seq_len": work.p + 1, "parallelism": f"dp{world}",
                   "l2": f"inputs > L2: full pool {work.bytes_full() / 1e9:.2f} GB read per step; windowed rings "
                         f"rotated over {len(work.rings)} copies ({len(work.rings) * work.bytes_swa() / 1e9:.2f} GB)"},
        "kernels": {
            "full_attn_decode": {"ms": round(ms_full, 4), "GB/s": round(gbs_full, 1),
                                 "hbm_frac": round(gbs_full / hbm, 4), "bytes": work.bytes_full(),
                                 "graph_ms": round(work.graph_ms[1], 4),
                                 "graph_GB/s": round(work.bytes_full() / work.graph_ms[1] / 1e6, 1),
                                 "note": "ms: CUDA events around the call in a second timed pass of the same steps "
                                         "(events between launches break their programmatic overlap, so the step "
                                         "time, value and ms_per_step, is taken in a pass without them)"},
            "swa_sink_decode": {"ms": round(ms_swa, 5), "GB/s": round(gbs_swa, 1),
                                "hbm_frac": round(gbs_swa / hbm, 4), "bytes": work.bytes_swa(),
                                "graph_ms": round(work.graph_ms[0], 5),
                                "graph_GB/s": round(work.bytes_swa() / work.graph_ms[0] / 1e6, 1),
                                "graph_hbm_frac": round(work.bytes_swa() / work.graph_ms[0] / 1e6 / hbm, 4),
                                "traffic": kernel_traffic("swa_decode_kernel"),
                                "note": "ms/GB/s: CUDA events around the call in a second timed pass of the same "
                                        "steps (include launch gaps); graph_*: the kernel replayed back to back in a "
                                        "CUDA graph"},
        },
        "roofline": with_nominal({"bound": "hbm", "achieved": round(gbs_full, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(gbs_full / hbm, 4), "peak_source": peaks_src,
                     "kernel": "full_attn_decode (split kernel + combine)",
                     "traffic": kernel_traffic("full_decode_kernel")}),
        "e2e": {"value": round(job_throughput(B, world, e2e_ms), 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "copies": "every step's inputs uploaded from pinned host memory and outputs read back, on their own "
                          "streams with two device buffer sets: step i+1's upload and step i-1's download overlap "
                          "step i; timed from the first upload to the end of the last download"},
        "gpu_launches": work.launches_per_step * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline_decode(work, max_seqs=16 if args.workload == "flash_decode" else 2)
    if args.workload == "flash_decode":
        m, mms, mck, mg = run_mtp(work, min(20, args.steps), 3)
        mms = max_over_ranks([mms], world, "cuda")[0]
        res["mtp"] = mtp_result(m, mms, mck, mg, hbm, world)
        res["gpu_launches"] += m.launches_per_step * min(20, args.steps)
        del m
        res["pool_ops"] = pool_ops_times(work, hbm, peaks_src)
    if not args.no_prefill and args.workload == "flash_decode":
        del work
        torch.cuda.empty_cache()
        psteps = min(5, args.steps)
        with Clocks(torch.cuda.current_device()) as pck:
            pw, pms = run_prefill(kvr, psteps, 3)
        pms = max_over_ranks([pms], world, "cuda")[0]
        tf_full = pw.flops_full() / (pw.t_full.mean_ms() / 1e3) / 1e12
        pk = peaks_d["bf16_tflops"]    # burst: the kernel is timed over a few short launches
        res["prefill"] = {
            "workload": "1 sequence, 8192-token chunk on 122880 cached tokens; 64 q heads; full layer 4 KV heads "
                        "theta 1e7 + windowed layer 8 KV heads theta 1e4, ring 128 + sink",
            "ms_per_step": round(pms, 3),
            "full_attn_prefill_chunk": {"ms": round(pw.t_full.mean_ms(), 3), "TFLOP/s": round(tf_full, 1),
                                        "flop": pw.flops_full()},
            "swa_sink_prefill_chunk": swa_prefill_entry(pw, pw.t_swa.mean_ms(), hbm, peaks_src),
            "roofline": with_nominal({"bound": "tensor", "achieved": round(tf_full, 1), "peak": pk, "unit": "TFLOP/s",
                         "frac": round(tf_full / pk, 4),
                         "peak_source": peaks_src + f" (burst; timed over {psteps} launches, "
                                                    f"{psteps * pw.t_full.mean_ms() / 1e3:.2f} s)",
                         "traffic": kernel_traffic("full_prefill_tc_kernel")}),
        }
        res["prefill"]["steps"] = psteps
        res["prefill"]["clocks"] = pck.summary()
        ams, abytes = append_bulk_time(pw)
        agbs = abytes / (ams / 1e3) / 1e9
        res["prefill"]["kv_ring_append_rope"] = {
            "workload": "65536 tokens x 4 KV heads into the paged pool (RoPE + value scale), CUDA graph replay",
            "ms": round(ams, 4), "bytes": abytes, "GB/s": round(agbs, 1),
            "roofline": with_nominal({"bound": "hbm", "achieved": round(agbs, 1), "peak": hbm, "unit": "GB/s",
                                      "frac": round(agbs / hbm, 4), "peak_source": peaks_src,
                                  "kernel": "append_kernel", "traffic": kernel_traffic("append_kernel")})}
        res["gpu_launches"] += pw.launches_per_step * psteps
        res["prefill"]["swa_sink_prefill_varlen"] = mixed_window_batch(kvr, hbm, peaks_src)
        del pw
        torch.cuda.empty_cache()
    if not args.no_long and args.workload == "flash_decode":
        res["small_batch_decode"] = small_batch_decode_entry(kvr, hbm, peaks_src)
        res["long_decode"] = long_decode_entry(kvr, hbm, peaks_src, world, rank)
        res["pro_mixed"] = pro_mixed_entry(kvr, hbm, peaks_src, world, rank)
        res["gpu_launches"] += res["long_decode"]["gpu_launches"] + res["pro_mixed"]["gpu_launches"]
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


def mtp_only(args, kvr, peaks_d, peaks_src, rank, world):
    """Draft verification as the step (see MtpStep)."""
    work = DecodeWorkload(kvr, B=args.batch, ctx=args.ctx, seed=rank_seed(1001, rank), swa_copies=None)
    torch.cuda.synchronize()
    steps = args.steps if "--steps" in sys.argv else 200
    m, ms, ck, g = run_mtp(work, steps, args.warmup, q_len=args.mtp_len)
    ms = max_over_ranks([ms], world, "cuda")[0]
    hbm = peaks_d["hbm_gbs"]
    r = mtp_result(m, ms, ck, g, hbm, world)
    kf = r["full_attn_prefill_varlen"]
    res = {"metric": METRIC, "value": r["verified_tokens_per_s"], "unit": "tokens/s", "n_gpus": world,
           "steps": steps, "warmup": args.warmup, "ms_per_step": r["ms_per_step"], "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
           "config": {"workload": "mtp_decode: " + r["workload"] + f"; full layer 4 KV heads at context {m.max_ctx}, "
                                  "windowed layer 8 KV heads ring 128 + sink; 64 q heads",
                      "global_batch": m.B * world, "seq_len": m.max_ctx, "parallelism": f"dp{world}",
                      "l2": f"inputs > L2: full pool {m.bytes_full() / 1e9:.2f} GB read per step; rings rotated over "
                            f"{len(work.rings)} copies"},
           "kernels": {k: v for k, v in r.items() if k.endswith("varlen")},
           "roofline": with_nominal({"bound": "hbm", "achieved": kf["GB/s"], "peak": hbm, "unit": "GB/s", "frac": kf["hbm_frac"],
                        "peak_source": peaks_src, "kernel": "full_attn_prefill_varlen (plan + tensor-core kernel + merge)",
                        "traffic": kernel_traffic("full_prefill_tc_kernel_varlen")}),
           "gpu_launches": m.launches_per_step * steps, "clocks": r["clocks"]}
    if rank == 0:
        print(json.dumps(res), flush=True)


def prefill_only(args, kvr, peaks_d, peaks_src, rank, world):
    """Chunked prefill as the step: KV write of the chunk into both layers +
    full_attn_prefill_chunk + swa_sink_prefill_chunk + ring commit."""
    steps = args.steps
    with Clocks(torch.cuda.current_device()) as ck:
        pw, pms = run_prefill(kvr, steps, args.warmup, P0=args.prefill_p0, C=args.prefill_c)
    ms_f, ms_s = pw.t_full.mean_ms(), pw.t_swa.mean_ms()
    pms = max_over_ranks([pms], world, "cuda")[0]
    flops = pw.flops_full() + pw.flops_swa()
    tf_full = pw.flops_full() / (ms_f / 1e3) / 1e12
    # the sustained (power-capped) peak for a region of seconds, else the burst one
    timed_s = steps * pms / 1e3
    long_run = timed_s >= 2.0 and "bf16_tflops_sustained" in peaks_d
    pk = peaks_d["bf16_tflops_sustained"] if long_run else peaks_d["bf16_tflops"]
    pk_note = f" ({'sustained' if long_run else 'burst'}; timed region {timed_s:.2f} s)"
    res = {"metric": METRIC, "value": round(job_throughput(flops, world, pms) / 1e12, 1), "unit": "TFLOP/s",
           "n_gpus": world, "steps": steps, "warmup": args.warmup, "ms_per_step": round(pms, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
           "config": {"workload": f"prefill: 1 sequence, {pw.C}-token chunk on {pw.P0} cached tokens; 64 q heads; "
                                  "full layer 4 KV heads + windowed layer 8 KV heads (ring 128 + sink)",
                      "parallelism": f"dp{world}", "l2": "K/V of the full layer re-read from L2 by every query tile"},
           "kernels": {"full_attn_prefill_chunk": {"ms": round(ms_f, 3), "TFLOP/s": round(tf_full, 1),
                                                   "flop": pw.flops_full()},
                       "swa_sink_prefill_chunk": swa_prefill_entry(pw, ms_s, peaks_d["hbm_gbs"], peaks_src)},
           "roofline": with_nominal({"bound": "tensor", "achieved": round(tf_full, 1), "peak": pk, "unit": "TFLOP/s",
                        "frac": round(tf_full / pk, 4), "peak_source": peaks_src + pk_note,
                        "kernel": "full_prefill_tc_kernel", "traffic": kernel_traffic("full_prefill_tc_kernel")}),
           "gpu_launches": pw.launches_per_step * steps, "clocks": ck.summary()}
    ams, abytes = append_bulk_time(pw)
    agbs = abytes / (ams / 1e3) / 1e9
    hbm = peaks_d["hbm_gbs"]
    res["kernels"]["kv_ring_append_rope"] = {
        "workload": "65536 tokens x 4 KV heads into the paged pool (RoPE + value scale), CUDA graph replay",
        "ms": round(ams, 4), "bytes": abytes, "GB/s": round(agbs, 1),
        "roofline": with_nominal({"bound": "hbm", "achieved": round(agbs, 1), "peak": hbm, "unit": "GB/s",
                                  "frac": round(agbs / hbm, 4), "peak_source": peaks_src,
                                  "kernel": "append_kernel", "traffic": kernel_traffic("append_kernel")})}
    res["kernels"]["swa_sink_prefill_varlen"] = mixed_window_batch(kvr, hbm, peaks_src)
    if rank == 0:
        print(json.dumps(res), flush=True)


class ProMixedWorkload:
    """One decode step over a 70-layer stack (layer i is full-attention iff
    i % 7 == 6: 10 full, 60 windowed), 128 sequences with contexts
    log-uniform over [1K, 1M], 64 q heads, windowed 8 KV heads, full 4 KV
    heads, value scale 0.612.  Full layers share `n_pools` distinct pools
    (layer l -> pool l mod n_pools; every pool is far larger than L2, so each
    layer still streams its full bytes from HBM)."""

    def __init__(self, kvr, B=128, hq=64, layers=70, vscale=0.612, seed=1004, n_pools=None, device="cuda",
                 hkv_full=4, hkv_swa=8, contexts=None, full_period=7):
        from sinks_kv_ring_gb300.synth import Synth, ragged_contexts
        self.kvr, self.B, self.hq, self.vscale = kvr, B, hq, vscale
        self.hkv_full, self.hkv_swa = hkv_full, hkv_swa
        dev = device
        # cached tokens per sequence
        self.ctx = list(contexts) if contexts is not None else ragged_contexts(B, 1024, 1 << 20, seed)
        self.max_ctx = max(self.ctx) + 1
        self.kinds = ["full" if i % full_period == full_period - 1 else "swa" for i in range(layers)]
        self.t4 = kvr.rope_table(1e4, self.max_ctx, device=dev)
        self.t7 = kvr.rope_table(1e7, self.max_ctx, device=dev)
        bsz = 64
        mb = [(c + 1 + bsz - 1) // bsz for c in self.ctx]
        nblk = sum(mb)
        pool_bytes = nblk * self.hkv_full * bsz * 640
        free = torch.cuda.mem_get_info()[0]
        if n_pools is None:
            n_pools = max(1, min(self.kinds.count("full"), int((free - 16e9) * 0.85 // pool_bytes)))
        self.n_pools = n_pools
        bt = torch.zeros(B, max(mb), dtype=torch.int32)
        off = 0
        for b, m in enumerate(mb):
            bt[b, :m] = torch.arange(off, off + m, dtype=torch.int32)
            off += m
        bt = bt.to(dev)
        syn_f = Synth(seed, layer=1, device=dev)
        k0 = torch.empty(nblk, self.hkv_full, bsz, 192, dtype=torch.bfloat16, device=dev)
        v0 = torch.empty(nblk, self.hkv_full, bsz, 128, dtype=torch.bfloat16, device=dev)
        first = kvr.PagedLayout(k0, v0, bt)
        _fill_pool(kvr, first, syn_f, range(B), self.ctx, self.t7, vscale)
        self.pools = [first] + [kvr.PagedLayout(k0.clone(), v0.clone(), bt) for _ in range(n_pools - 1)]
        syn_s = Synth(seed, layer=0, device=dev)
        ring0 = kvr.RingLayout.empty(B, self.hkv_swa, device=dev)
        for b, c in enumerate(self.ctx):
            lo = max(0, c - 127)
            kk, vv = syn_s.k(c - lo, self.hkv_swa, seq=b, start=lo), syn_s.v(c - lo, self.hkv_swa, seq=b, start=lo)
            kvr.kv_ring_append_rope(kk, vv, torch.arange(lo, c, device=dev),
                                    torch.full((c - lo,), b, dtype=torch.int32, device=dev), self.t4, vscale, ring0)
        n_swa = self.kinds.count("swa")
        self.rings = [ring0] + [kvr.RingLayout(ring0.k.clone(), ring0.v.clone(), ring0.slot_pos.clone())
                                for _ in range(n_swa - 1)]
        self.pos = torch.tensor(self.ctx, dtype=torch.int64, device=dev)   # the new token's position
        self.seq = torch.arange(B, dtype=torch.int32, device=dev)
        self.q = syn_s.q(B, hq, self.hkv_swa, seq=50_000)
        self.k_new = {h: syn_s.k(B, h, seq=60_000) for h in {hkv_full, hkv_swa}}
        self.v_new = {h: syn_s.v(B, h, seq=60_000) for h in {hkv_full, hkv_swa}}
        self.sinks = syn_s.sinks(hq).to(dev)
        self.ws = torch.empty(kvr.full_attn_decode_workspace_size(B, hq, self.hkv_full, self.max_ctx),
                              dtype=torch.uint8, device=dev)
        self.out = torch.empty(B, hq, 128, dtype=torch.bfloat16, device=dev)
        self.launches_per_step = sum(4 if k == "full" else 2 for k in self.kinds)
        self.graph = None

    def bytes_per_step(self):
        ctx = [c + 1 for c in self.ctx]
        full = layer_kv_bytes(ctx, self.hkv_full)
        swa = layer_kv_bytes(ctx, self.hkv_swa, window=128)
        return self.kinds.count("full") * full + self.kinds.count("swa") * swa

    BUCKETS = [(0, 65536, "0-64K"), (65536, 262144, "64K-256K"), (262144, 1 << 21, "256K-1M")]

    def buckets(self):
        out = {}
        for lo, hi, name in self.BUCKETS:
            sel = [c for c in self.ctx if lo <= c + 1 < hi]
            out[name] = {"sequences": len(sel), "tokens": int(sum(sel))}
        return out

    def bucket_times(self, hbm):
        """One full layer's decode for each length bucket's sequences alone
        (the batch a scheduler that groups requests by these buckets would
        form; its own split plan), replayed over the distinct pools."""
        kvr, dev = self.kvr, self.pos.device
        out = {}
        for lo, hi, name in self.BUCKETS:
            idx = [b for b, c in enumerate(self.ctx) if lo <= c + 1 < hi]
            if not idx:
                continue
            sel = torch.tensor(idx, dtype=torch.int64, device=dev)
            seq, pos, q = sel.to(torch.int32), self.pos[sel].contiguous(), self.q[sel].contiguous()
            mx = max(self.ctx[b] for b in idx) + 1
            ws = torch.empty(kvr.full_attn_decode_workspace_size(len(idx), self.hq, self.hkv_full, mx),
                             dtype=torch.uint8, device=dev)
            o = torch.empty(len(idx), self.hq, 128, dtype=torch.bfloat16, device=dev)
            calls = [(lambda st, pl=pl: kvr.full_attn_decode(q, pos, seq, pl, self.t7, SCALE, mx, workspace=ws, out=o,
                                                             stream=st)) for pl in self.pools] * max(1, 8 // self.n_pools)
            ms = graph_time_ms(calls)
            nbytes = layer_kv_bytes([self.ctx[b] + 1 for b in idx], self.hkv_full)
            gbs = nbytes / (ms / 1e3) / 1e9
            out[name] = {"sequences": len(idx), "full_layer_ms": round(ms, 4), "bytes": nbytes, "GB/s": round(gbs, 1),
                         "hbm_frac": round(gbs / hbm, 4)}
        return out

    def _eager_step(self, stream):
        kvr = self.kvr
        fi = si = 0
        for kind in self.kinds:
            if kind == "full":
                pool = self.pools[fi % self.n_pools]
                fi += 1
                kvr.kv_ring_append_rope(self.k_new[self.hkv_full], self.v_new[self.hkv_full], self.pos, self.seq,
                                        self.t7, self.vscale, pool, stream=stream)
                kvr.full_attn_decode(self.q, self.pos, self.seq, pool, self.t7, SCALE, self.max_ctx,
                                     workspace=self.ws, out=self.out, stream=stream)
            else:
                ring = self.rings[si]
                si += 1
                kvr.kv_ring_append_rope(self.k_new[self.hkv_swa], self.v_new[self.hkv_swa], self.pos, self.seq,
                                        self.t4, self.vscale, ring, stream=stream)
                kvr.swa_sink_decode(self.q, self.pos, self.seq, ring, self.sinks, self.t4, SCALE, out=self.out,
                                    stream=stream)

    def capture(self):
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self._eager_step(s)          # warm (attributes, maps)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self._eager_step(torch.cuda.current_stream())
        torch.cuda.synchronize()

    def step(self, stream, timed=False):
        self.graph.replay()


def pro_mixed(args, kvr, peaks_d, peaks_src, rank, world):
    if args.workload == "pro_true":   # the head counts the pages imply for the real Pro: 128 q / 8 KV heads
        work = ProMixedWorkload(kvr, hq=128, hkv_full=8, hkv_swa=8, seed=rank_seed(1004, rank))
        shape = "128 sequences, contexts log-uniform 1K-1M (seed 1004); 70 layers (i % 7 == 6 full: 10 full, 60 windowed)"
    elif args.workload == "long_stack":   # long-context decode through a Flash-shaped 48-layer stack
        work = ProMixedWorkload(kvr, B=16, hq=64, layers=48, vscale=0.707, seed=rank_seed(1003, rank),
                                contexts=[524288] * 16, full_period=5)
        shape = "16 sequences at 524288 cached tokens; 48 layers (i % 5 == 4 full: 9 full, 39 windowed)"
    else:
        work = ProMixedWorkload(kvr, seed=rank_seed(1004, rank))
        shape = "128 sequences, contexts log-uniform 1K-1M (seed 1004); 70 layers (i % 7 == 6 full: 10 full, 60 windowed)"
    work.capture()
    stream = torch.cuda.current_stream()
    steps = args.steps if "--steps" in sys.argv else 20
    with Clocks(torch.cuda.current_device()) as ck:
        ms = timed_run(work, steps, args.warmup, stream)
    ms = max_over_ranks([ms], world, "cuda")[0]
    gbs = work.bytes_per_step() / (ms / 1e3) / 1e9
    hbm = peaks_d["hbm_gbs"]
    res = {"metric": METRIC, "value": round(job_throughput(work.B, world, ms), 1), "unit": "tokens/s",
           "n_gpus": world, "steps": steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
           "config": {"workload": f"{args.workload}: {shape}; {work.hq} q heads, windowed "
                                  f"{work.hkv_swa} KV heads, full {work.hkv_full} KV heads; value scale {work.vscale}; "
                                  "one decode step as one CUDA graph",
                      "global_batch": work.B * world, "seq_len": work.max_ctx, "parallelism": f"dp{world}",
                      "buckets": work.buckets(), "distinct_full_pools": work.n_pools,
                      "total_context_tokens": int(sum(work.ctx)),
                      "l2": f"inputs > L2: each full layer streams its pool (tens of GB); "
                            f"{work.kinds.count('swa')} distinct rings"},
           "hbm_gbs": round(gbs, 1),
           "roofline": with_nominal({"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                        "frac": round(gbs / hbm, 4), "peak_source": peaks_src,
                        "kernel": f"whole {len(work.kinds)}-layer step",
                        "traffic": None}),
           "gpu_launches": work.launches_per_step * steps, "clocks": ck.summary()}
    if len(set(work.ctx)) > 1:
        res["buckets"] = work.bucket_times(hbm)
    if rank == 0:
        print(json.dumps(res), flush=True)


def run_reference(args, rank, world):
    """The fp64 CPU oracle, as it stands, on a bounded sample of the decode
    workload (one sequence per step, both layers, all heads)."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    from sinks_kv_ring_gb300.synth import Synth
    cores = os.cpu_count() or 1
    B, hq, p = 64, 64, 32768
    syn_s, syn_f = Synth(1001, layer=0), Synth(1001, layer=1)
    times = []
    for i in range(args.warmup + args.steps):
        b = i % B
        kf = syn_f.k(p + 1, 4, seq=b)
        vf = syn_f.v(p + 1, 4, seq=b)
        ks = syn_s.k(128, 8, seq=b, start=p - 127)
        vs = syn_s.v(128, 8, seq=b, start=p - 127)
        qf, qs = syn_f.q(1, hq, 4, seq=10_000 + b), syn_s.q(1, hq, 8, seq=10_000 + b)
        sk = syn_s.sinks(hq).double().numpy()
        t0 = time.perf_counter()
        oracle.attend_seq(qf, [p], kf, vf, 0, 1e7, 0.707, SCALE, 0, None, nthreads=cores)
        oracle.attend_seq(qs, [p], ks, vs, p - 127, 1e4, 0.707, SCALE, 128, sk, nthreads=cores)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    ms = 1e3 * sum(times) / len(times)
    value = 1.0 / (ms / 1e3)
    sample = (f"one of the 64 sequences per step (all 64 heads, one windowed + one full layer at context {p + 1}); "
              f"fp64 oracle on {cores} threads")
    res = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": f"flash_decode: batch {B}, 64 q heads; windowed layer 8 KV heads ring 128 + sink; "
                                  "full layer 4 KV heads at context 32769 (oracle: one sequence per step)",
                      "global_batch": B, "seq_len": p + 1, "parallelism": "host cores"},
           "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
