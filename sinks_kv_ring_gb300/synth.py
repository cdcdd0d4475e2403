"""Seeded synthetic inputs for the hybrid-SWA attention path.

This module only draws numbers: it holds none of the attention arithmetic
(no RoPE, no softmax, no value scale).  Both the CUDA path and the fp64
oracle take their inputs from here, so the two always see the same bits.

Statistics follow the workloads described for MiMo-V2 attention
(gaudi-cookbook "MiMo-V2.6-Flash on Gaudi 2", section "What was built": raw
q.k logits sit near -25 while the per-head sinks sit near +1):

* ``dist="shifted"`` -- q = z_q + alpha*u, k = z_k - beta*u with z ~ N(0,1)
  and u a seeded unit vector living in dims 64..191 of each KV head (the dims
  RoPE leaves untouched).  With alpha*beta/sqrt(192) = 25 and
  1 + (alpha^2+beta^2)/192 = 9 the scaled logit q.k/sqrt(192) has mean -25 and
  standard deviation 3.
* ``dist="plain"`` -- q, k ~ N(0,1): scaled logits with mean 0 and std 1, so
  the sink does not swallow the softmax.

v ~ N(0,1); sinks ~ N(1, 0.5) in fp32.  Everything else is rounded to bf16.

Every tensor is drawn from its own torch.Generator, seeded by a 64-bit mix of
(seed, tag, index), so one sequence's K/V can be regenerated without drawing
the rest.  Draws on CUDA and on CPU differ (different Philox streams); a test
that needs a CPU copy of a CUDA draw copies it.
"""
from __future__ import annotations

import math

import torch

DQK = 192
DV = 128
DROT = 64

_MASK64 = (1 << 64) - 1


def _mix(*vals: int) -> int:
    """SplitMix64-style mix of integers into a 63-bit generator seed."""
    h = 0x9E3779B97F4A7C15
    for v in vals:
        h = (h ^ (int(v) & _MASK64)) & _MASK64
        h = (h + 0x9E3779B97F4A7C15) & _MASK64
        z = h
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
        h = z ^ (z >> 31)
    return h & ((1 << 63) - 1)


_TAGS = {"u": 1, "q": 2, "k": 3, "v": 4, "sink": 5, "ctx": 6, "misc": 7}


def shift_coeffs(mean: float = -25.0, std: float = 3.0, d: int = DQK) -> tuple[float, float]:
    """alpha, beta such that (z_q + alpha u).(z_k - beta u)/sqrt(d) has the given mean and std."""
    prod = -mean * math.sqrt(d)            # alpha*beta
    ssum = d * (std * std - 1.0)           # alpha^2 + beta^2
    a = math.sqrt(ssum + 2 * prod)
    b = math.sqrt(ssum - 2 * prod)
    return (a - b) / 2.0, (a + b) / 2.0


class Synth:
    """Seeded draws for one layer of one workload."""

    def __init__(self, seed: int, layer: int = 0, dist: str = "shifted", device="cpu"):
        if dist not in ("shifted", "plain"):
            raise ValueError(dist)
        self.seed = int(seed)
        self.layer = int(layer)
        self.dist = dist
        self.device = torch.device(device)
        self.alpha, self.beta = shift_coeffs()

    def _gen(self, tag: str, *idx: int) -> torch.Generator:
        g = torch.Generator(device=self.device)
        g.manual_seed(_mix(self.seed, self.layer, _TAGS[tag], *idx))
        return g

    def _randn(self, shape, tag: str, *idx: int) -> torch.Tensor:
        return torch.randn(shape, generator=self._gen(tag, *idx), device=self.device,
                           dtype=torch.float32)

    def direction(self, hkv: int) -> torch.Tensor:
        """[hkv, 192] fp32 unit vectors, zero on the rotary dims 0..63."""
        u = torch.zeros(hkv, DQK, device=self.device)
        r = self._randn((hkv, DQK - DROT), "u")
        u[:, DROT:] = r / r.norm(dim=1, keepdim=True)
        return u

    def q(self, n: int, hq: int, hkv: int, seq: int = 0, start: int = 0) -> torch.Tensor:
        """[n, hq, 192] bf16 queries; (seq, start) index the draw."""
        z = self._randn((n, hq, DQK), "q", seq, start)
        if self.dist == "shifted":
            u = self.direction(hkv)
            z = z + self.alpha * u.repeat_interleave(hq // hkv, dim=0)[None]
        return z.to(torch.bfloat16)

    def k(self, n: int, hkv: int, seq: int = 0, start: int = 0) -> torch.Tensor:
        """[n, hkv, 192] bf16 raw (un-rotated) keys for positions start..start+n-1."""
        z = self._randn((n, hkv, DQK), "k", seq, start)
        if self.dist == "shifted":
            z = z - self.beta * self.direction(hkv)[None]
        return z.to(torch.bfloat16)

    def v(self, n: int, hkv: int, seq: int = 0, start: int = 0) -> torch.Tensor:
        """[n, hkv, 128] bf16 raw (unscaled) values."""
        return self._randn((n, hkv, DV), "v", seq, start).to(torch.bfloat16)

    def sinks(self, hq: int) -> torch.Tensor:
        """[hq] fp32 sink logits ~ N(1, 0.5)."""
        return 1.0 + 0.5 * self._randn((hq,), "sink")


def ragged_contexts(n: int, lo: int, hi: int, seed: int) -> list[int]:
    """n context lengths log-uniform over [lo, hi] (host ints, seeded)."""
    g = torch.Generator()
    g.manual_seed(_mix(seed, _TAGS["ctx"]))
    u = torch.rand((n,), generator=g, dtype=torch.float64)
    vals = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
    return [int(x) for x in vals.round().tolist()]
