"""The no-allocation variant of the full-attention decode.

Callers that are handed only input and output buffers (no allocator, no
workspace) use full_attn_decode_noalloc, whose split partials live in a fixed
array inside the library.  Its results must match full_attn_decode (which
takes a caller-owned workspace) within the parity tolerance, on consecutive
calls that reuse the array.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import sinks_kv_ring_gb300 as kvr
from sinks_kv_ring_gb300.synth import Synth

from kvr_cases import SCALE, compare, fill_paged

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sinks_kv_ring_gb300 import build
    build.build()
    table = kvr.rope_table(1e7, 8192)
    return table


def test_noalloc_decode_matches_workspace_decode_on_two_calls(setup):
    table = setup
    hq, hkv, max_ctx = 64, 4, 8192
    ctx = [1, 17, 64, 65, 1000, 4097, 8192]
    B = len(ctx)
    syn = Synth(4242, dist="plain", device=DEV)
    pool = kvr.PagedLayout.contiguous(B, hkv, max_ctx, block_size=64)
    fill_paged(pool, syn, list(range(B)), ctx, table, 0.707)
    pos = torch.tensor([c - 1 for c in ctx], dtype=torch.int64, device=DEV)
    seq = torch.arange(B, dtype=torch.int32, device=DEV)
    for call in range(2):
        q = syn.q(B, hq, hkv, seq=100 + call)
        want = kvr.full_attn_decode(q, pos, seq, pool, table, SCALE, max_ctx)
        got = kvr.full_attn_decode_noalloc(q, pos, seq, pool, table, SCALE, max_ctx)
        torch.cuda.synchronize()
        compare(got, want.double().cpu().numpy(), f"noalloc call {call}")


def test_noalloc_decode_rejects_batches_past_the_scratch_size(setup):
    # partials of 2048 sequences x 4 KV heads x 16 q heads at one split each: 68 MB
    B, max_ctx = 2048, 131072
    need = kvr.full_attn_decode_workspace_size(B, 64, 4, max_ctx)
    assert need > kvr.NOALLOC_SCRATCH_BYTES
    table = torch.zeros(max_ctx, 32, 2, dtype=torch.float32, device=DEV)
    pool = kvr.PagedLayout.contiguous(1, 4, max_ctx, block_size=64)
    q = torch.zeros(B, 64, 192, dtype=torch.bfloat16, device=DEV)
    pos = torch.zeros(B, dtype=torch.int64, device=DEV)
    seq = torch.zeros(B, dtype=torch.int32, device=DEV)
    with pytest.raises(kvr.KvrError) as e:
        kvr.full_attn_decode_noalloc(q, pos, seq, pool, table, SCALE, max_ctx)
    assert e.value.code == -3 and "scratch" in str(e.value)
