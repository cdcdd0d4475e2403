"""The no-allocation variant of the full-attention decode.

Some callers are handed only their input and output buffers and may not
allocate device memory: a plugin whose host owns all device memory, or a
server that reserves the whole GPU for its KV pools at start-up.  For them
full_attn_decode_noalloc keeps its split partials in a fixed array inside the
library instead of a caller-owned workspace.  It runs the same kernels with
the same split plan as full_attn_decode, so its output must be bit-equal to
it, on consecutive calls that reuse the array -- a larger batch first, then a
smaller one with another split plan, so that a merge reading partials left
over from the earlier call would show.  The array's address is looked up by
the first call on a device, which must not run inside a stream capture: in a
fresh process, such a call is refused with a message that says so.  This file
is collected last on purpose.
"""
import os
import subprocess
import sys

import pytest
import torch

import sinks_kv_ring_gb300 as kvr
from sinks_kv_ring_gb300.synth import Synth

from kvr_cases import SCALE, fill_paged

pytestmark = pytest.mark.gpu
DEV = "cuda"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sinks_kv_ring_gb300 import build
    build.build()
    return kvr.rope_table(1e7, 16384)


def test_noalloc_decode_equals_workspace_decode_large_then_small(setup):
    table = setup
    hq, hkv = 64, 4
    cases = [
        # 48 sequences up to 16384 tokens: many splits and partials
        ([1 + (977 * b) % 16384 for b in range(47)] + [16384], 16384, 5101),
        # then 5 short ones (another split plan, fewer partials)
        ([1, 17, 64, 65, 1000], 4096, 5102),
    ]
    for call, (ctx, max_ctx, seed) in enumerate(cases):
        B = len(ctx)
        syn = Synth(seed, dist="plain", device=DEV)
        pool = kvr.PagedLayout.contiguous(B, hkv, max_ctx, block_size=64)
        fill_paged(pool, syn, list(range(B)), ctx, table, 0.707)
        pos = torch.tensor([c - 1 for c in ctx], dtype=torch.int64, device=DEV)
        seq = torch.arange(B, dtype=torch.int32, device=DEV)
        q = syn.q(B, hq, hkv, seq=100 + call)
        want = kvr.full_attn_decode(q, pos, seq, pool, table, SCALE, max_ctx)
        got = kvr.full_attn_decode_noalloc(q, pos, seq, pool, table, SCALE, max_ctx)
        torch.cuda.synchronize()
        assert torch.equal(got, want), f"call {call} (B={B}) differs from full_attn_decode"
    assert kvr.device_status() == 0


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


_FIRST_CALL_IN_CAPTURE = r"""
import sys, torch
sys.path.insert(0, sys.argv[1])
import sinks_kv_ring_gb300 as kvr
table = kvr.rope_table(1e7, 256)
pool = kvr.PagedLayout.contiguous(1, 4, 256, block_size=64)
q = torch.zeros(1, 64, 192, dtype=torch.bfloat16, device="cuda")
pos = torch.zeros(1, dtype=torch.int64, device="cuda")
seq = torch.zeros(1, dtype=torch.int32, device="cuda")
out = torch.empty(1, 64, 128, dtype=torch.bfloat16, device="cuda")
torch.cuda.synchronize()
g = torch.cuda.CUDAGraph()
try:
    with torch.cuda.graph(g):
        kvr.full_attn_decode_noalloc(q, pos, seq, pool, table, 0.1, 1, out=out)
except kvr.KvrError as e:
    print("REFUSED", e.code, str(e).replace("\n", " "))
    sys.exit(0)
except Exception as e:  # the capture may report the refusal on its own way out
    print("OTHER", type(e).__name__, str(e).replace("\n", " "))
    sys.exit(0)
print("ACCEPTED")
"""


def test_first_noalloc_call_inside_a_capture_is_refused(setup):
    # a fresh process: nothing of the library has run on the device yet
    r = subprocess.run([sys.executable, "-c", _FIRST_CALL_IN_CAPTURE, ROOT], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = [ln for ln in r.stdout.splitlines() if ln.startswith(("REFUSED", "OTHER", "ACCEPTED"))]
    assert line and line[0].startswith("REFUSED -1 "), r.stdout[-2000:] + r.stderr[-2000:]
    assert "before capturing" in line[0]
