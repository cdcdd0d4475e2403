"""Pool management of a windowed layer kept in pages: the plain definitions.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
path never imports it and shares no code with it.

Integer and bit-copy work, written with plain Python loops over lists and
numpy arrays (no vectorised shortcuts), so each step can be read against
its source:

* ``release_window`` -- Xiaomi "Full-Pipeline Inference Optimization for
  MiMo-V2.5 Series", section 2.1, "SWA KVCache Management" (the SWA pool
  keeps only the window and releases the rest by the window) and
  "SWA-Aware Prefix Cache Tree" (the end of a prefill chunk, the end of a
  request and every N decoded tokens trigger the release of SWA KV that has
  left the window); gaudi-cookbook "MiMo-V2.6-Flash on Gaudi 2", "Windowed
  KV groups" (vLLM's hybrid manager frees the sliding layers' out-of-window
  blocks).  A query at position q of a windowed layer attends positions
  q-W+1..q (colibri "What the engine implements"; gaudi-cookbook "What was
  built": exactly the last 128 positions), so once the next query of a
  sequence is at position P no later query reads a position below P-W+1,
  and a block all of whose positions lie below P-W+1 can go.
* ``ring_from_pages`` -- colibri "System One mode and prompt reuse": position
  p of a windowed layer lives in ring slot p mod 128 and the ring records the
  position each slot holds.  The ring a sequence has after its positions
  0..E-1 were appended in order holds, in slot c, the last of those positions
  congruent to c mod 128; this builds that ring from a paged copy of the same
  rows.

Pins (tests/test_oracle_pins.py): a worked example written out by hand
(tests/golden/pages_release_example.txt); a brute-force check of every block
against the windows of all later queries; the ring built by appending the
positions one by one.
"""
from __future__ import annotations

import numpy as np

WINDOW = 128

# status bits (the same meaning as the library's device status word)
BAD_SEQ, BAD_BLOCK, FREE_FULL = 2, 4, 32


def release_window(block_table, num_blocks, block_size, seqs, next_pos, window, lo=None,
                   free_ids=None, free_count=0, free_cap=None):
    """Release the blocks of a paged windowed pool that no later query reads.

    block_table: list of per-sequence lists (or a 2-D int array) of block ids,
      -1 = no block.  num_blocks: ids outside [0, num_blocks) are not released
      (ids >= num_blocks set BAD_BLOCK).
    seqs[i], next_pos[i]: sequence seqs[i]'s next query is at next_pos[i].
    lo: per-sequence count of leading table entries already released (or
      None = 0); entries below it are not looked at again.
    free_ids / free_count / free_cap: the free list the released ids are
      appended to, its current length and its capacity (None = unbounded).
      If the ids released by the whole call would not fit, nothing changes
      and FREE_FULL is returned.

    Returns (table, lo, free_ids, free_count, flags), all new objects.
    Entries are visited in the order (i, block index), which is the order the
    released ids are appended in.
    """
    table = [list(int(x) for x in row) for row in block_table]
    max_blocks = len(table[0]) if table else 0
    lo_new = None if lo is None else [int(x) for x in lo]
    ids = [] if free_ids is None else [int(x) for x in free_ids]
    flags = 0
    released = []      # (seq, block index, id) in visiting order
    bounds = []        # (seq, bound) per entry
    for i in range(len(seqs)):
        s = int(seqs[i])
        if s < 0 or s >= len(table):
            flags |= BAD_SEQ
            continue
        first_kept = int(next_pos[i]) - window + 1   # earliest position a later query reads
        bound = first_kept // block_size if first_kept > 0 else 0   # blocks [0, bound) hold only earlier ones
        bound = min(bound, max_blocks)
        start = 0 if lo_new is None else min(max(lo_new[s], 0), max_blocks)
        for bi in range(start, bound):
            b = table[s][bi]
            if 0 <= b < num_blocks:
                released.append((s, bi, b))
            elif b >= num_blocks:
                flags |= BAD_BLOCK
        bounds.append((s, bound))
    if free_cap is not None and free_count + len(released) > free_cap:
        # all or nothing: the call changes no table entry, no lo and no free-list entry
        return ([[int(x) for x in row] for row in block_table], None if lo is None else [int(x) for x in lo],
                ids, free_count, flags | FREE_FULL)
    for j, (s, bi, b) in enumerate(released):
        table[s][bi] = -1
        at = free_count + j
        if at < len(ids):
            ids[at] = b
        else:
            ids.append(b)
    if lo_new is not None:
        for s, bound in bounds:
            lo_new[s] = max(lo_new[s], bound)
    return table, lo_new, ids, free_count + len(released), flags


def ring_slot_position(end: int, c: int, window: int = WINDOW) -> int:
    """The position ring slot c holds after positions 0..end-1 were appended in
    order: the largest p < end with p mod window == c, or -1 if there is none."""
    best = -1
    for p in range(max(0, end - window), end):
        if p % window == c:
            best = p
    return best


def ring_from_pages(pages_k, pages_v, block_table, block_size, src_seq, end, ring_k, ring_v, ring_tags):
    """Fill one sequence's ring (k [Hkv][128][192], v [Hkv][128][128] bf16 bits,
    tags [128]) from a paged pool (k [nblk][Hkv][bsz][192], v [..][128]):
    slot c gets the row of position ring_slot_position(end, c) of sequence
    src_seq, its tag that position; slots with no position get tag -1 and
    keep their rows.  A needed position whose block entry is not a valid
    block id also gets tag -1 (and BAD_BLOCK).  Works on copies; returns
    (k, v, tags, flags)."""
    k, v, tags = np.array(ring_k, copy=True), np.array(ring_v, copy=True), np.array(ring_tags, copy=True)
    nblk = pages_k.shape[0]
    max_blocks = len(block_table[src_seq])
    flags = 0
    for c in range(WINDOW):
        p = ring_slot_position(int(end), c)
        if p < 0:
            tags[c] = -1
            continue
        bi = p // block_size
        b = int(block_table[src_seq][bi]) if bi < max_blocks else -1
        if not (0 <= b < nblk):
            tags[c] = -1
            flags |= BAD_BLOCK
            continue
        for h in range(k.shape[0]):
            k[h, c, :] = pages_k[b, h, p % block_size, :]
            v[h, c, :] = pages_v[b, h, p % block_size, :]
        tags[c] = p
    return k, v, tags, flags
