"""Plain CPU oracle of the KV rollback hand-off after verification.

TEST INFRASTRUCTURE ONLY (same rules as the rest of ``oracle/``: only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may use it; it shares no code with the CUDA path).

Source: the speculative-decoding tutorial page at dpshk.com/news/5598276
("P3"), §5.4 (KV-cache management after a rejection): the KV entries of the
drafted tokens are written first and marked tentative; after verification the
cache is cut at num_accepted and the blocks past the cut go back to the block
pool; the KV of the corrected token is computed in the next step.  The page
describes the behaviour of a paged KV cache (PagedAttention blocks) without a
layout; the readings below are this repository's:

- request b had seq_lens[b] = L committed tokens before the drafts; its g
  drafts (draft_lens[b], else gamma_max) occupy positions L .. L + g - 1, so
  ceil((L + g) / block_size) blocks of block_tables[b] were in use;
- k = num_accepted[b] drafts are kept (k < 0 marks a request with invalid
  data: none of its drafts is kept, k = 0), so ceil((L + k) / block_size)
  blocks stay; the emitted token at position k has no KV yet;
- every block index j in [kept, used) whose entry is a block id (>= 0) is
  appended to the free list, request after request and in increasing j, and
  its entry becomes -1; seq_lens[b] becomes L + k;
- a request with an invalid draft length or a negative length is left as it
  is and sets STATUS_BAD_LENGTH; entries past max_blocks are not touched and
  set STATUS_TABLE_SHORT; an entry that should hold a block but is -1 sets
  STATUS_MISSING_BLOCK; a block that does not fit in the free list stays in
  the table and sets STATUS_FREE_LIST_FULL.
The CUDA path may append the freed ids in any order; everything else is
unique.
"""
from __future__ import annotations

import numpy as np

STATUS_FREE_LIST_FULL = 1
STATUS_MISSING_BLOCK = 2
STATUS_BAD_LENGTH = 4
STATUS_TABLE_SHORT = 8


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def kv_rollback(num_accepted, seq_lens, block_tables, block_size, free_list, free_count,
                draft_lens=None, gamma_max=None):
    """Return (seq_lens, block_tables, free_list, free_count, status), new
    arrays; the inputs are not modified."""
    nacc = np.asarray(num_accepted, dtype=np.int64)
    lens_in = np.asarray(seq_lens, dtype=np.int64)
    tables = np.array(block_tables, dtype=np.int64, copy=True)
    free = np.array(free_list, dtype=np.int64, copy=True)
    count = int(free_count)
    B, max_blocks = tables.shape
    g_max = int(gamma_max) if gamma_max is not None else None
    out_lens = lens_in.copy()
    status = 0
    for b in range(B):
        g = int(draft_lens[b]) if draft_lens is not None else g_max
        L = int(lens_in[b])
        if g is None or g < 0 or (g_max is not None and g > g_max) or L < 0:
            status |= STATUS_BAD_LENGTH
            continue
        k = int(nacc[b])
        k = 0 if k < 0 else min(k, g)
        used = _ceil_div(L + g, block_size)
        kept = _ceil_div(L + k, block_size)
        if used > max_blocks:
            status |= STATUS_TABLE_SHORT
            used = max_blocks
        for j in range(kept, used):
            blk = int(tables[b, j])
            if blk < 0:
                status |= STATUS_MISSING_BLOCK
                continue
            if count >= free.size:
                status |= STATUS_FREE_LIST_FULL
                continue
            free[count] = blk
            count += 1
            tables[b, j] = -1
        out_lens[b] = L + k
    return out_lens, tables, free, count, status


def rollback_by_positions(num_accepted, seq_lens, block_tables, block_size, draft_lens):
    """Brute-force restatement for tiny cases: mark every token position a
    block covers, drop the positions of rejected drafts, and free the blocks
    left without any position.  Returns (seq_lens, freed ids per request)."""
    tables = np.asarray(block_tables)
    out_lens, freed = [], []
    for b in range(tables.shape[0]):
        L, g = int(seq_lens[b]), int(draft_lens[b])
        k = max(0, min(int(num_accepted[b]), g))
        live = set(range(L + k))  # committed tokens plus the kept drafts
        blocks_used = {pos // block_size for pos in range(L + g)}
        blocks_live = {pos // block_size for pos in live}
        freed.append(sorted(int(tables[b, j]) for j in blocks_used - blocks_live))
        out_lens.append(L + k)
    return np.array(out_lens), freed
