"""Mirror construction from refreshed critical positions, in fp64.

Sources:

* TokenDance summary, section 2: at the check layers the runtime finds each
  request's critical positions (where cached and newly computed values differ
  significantly) and refreshes only those positions of the request's cached
  K/V; the rest of the cache is reused as is.
* TokenDance summary, section 3 (Fig. 7): one dense master cache is kept and
  every other cache of the family is stored as a mirror holding only
  block-sparse K/V differences from the master; a block without a difference
  costs nothing but metadata.  On restore the diffs are applied and then the
  RoPE positions restored (Fig. 8), so a diff lives in the master's frame.

Readings (the pages fix the idea, not a format): an agent's mirror is its
block table into the shared master blocks plus a diff table; a logical block
is dirty when at least one of its positions was refreshed; dirty blocks get
consecutive diff ids in agent order, then logical-block order; inside a dirty
block the refreshed rows hold (refreshed value, taken back to the master's
frame) - (master value) and every other row holds zero.  A refreshed K row is
given in the agent's frame, so it is rotated by -delta of the segment covering
its block before the difference; V has no position.

Test infrastructure only: nothing under shared_paged_kv_gb300/ imports this.
"""
from __future__ import annotations

import numpy as np

from . import rope as _rope
from .attention import segment_delta_per_block


def mirror_build(block_table, idx, idx_off, k_new, v_new, k_pool, v_pool, block_tokens: int,
                 rope_off=None, rope_segs=None, theta: float = 1e4):
    """Diff table and block-sparse diffs of every agent's refreshed cache.

    idx / idx_off: per agent, the refreshed logical token positions (CSR, each
    agent's list ascending).  k_new / v_new: [n_rows][Hkv][d], row r holds the
    refreshed values of position idx[r].  Returns dict(diff_table int32
    [n_seq][max_blocks] (-1 = clean), n_diff, dk, dv fp64 [n_diff][Hkv][B][d]).
    """
    block_table = np.asarray(block_table)
    n_seq, max_blocks = block_table.shape
    B = block_tokens
    hkv, d = k_pool.shape[1], k_pool.shape[3]
    diff_table = np.full((n_seq, max_blocks), -1, dtype=np.int32)
    n_diff = 0
    for a in range(n_seq):
        dirty = sorted({int(t) // B for t in idx[idx_off[a]:idx_off[a + 1]]})
        for b in dirty:
            diff_table[a, b] = n_diff
            n_diff += 1
    dk = np.zeros((n_diff, hkv, B, d), dtype=np.float64)
    dv = np.zeros((n_diff, hkv, B, d), dtype=np.float64)
    for a in range(n_seq):
        deltas = segment_delta_per_block(max_blocks, rope_off, rope_segs, a)
        for r in range(int(idx_off[a]), int(idx_off[a + 1])):
            b, o = divmod(int(idx[r]), B)
            p = int(block_table[a, b])
            i = int(diff_table[a, b])
            kn = np.asarray(k_new[r], dtype=np.float64)
            if deltas[b] != 0:
                kn = _rope.rotate(kn, -int(deltas[b]), theta)
            dk[i, :, o, :] = kn - np.asarray(k_pool[p, :, o, :], dtype=np.float64)
            dv[i, :, o, :] = np.asarray(v_new[r], dtype=np.float64) - np.asarray(v_pool[p, :, o, :], dtype=np.float64)
    return dict(diff_table=diff_table, n_diff=n_diff, dk=dk, dv=dv)
