"""Decode-step attention over a shared paged KV pool, in fp64.

Sources:

* INMS walkthrough §2.2 (block table mapping[seq][position] -> physical
  block, shared blocks referenced by many sequences) and §3.2 (K of a reused
  segment is rotated by the position shift; V is not).
* TokenDance summary, section 3 (Fig. 7, Fig. 8): one dense master cache; each
  other cache of the family is a mirror that stores only block-sparse K/V
  differences; on restore, blocks with a difference are corrected before
  attention and their RoPE positions restored — the order being "apply the
  block-sparse diffs, then restore RoPE positions".
* MemDecay post §4.2: scores are q.k / sqrt(head_dim), softmax, weighted sum
  of V.

The oracle materialises every agent's dense K and V (master + diff, then
rotation), exactly the thing the fused GPU path never builds, and evaluates
softmax(q K^T * scale) V with fp64 accumulation.  Readings: the diff is
additive in the master's frame; query heads map to KV heads in contiguous
groups (kv = h // (Hq/Hkv)); the decode query is already position-encoded and
attends to every cached position with no mask; an empty context gives a zero
output.
"""
from __future__ import annotations

import numpy as np

from . import rope as _rope


def segment_delta_per_block(max_blocks: int, rope_off, rope_segs, a: int) -> np.ndarray:
    """Per logical block of agent a, the RoPE shift of the segment covering it
    (0 outside every segment)."""
    out = np.zeros(max_blocks, dtype=np.int64)
    if rope_off is None:
        return out
    for (fb, nb, delta, _) in np.asarray(rope_segs)[rope_off[a]:rope_off[a + 1]]:
        out[fb:fb + nb] = delta
    return out


def materialise(a: int, seq_len: int, k_pool, v_pool, block_table, block_tokens: int,
                diff_table=None, dk_pool=None, dv_pool=None,
                rope_off=None, rope_segs=None, theta: float = 1e4, diff_block_tokens=None):
    """Dense fp64 K, V of agent a: [L][Hkv][d].  Mirror diffs are kept per
    diff block of diff_block_tokens tokens (default: the pool's block size):
    diff_table[a, t // diff_block_tokens] names the diff block holding token
    t's differences at row t % diff_block_tokens."""
    B = block_tokens
    DB = B if diff_block_tokens is None else diff_block_tokens
    hkv, d = k_pool.shape[1], k_pool.shape[3]
    K = np.zeros((seq_len, hkv, d), dtype=np.float64)
    V = np.zeros((seq_len, hkv, d), dtype=np.float64)
    deltas = segment_delta_per_block(block_table.shape[1], rope_off, rope_segs, a)
    for t in range(seq_len):
        b, o = divmod(t, B)
        p = int(block_table[a, b])
        k = np.array(k_pool[p, :, o, :], dtype=np.float64)
        v = np.array(v_pool[p, :, o, :], dtype=np.float64)
        db, do = divmod(t, DB)
        if diff_table is not None and diff_table[a, db] >= 0:
            q = int(diff_table[a, db])
            k = k + dk_pool[q, :, do, :]
            v = v + dv_pool[q, :, do, :]
        if deltas[b] != 0:
            k = _rope.rotate(k, int(deltas[b]), theta)
        K[t] = k
        V[t] = v
    return K, V


def attend(q, K, V, scale: float) -> np.ndarray:
    """softmax(q . K_t * scale) weighted sum of V_t, fp64; q [d], K,V [L][d]."""
    if K.shape[0] == 0:
        return np.zeros(q.shape[-1], dtype=np.float64)
    s = (K @ np.asarray(q, dtype=np.float64)) * scale
    s = s - s.max()
    p = np.exp(s)
    p /= p.sum()
    return p @ V


def decode_attention(q, k_pool, v_pool, block_table, seq_len, block_tokens: int, scale: float,
                     diff_table=None, dk_pool=None, dv_pool=None,
                     rope_off=None, rope_segs=None, theta: float = 1e4, agents=None, heads=None,
                     diff_block_tokens=None):
    """out [N][Hq][d] fp64 (rows not in ``agents``/``heads`` stay zero)."""
    q = np.asarray(q, dtype=np.float64)
    n, hq, d = q.shape
    hkv = k_pool.shape[1]
    g = hq // hkv
    out = np.zeros((n, hq, d), dtype=np.float64)
    agents = range(n) if agents is None else agents
    for a in agents:
        K, V = materialise(a, int(seq_len[a]), k_pool, v_pool, block_table, block_tokens,
                           diff_table, dk_pool, dv_pool, rope_off, rope_segs, theta, diff_block_tokens)
        for h in (range(hq) if heads is None else heads):
            out[a, h] = attend(q[a, h], K[:, h // g, :], V[:, h // g, :], scale)
    return out
