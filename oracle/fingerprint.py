"""Block fingerprints and deduplication into a shared physical block pool.

Sources:

* shared-memory KV pool post, §3.2 (CalcHash): a 64-bit FNV-1a-style hash
  whose offset basis is 1469598103934665603 and whose prime is
  1099511628211.  Each whole 32-bit token id is XORed in and the state is
  multiplied by the prime (mod 2^64); finally a tag is XORed in and the state
  multiplied once more.  The page's tag is a layer id; here the tag is the
  memory tier, because the INMS walkthrough §5.1 folds the tier into the
  block fingerprint so that blocks of different tiers never match.  Note the
  page's offset basis differs from the textbook FNV value; the page is
  followed as printed.
* INMS walkthrough §2.2 and §3.2: fixed-size blocks; a block is reused from
  the shared pool only when the content, the tier and the position range are
  compatible; sharing runs up to the first divergence and every later block
  of the sequence is private.  The shared-memory post §3.3 (FindMatchLength)
  states the same longest-prefix rule.
* TokenDance summary, section 1: with explicit segment boundaries, hashing
  becomes segment-based, so a shared segment maps to the same cached blocks
  whatever its absolute position.

Dedup rule used here (the plainest reading of the above): two full blocks
(s, b) and (s', b') share one physical block iff their sequences have the
same tier, the tier is not PRIVATE, both blocks sit at the same index k inside
their hashed segment, and the token runs from their segment starts through
the end of the blocks are identical.  Without segment boundaries every
sequence is one segment starting at block 0, which is the prefix rule.
Partial tail blocks and PRIVATE-tier blocks always get a fresh physical
block.  Physical ids are assigned in first-occurrence order scanning
sequences 0..N-1 and, inside each, blocks 0, 1, ...; refcount[id] is the
number of (sequence, block) slots that map to id.
"""
from __future__ import annotations

import numpy as np

FNV_OFFSET = 1469598103934665603
FNV_PRIME = 1099511628211
MASK64 = (1 << 64) - 1
PRIVATE_TIER = 0xFFFFFFFF


def calc_hash(token_ids, tag: int) -> int:
    """CalcHash of the shared-memory KV pool post §3.2 (tag = tier)."""
    h = FNV_OFFSET
    for t in token_ids:
        h ^= int(t) & 0xFFFFFFFF
        h = (h * FNV_PRIME) & MASK64
    h ^= int(tag) & 0xFFFFFFFF
    h = (h * FNV_PRIME) & MASK64
    return h


def _segment_starts(seg_start_off, seg_start_blocks, s):
    if seg_start_off is None:
        return [0]
    st = sorted(set([0] + [int(x) for x in seg_start_blocks[seg_start_off[s]:seg_start_off[s + 1]]]))
    return st


def dedup(tokens, seq_off, tier, block_tokens: int, max_blocks: int,
          seg_start_off=None, seg_start_blocks=None):
    """Returns dict(fp [N][max_blocks] uint64 (0 for non-full blocks),
    block_table [N][max_blocks] int32 (-1 unused), refcount [n_phys] int32,
    n_phys int, owner [n_phys] (sequence of first occurrence))."""
    B = block_tokens
    n = len(seq_off) - 1
    tokens = np.asarray(tokens, dtype=np.uint32)
    if tier is None:
        tier = np.zeros(n, dtype=np.uint32)
    fp = np.zeros((n, max_blocks), dtype=np.uint64)
    table = np.full((n, max_blocks), -1, dtype=np.int32)
    classes = {}
    refcount = []
    owner = []
    for s in range(n):
        base = int(seq_off[s])
        length = int(seq_off[s + 1]) - base
        nblk = -(-length // B)
        full = length // B
        if nblk > max_blocks:
            raise ValueError("sequence longer than max_blocks blocks")
        starts = _segment_starts(seg_start_off, seg_start_blocks, s)
        seq = tokens[base:base + length]
        t = int(tier[s])
        for b in range(nblk):
            if b < full:
                fp[s, b] = calc_hash(seq[b * B:(b + 1) * B], t)
            shareable = b < full and t != PRIVATE_TIER
            pid = None
            if shareable:
                st = max(x for x in starts if x <= b)
                key = (t, b - st, seq[st * B:(b + 1) * B].tobytes())
                pid = classes.get(key)
                if pid is None:
                    pid = len(refcount)
                    classes[key] = pid
                    refcount.append(0)
                    owner.append(s)
            else:
                pid = len(refcount)
                refcount.append(0)
                owner.append(s)
            table[s, b] = pid
            refcount[pid] += 1
    return dict(fp=fp, block_table=table, refcount=np.array(refcount, dtype=np.int32),
                n_phys=len(refcount), owner=np.array(owner, dtype=np.int32))


def references(block_table, n_phys: int):
    """The references of every physical block as a CSR.

    INMS walkthrough §2.2: a physical block's reference count is the number of
    sequence blocks that point at it, and the block is shared while that
    count exceeds one; §3.3: the engine's hooks walk these references.
    Returns (off [n_phys + 1] int64, seq [total] int32): seq[off[p]:off[p+1]]
    are the sequences s of the slots (s, b) whose table entry is p, in
    ascending (s, b) order (a sequence appears once per slot)."""
    table = np.asarray(block_table)
    lists = [[] for _ in range(n_phys)]
    for s in range(table.shape[0]):
        for b in range(table.shape[1]):
            p = int(table[s, b])
            if p >= 0:
                lists[p].append(s)
    off, seq = [0], []
    for p in range(n_phys):
        seq.extend(lists[p])
        off.append(len(seq))
    return np.array(off, dtype=np.int64), np.array(seq, dtype=np.int32)


def find_match_length(input_ids, checkpoint_len: int, pool_hashes, tag: int = 0) -> int:
    """Longest matched prefix (in tokens) against a set of stored block
    hashes, scanning checkpoints from 0 and stopping at the first miss —
    shared-memory KV pool post §3.3."""
    matched = 0
    c = 0
    while c + checkpoint_len <= len(input_ids):
        if calc_hash(input_ids[c:c + checkpoint_len], tag) not in pool_hashes:
            break
        matched += checkpoint_len
        c += checkpoint_len
    return matched
