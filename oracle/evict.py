"""Block-granular MemDecay eviction scoring, in fp64.

Sources:

* MemDecay post §3.2: every region has an initial importance score and a
  decay factor; a token inherits its region's initial score when stored and
  its current score is  initial * exp(-decay * steps since it was stored);
  eviction sorts by current score and removes the lowest first.
* MemDecay post §4.1 (the cache's scoring code): a token that attention has
  accessed decays more slowly: the score is multiplied by
  (1 + 0.1 * ln(1 + access_count)) when the count is positive.
* MemDecay post §5.3: in a paged engine eviction works on whole blocks, a
  block being judged by the average score of its tokens.

Readings: a block's score is the mean over its stored tokens (the last block
of a sequence may be partial); a sequence evicts its k lowest-scored logical
blocks, ties going to the lower block index, reported in ascending block
order; "steps since stored" is step - created.

Test infrastructure only: nothing under shared_paged_kv_gb300/ imports this.
"""
from __future__ import annotations

import numpy as np


def token_scores(region, created, access, init, decay, step):
    """Current score of every token (arrays of equal shape)."""
    region = np.asarray(region, dtype=np.int64)
    init = np.asarray(init, dtype=np.float64)
    decay = np.asarray(decay, dtype=np.float64)
    age = np.float64(step) - np.asarray(created, dtype=np.float64)
    s = init[region] * np.exp(-decay[region] * age)
    acc = np.asarray(access, dtype=np.float64)
    return np.where(acc > 0, s * (1.0 + 0.1 * np.log1p(acc)), s)


def block_scores(region, created, access, seq_len, init, decay, step, block_tokens: int):
    """[n_seq][max_blocks] mean token score per logical block (+inf past the
    sequence's blocks)."""
    region = np.asarray(region)
    n_seq, max_tokens = region.shape
    max_blocks = max_tokens // block_tokens
    out = np.full((n_seq, max_blocks), np.inf)
    ts = token_scores(region, created, access, init, decay, step)
    for a in range(n_seq):
        L = int(seq_len[a])
        for b in range(-(-L // block_tokens)):
            t0, t1 = b * block_tokens, min(L, (b + 1) * block_tokens)
            out[a, b] = ts[a, t0:t1].mean()
    return out


def victims(scores, seq_len, k, block_tokens: int):
    """Per sequence the k lowest-scored blocks (ties: lower index), ascending."""
    idx, off = [], [0]
    for a in range(scores.shape[0]):
        nb = -(-int(seq_len[a]) // block_tokens)
        kk = max(0, min(int(k[a]), nb))
        order = sorted(range(nb), key=lambda b: (scores[a, b], b))
        idx.extend(sorted(order[:kk]))
        off.append(len(idx))
    return np.array(idx, dtype=np.int32), np.array(off, dtype=np.int64)
