"""RoPE position compensation of reused K, in fp64.

Sources:

* INMS walkthrough §3.2: a block stored from source position p_s and reused
  at position p_t needs its keys rotated by an extra angle that depends only
  on p_t - p_s; values need no compensation; rotation factors may be cached;
  prefix reuse from position 0 needs none.  §5.1: rotating the wrong way
  corrupts attention (the sign used here: K stored at p_s, reused at p_t, is
  rotated by +(p_t - p_s)).
* TokenDance summary, section 2: one batched RoPE call covers all requests of
  a compatible group.

The pages give no pairing convention or frequency formula.  The reading used
here is the rotate-half form used by Llama/Qwen-family models: dimension i is
paired with i + d/2 for i < d/2, with angular frequency theta^(-2i/d).
"""
from __future__ import annotations

import numpy as np


def inv_freq(head_dim: int, theta: float) -> np.ndarray:
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(np.float64(theta), -2.0 * i / head_dim)


def rotate(x: np.ndarray, delta, theta: float) -> np.ndarray:
    """Rotate the last axis of x (length d) by position shift delta."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    h = d // 2
    ang = np.float64(delta) * inv_freq(d, theta)
    c, s = np.cos(ang), np.sin(ang)
    lo, hi = x[..., :h], x[..., h:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


def rerotate_jobs(k_slab: np.ndarray, jobs: np.ndarray, src_table: np.ndarray,
                  dst_table: np.ndarray, block_tokens: int, theta: float):
    """Apply re-rotation jobs to a K slab [cap][Hkv][B][d] (fp64 values).

    Each job (src_row, src_tok0, dst_row, dst_tok0, n_tok, src_pos, dst_pos)
    reads token src_tok0+t of block-table row src_row and writes it, rotated
    by dst_pos - src_pos, to token dst_tok0+t of row dst_row of dst_table, for
    every KV head.  Returns (new slab, list of written (block, offset))."""
    B = block_tokens
    out = np.array(k_slab, dtype=np.float64, copy=True)
    written = []
    for (sr, st0, dr, dt0, n, sp, dp) in np.asarray(jobs)[:, :7]:
        delta = int(dp) - int(sp)
        for t in range(int(n)):
            ps = int(src_table[sr, (st0 + t) // B]); os_ = (st0 + t) % B
            pd = int(dst_table[dr, (dt0 + t) // B]); od = (dt0 + t) % B
            out[pd, :, od, :] = rotate(k_slab[ps, :, os_, :], delta, theta)
            written.append((pd, od))
    return out, written
