"""Critical-position selection by K difference, in fp64.

Source: TokenDance summary, section 2 — at check layers one batched
difference computation finds, for every request, the positions whose cached
and newly computed values differ most, and only those are refreshed.

Readings: the difference of a position is the L2 norm of K_cached - K_new
over all KV heads and head dims of that position; the number kept per agent is
k = ceil(ratio * n) (ratio taken as the float32 value passed in, the product
formed in fp64); ties are broken toward the lower position; the selected
positions are returned in ascending order, relative to the agent's first row.
"""
from __future__ import annotations

import math

import numpy as np


def count_for(ratio: float, n: int) -> int:
    k = math.ceil(float(np.float32(ratio)) * n)
    return max(0, min(n, k))


def scores(k_cached: np.ndarray, k_new: np.ndarray) -> np.ndarray:
    diff = np.asarray(k_cached, np.float64) - np.asarray(k_new, np.float64)
    return np.sqrt(np.sum(diff * diff, axis=-1))


def select_critical(k_cached, k_new, row_off, ratio: float):
    """Returns (idx [sum k_a] int32, idx_off [n_agents+1] int64, scores fp64)."""
    sc = scores(k_cached, k_new)
    out, off = [], [0]
    for a in range(len(row_off) - 1):
        s = sc[row_off[a]:row_off[a + 1]]
        n = len(s)
        k = count_for(ratio, n)
        order = sorted(range(n), key=lambda t: (-s[t], t))
        out.extend(sorted(order[:k]))
        off.append(off[-1] + k)
    return np.array(out, dtype=np.int32), np.array(off, dtype=np.int64), sc
