"""Pins of the MemDecay eviction oracle: the post's §5.2 worked tuning value
(which fixes the exponential form and its sign), the access factor, block
means, and the victim rule against a brute force over subsets."""
import itertools
import math

import numpy as np

from oracle import evict as OE
import golden_io as G


def test_worked_tuning_value_fixes_the_decay_law():
    g = {r[0]: [float(x) for x in r[1:]] for r in G.rows("memdecay_tuning.txt")}
    thr, init, steps, printed = g["threshold"][0], g["init"][0], g["survive_steps"][0], g["decay"][0]
    decay = math.log(init / thr) / steps
    assert round(decay, 4) == printed
    # a token of that region, stored at step 0, is exactly at the threshold
    # after the survival span and above it one step earlier
    s_end = OE.token_scores([0], [0], [0], [init], [decay], steps)[0]
    s_before = OE.token_scores([0], [0], [0], [init], [decay], steps - 1)[0]
    assert abs(s_end - thr) < 1e-12 and s_before > thr


def test_region_order_and_zero_decay():
    init = [float(x) for x in G.rows("memdecay_tuning.txt")[-1][1:]]
    decay = [0.0, 0.001, 0.01, 0.05, 0.2]
    s = OE.token_scores(np.arange(5), np.zeros(5), np.zeros(5), init, decay, 40)
    assert s[0] == 100.0                      # no decay: kept for ever
    assert list(np.argsort(-s)) == [0, 1, 2, 3, 4]


def test_access_factor():
    s0 = OE.token_scores([0], [0], [0], [2.0], [0.0], 5)[0]
    s3 = OE.token_scores([0], [0], [3], [2.0], [0.0], 5)[0]
    assert s0 == 2.0 and abs(s3 - 2.0 * (1 + 0.1 * math.log(4.0))) < 1e-15


def test_block_mean_and_partial_block():
    region = np.array([[0, 1, 1, 1, 0, 0, 0, 0]])
    sc = OE.block_scores(region, np.zeros((1, 8)), np.zeros((1, 8)), [6], [1.0, 3.0], [0.0, 0.0], 0, 4)
    assert sc[0, 0] == (1 + 3 + 3 + 3) / 4
    assert sc[0, 1] == 1.0                    # tokens 4, 5 only
    assert math.isinf(OE.block_scores(region, np.zeros((1, 8)), np.zeros((1, 8)), [4], [1.0, 3.0],
                                      [0.0, 0.0], 0, 4)[0, 1])


def test_victims_are_the_lowest_by_brute_force():
    rng = np.random.default_rng(0)
    for trial in range(30):
        nb = int(rng.integers(1, 8))
        sc = rng.integers(0, 4, size=nb).astype(float)    # many ties
        k = int(rng.integers(0, nb + 1))
        idx, off = OE.victims(sc[None, :], [nb * 16], [k], 16)
        got = tuple(idx.tolist())
        best = None
        for sub in itertools.combinations(range(nb), k):
            key = (sorted(sc[list(sub)]), sorted(sub))
            if best is None or key < best[0]:
                best = (key, sub)
        assert got == tuple(sorted(best[1]))
