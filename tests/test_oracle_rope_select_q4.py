"""Pins of oracle.rope, oracle.select and oracle.q4."""
import itertools
from fractions import Fraction

import numpy as np
import pytest

from oracle import rope as R, select as S, q4 as Q
from shared_paged_kv_gb300.workloads import f32_to_bf16_bits, bf16_bits_to_f32


# ---------------------------------------------------------------- RoPE ----
def complex_rotate_at(x, pos, theta):
    """Position-encode x at absolute position pos by complex multiplication
    of the pairs (x_i, x_{i+d/2}) with exp(i * pos * theta^(-2i/d))."""
    d = x.shape[-1]
    h = d // 2
    w = theta ** (-2.0 * np.arange(h) / d)
    z = (x[..., :h] + 1j * x[..., h:]) * np.exp(1j * pos * w)
    return np.concatenate([z.real, z.imag], axis=-1)


def test_rope_zero_is_identity():
    x = np.random.default_rng(0).standard_normal((3, 128))
    assert np.array_equal(R.rotate(x, 0, 1e6), x)


def test_rope_frequencies_closed_form():
    w = R.inv_freq(128, 1e6)
    assert w[0] == 1.0
    np.testing.assert_allclose(w[1:] / w[:-1], 1e6 ** (-2 / 128), rtol=1e-12)


@pytest.mark.parametrize("ps,pt", [(0, 5), (128, 4000), (6000, 300), (7, 7)])
def test_rope_shift_direction(ps, pt):
    # A key stored at p_s and reused at p_t, rotated by +(p_t - p_s), equals
    # the key encoded at p_t directly (the INMS failure story was exactly a
    # wrong rotation direction).
    k = np.random.default_rng(ps + pt).standard_normal((4, 128))
    stored = complex_rotate_at(k, ps, 1e6)
    np.testing.assert_allclose(R.rotate(stored, pt - ps, 1e6), complex_rotate_at(k, pt, 1e6), atol=1e-9)


def test_rope_composes_and_preserves_norm():
    x = np.random.default_rng(1).standard_normal(64)
    np.testing.assert_allclose(R.rotate(R.rotate(x, 37, 1e4), -12, 1e4), R.rotate(x, 25, 1e4), atol=1e-12)
    np.testing.assert_allclose(np.linalg.norm(R.rotate(x, 999, 1e4)), np.linalg.norm(x), rtol=1e-12)


def test_rope_query_side_identity():
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    assert abs(q @ R.rotate(k, 1234, 1e6) - R.rotate(q, -1234, 1e6) @ k) < 1e-10


def test_rerotate_jobs_writes_only_destinations():
    rng = np.random.default_rng(3)
    B, cap = 4, 10
    slab = rng.standard_normal((cap, 2, B, 8))
    src = np.array([[0, 1, 2]], dtype=np.int32)
    dst = np.array([[-1, 7, 8]], dtype=np.int32)
    jobs = np.array([[0, 2, 0, 5, 6, 100, 103, 0]], dtype=np.int32)  # tokens 2..7 -> 5..10
    out, written = R.rerotate_jobs(slab, jobs, src, dst, B, 1e4)
    assert len(written) == 6
    for t in range(6):
        ps, os_ = src[0, (2 + t) // B], (2 + t) % B
        pd, od = dst[0, (5 + t) // B], (5 + t) % B
        np.testing.assert_allclose(out[pd, :, od], complex_rotate_at(slab[ps, :, os_], 3, 1e4), atol=1e-12)
    mask = np.ones(out.shape[:1] + out.shape[2:3], bool)
    for (p, o) in written:
        mask[p, o] = False
    for p in range(cap):
        for o in range(B):
            if mask[p, o]:
                assert np.array_equal(out[p, :, o], slab[p, :, o])


# ----------------------------------------------------------- selection ----
def test_select_count_rule():
    assert S.count_for(0.15, 8192) == 1229
    assert S.count_for(0.15, 0) == 0
    assert S.count_for(1.0, 7) == 7
    assert S.count_for(0.0, 7) == 0


@pytest.mark.parametrize("seed", range(6))
def test_select_is_best_subset(seed):
    # top-k by score = the k-subset with the largest score sum (distinct scores)
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 10))
    kc = rng.standard_normal((n, 6))
    kn = kc + rng.standard_normal((n, 6)) * rng.uniform(0.1, 1, (n, 1))
    idx, off, sc = S.select_critical(kc, kn, np.array([0, n]), 0.35)
    k = S.count_for(0.35, n)
    best = max(itertools.combinations(range(n), k), key=lambda c: sum(np.linalg.norm(kc[list(c)] - kn[list(c)], axis=1)))
    assert list(idx) == sorted(best)
    assert list(off) == [0, k]


def test_select_planted_positions():
    rng = np.random.default_rng(7)
    rows = [50, 80]
    kc = rng.standard_normal((130, 32))
    kn = kc.copy()
    planted = {0: [3, 17, 40], 1: [0, 5, 33, 60, 79]}
    for a, ps in planted.items():
        base = 0 if a == 0 else 50
        for p in ps:
            kn[base + p] += 5.0
    # ratio so that k equals the number planted in each agent
    idx, off, _ = S.select_critical(kc[:50], kn[:50], np.array([0, 50]), 3 / 50)
    assert list(idx) == planted[0]
    idx, off, _ = S.select_critical(kc[50:], kn[50:], np.array([0, 80]), 5 / 80)
    assert list(idx) == planted[1]


def test_select_ties_prefer_lower_position():
    kc = np.zeros((6, 4))
    kn = np.ones((6, 4))           # all scores equal
    idx, _, _ = S.select_critical(kc, kn, np.array([0, 6]), 0.5)
    assert list(idx) == [0, 1, 2]


# ------------------------------------------------------------------ Q4 ----
def test_q4_hand_example():
    x = (np.arange(64) % 16).astype(np.float32)[None, :]
    codes, sb = Q.quantize(x)
    assert sb[0, 0, 0] == 1.0 and sb[0, 0, 1] == 0.0
    assert codes[0, 0] == 0x10 and codes[0, 1] == 0x32 and codes[0, 7] == 0xFE
    assert np.array_equal(Q.dequantize(codes, sb), x.astype(np.float64))


def test_q4_constant_group():
    x = np.full((1, 128), 0.3, np.float32)
    codes, sb = Q.quantize(x)
    assert (codes == 0).all() and (sb[..., 0] == 0).all()
    assert np.all(Q.dequantize(codes, sb) == float(np.float16(0.3)))


def test_q4_error_bound_and_range():
    rng = np.random.default_rng(4)
    x = bf16_bits_to_f32(f32_to_bf16_bits(rng.standard_normal((200, 128)).astype(np.float32)))
    codes, sb = Q.quantize(x)
    c = Q.unpack(codes)
    assert c.max() <= 15
    xh = Q.dequantize(codes, sb)
    g = x.reshape(200, 2, 64).astype(np.float64)
    s = sb[..., 0].astype(np.float64)
    b = sb[..., 1].astype(np.float64)
    s_true = (g.max(-1) - g.min(-1)) / 15
    bound = 0.5 * s + np.abs(b - g.min(-1)) + 15 * np.abs(s - s_true) + 1e-6
    err = np.abs(xh.reshape(200, 2, 64) - g).max(-1)
    assert (err <= bound).all()
    assert (err <= 0.5 * s + 0.01).all()


def test_q4_dequant_exact():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 64)).astype(np.float32)
    codes, sb = Q.quantize(x)
    xh = Q.dequantize(codes, sb)
    c = Q.unpack(codes)
    for r in range(3):
        for i in (0, 17, 63):
            s = Fraction(float(sb[r, 0, 0]))
            b = Fraction(float(sb[r, 0, 1]))
            assert Fraction(xh[r, i]) == s * int(c[r, i]) + b
