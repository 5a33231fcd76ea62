"""Pins of oracle.attention: closed forms, special cases and the layout
invariants the pages state (shared vs private storage, mirror = master +
diff, collective rotation = per-agent rotation)."""
import numpy as np
import pytest

from oracle import attention as AT, fingerprint as F, rope as R


def pool(rng, cap, hkv, B, d):
    return rng.standard_normal((cap, hkv, B, d)), rng.standard_normal((cap, hkv, B, d))


def test_uniform_values_give_that_value():
    rng = np.random.default_rng(0)
    k, v = pool(rng, 3, 1, 4, 8)
    v[:] = np.arange(8.0)
    bt = np.array([[0, 1, 2]], np.int32)
    out = AT.decode_attention(rng.standard_normal((1, 1, 8)), k, v, bt, [11], 4, 0.3)
    np.testing.assert_allclose(out[0, 0], np.arange(8.0), atol=1e-12)


def test_single_token_and_empty_context():
    rng = np.random.default_rng(1)
    k, v = pool(rng, 2, 1, 4, 8)
    bt = np.array([[1, -1], [0, -1]], np.int32)
    out = AT.decode_attention(rng.standard_normal((2, 1, 8)), k, v, bt, [1, 0], 4, 0.3)
    np.testing.assert_allclose(out[0, 0], v[1, 0, 0], atol=1e-15)
    assert np.all(out[1] == 0)


def test_zero_query_is_mean_and_two_token_closed_form():
    rng = np.random.default_rng(2)
    k, v = pool(rng, 1, 1, 4, 8)
    bt = np.array([[0]], np.int32)
    out = AT.decode_attention(np.zeros((1, 1, 8)), k, v, bt, [3], 4, 0.5)
    np.testing.assert_allclose(out[0, 0], v[0, 0, :3].mean(0), atol=1e-12)
    q = rng.standard_normal((1, 1, 8))
    out = AT.decode_attention(q, k, v, bt, [2], 4, 0.5)
    s0, s1 = 0.5 * q[0, 0] @ k[0, 0, 0], 0.5 * q[0, 0] @ k[0, 0, 1]
    w0 = 1 / (1 + np.exp(s1 - s0))
    np.testing.assert_allclose(out[0, 0], w0 * v[0, 0, 0] + (1 - w0) * v[0, 0, 1], atol=1e-12)


def test_gqa_head_mapping():
    rng = np.random.default_rng(3)
    k, v = pool(rng, 2, 2, 4, 8)
    v[:, 1] = 7.0                     # KV head 1 holds a constant value
    bt = np.array([[0, 1]], np.int32)
    out = AT.decode_attention(rng.standard_normal((1, 4, 8)), k, v, bt, [8], 4, 0.3)
    np.testing.assert_allclose(out[0, 2:], 7.0, atol=1e-12)   # q heads 2,3 -> kv 1
    assert np.abs(out[0, :2] - 7.0).max() > 1


def test_shared_layout_equals_private_layout():
    # The same contexts, stored once with refcounted shared blocks or fully
    # private per agent, give identical outputs.
    rng = np.random.default_rng(4)
    B, d = 4, 16
    prefix = rng.integers(0, 100, size=12, dtype=np.uint32)
    seqs = [np.concatenate([prefix, rng.integers(0, 100, size=n, dtype=np.uint32)]) for n in (5, 9, 2)]
    off = np.concatenate([[0], np.cumsum([len(s) for s in seqs])]).astype(np.int64)
    mb = max(-(-len(s) // B) for s in seqs)
    sh = F.dedup(np.concatenate(seqs), off, None, B, mb)
    # private layout: every (agent, block) gets its own copy of the same values
    kp, vp = pool(rng, sh["n_phys"], 2, B, d)
    priv_table = np.full_like(sh["block_table"], -1)
    rows_k, rows_v, nxt = [], [], 0
    for a in range(3):
        for b in range(mb):
            p = sh["block_table"][a, b]
            if p >= 0:
                rows_k.append(kp[p]); rows_v.append(vp[p]); priv_table[a, b] = nxt; nxt += 1
    kq, vq = np.stack(rows_k), np.stack(rows_v)
    q = rng.standard_normal((3, 4, d))
    lens = np.diff(off)
    o1 = AT.decode_attention(q, kp, vp, sh["block_table"], lens, B, 0.25)
    o2 = AT.decode_attention(q, kq, vq, priv_table, lens, B, 0.25)
    assert np.array_equal(o1, o2)
    assert sh["n_phys"] < nxt


def test_mirror_overlay_equals_dense_mirror():
    rng = np.random.default_rng(5)
    B, d = 4, 8
    k, v = pool(rng, 4, 1, B, d)
    dk, dv = 0.1 * rng.standard_normal((2, 1, B, d)), 0.1 * rng.standard_normal((2, 1, B, d))
    bt = np.array([[0, 1, 2, 3], [0, 1, 2, 3]], np.int32)
    dt = np.array([[-1, 0, -1, -1], [-1, -1, -1, 1]], np.int32)
    q = rng.standard_normal((2, 1, d))
    o1 = AT.decode_attention(q, k, v, bt, [16, 15], B, 0.4, diff_table=dt, dk_pool=dk, dv_pool=dv)
    # dense mirrors: copy the master and add the diffs into private blocks
    k2 = np.concatenate([k, k[1:2] + dk[0:1], k[3:4] + dk[1:2]])
    v2 = np.concatenate([v, v[1:2] + dv[0:1], v[3:4] + dv[1:2]])
    bt2 = np.array([[0, 4, 2, 3], [0, 1, 2, 5]], np.int32)
    o2 = AT.decode_attention(q, k2, v2, bt2, [16, 15], B, 0.4)
    np.testing.assert_allclose(o1, o2, atol=1e-13)


def test_sub_block_diffs_equal_dense_mirror():
    # Q4 pools keep mirror diffs per 16-token sub-block of their 256-token
    # blocks: a diff block smaller than the pool block.  Pool blocks of 8
    # tokens, diff blocks of 2: the overlay must equal a dense mirror built by
    # copying the master and adding each diff row by hand.
    rng = np.random.default_rng(9)
    B, DB, d = 8, 2, 8
    k, v = pool(rng, 3, 2, B, d)
    dk, dv = 0.1 * rng.standard_normal((3, 2, DB, d)), 0.1 * rng.standard_normal((3, 2, DB, d))
    bt = np.array([[0, 1, 2], [0, 1, -1]], np.int32)
    dt = np.full((2, 3 * B // DB), -1, np.int32)
    dt[0, 1], dt[0, 10], dt[1, 7] = 0, 2, 1      # tokens 2-3 and 20-21 of agent 0, 14-15 of agent 1
    q = rng.standard_normal((2, 4, d))
    o1 = AT.decode_attention(q, k, v, bt, [23, 16], B, 0.3, diff_table=dt, dk_pool=dk, dv_pool=dv,
                             diff_block_tokens=DB)
    k2 = np.concatenate([k, k[0:2], k[2:3]])      # agent 0's mirror blocks 3, 4; agent 1's block 5
    v2 = np.concatenate([v, v[0:2], v[2:3]])
    for (blk, row, src) in [(3, 2, 0), (3, 3, 0), (5, 4, 2), (5, 5, 2)]:
        r = row - 2 if src == 0 else row - 4
        k2[blk, :, row] += dk[src, :, r]
        v2[blk, :, row] += dv[src, :, r]
    k3 = np.concatenate([k2, k[0:2]])              # agent 1's mirror of blocks 0 and 1 -> 6, 7
    v3 = np.concatenate([v2, v[0:2]])
    k3[7, :, 6:8] += dk[1]
    v3[7, :, 6:8] += dv[1]
    bt2 = np.array([[3, 4, 5], [6, 7, -1]], np.int32)
    o2 = AT.decode_attention(q, k3, v3, bt2, [23, 16], B, 0.3)
    np.testing.assert_allclose(o1, o2, atol=1e-13)


def test_segment_rotation_collective_equals_per_agent():
    # Collective path: one shared master segment rotated per agent inside the
    # read.  Per-agent path: each agent's materialised copy rotated from the
    # master position to its own (complex-number restatement of the shift).
    rng = np.random.default_rng(6)
    B, d, theta = 4, 16, 1e6
    k, v = pool(rng, 3, 1, B, d)     # blocks 0: private, 1-2: master segment
    bt = np.array([[0, 1, 2], [0, 1, 2]], np.int32)
    segs = np.array([[1, 2, 300, 0], [1, 2, -50, 0]], np.int32)
    r_off = np.array([0, 1, 2], np.int32)
    q = rng.standard_normal((2, 1, d))
    o1 = AT.decode_attention(q, k, v, bt, [12, 12], B, 0.3, rope_off=r_off, rope_segs=segs, theta=theta)
    h = d // 2
    w = theta ** (-2.0 * np.arange(h) / d)
    for a, delta in ((0, 300), (1, -50)):
        K = np.concatenate([k[0, 0], k[1, 0], k[2, 0]]).copy()
        z = (K[4:, :h] + 1j * K[4:, h:]) * np.exp(1j * delta * w)
        K[4:] = np.concatenate([z.real, z.imag], axis=-1)
        V = np.concatenate([v[0, 0], v[1, 0], v[2, 0]])
        s = 0.3 * K @ q[a, 0]
        p = np.exp(s - s.max()); p /= p.sum()
        np.testing.assert_allclose(o1[a, 0], p @ V, atol=1e-12)
        # the same with the query rotated the other way against the stored K
        Ks = np.concatenate([k[0, 0], k[1, 0], k[2, 0]])
        s2 = 0.3 * np.concatenate([Ks[:4] @ q[a, 0], Ks[4:] @ R.rotate(q[a, 0], -delta, theta)])
        p2 = np.exp(s2 - s2.max()); p2 /= p2.sum()
        np.testing.assert_allclose(o1[a, 0], p2 @ V, atol=1e-12)
