"""Pins of the mirror-construction oracle (TokenDance summary sections 2-3):
a hand example, the restore property through the attention oracle's own
materialisation (apply the diff, then restore RoPE), and the dirty-block id
order by an independent count."""
import numpy as np

from oracle import attention as OA, mirror as OM, rope as OR


def _pool(rng, n_blocks, hkv, d, B=16):
    k = rng.standard_normal((n_blocks, hkv, B, d))
    v = rng.standard_normal((n_blocks, hkv, B, d))
    return k, v


def test_hand_example():
    rng = np.random.default_rng(0)
    k, v = _pool(rng, 4, 1, 4)
    table = np.array([[2, 0, 3]], dtype=np.int32)
    idx = np.array([3, 20, 21])
    off = np.array([0, 3])
    kn = rng.standard_normal((3, 1, 4))
    vn = rng.standard_normal((3, 1, 4))
    r = OM.mirror_build(table, idx, off, kn, vn, k, v, 16)
    assert r["n_diff"] == 2
    assert r["diff_table"].tolist() == [[0, 1, -1]]
    # position 3 lives in logical block 0 = physical 2, row 3
    assert np.allclose(r["dk"][0, :, 3, :], kn[0] - k[2, :, 3, :], rtol=0, atol=0)
    assert np.allclose(r["dv"][0, :, 3, :], vn[0] - v[2, :, 3, :], rtol=0, atol=0)
    # positions 20, 21 live in logical block 1 = physical 0, rows 4 and 5
    assert np.array_equal(r["dk"][1, :, 4, :], kn[1] - k[0, :, 4, :])
    assert np.array_equal(r["dk"][1, :, 5, :], kn[2] - k[0, :, 5, :])
    # every other row of a dirty block is zero
    mask = np.ones((2, 16), bool)
    mask[0, 3] = mask[1, 4] = mask[1, 5] = False
    assert not r["dk"][:, :, :, :].transpose(0, 2, 1, 3)[mask].any()
    assert not r["dv"][:, :, :, :].transpose(0, 2, 1, 3)[mask].any()


def _random_family(seed):
    """Agents sharing master blocks at shifted positions, some refreshed rows."""
    rng = np.random.default_rng(seed)
    n_seq, hkv, d, B, max_blocks = 3, 2, 8, 16, 6
    k, v = _pool(rng, 10, hkv, d, B)
    table = rng.integers(0, 10, size=(n_seq, max_blocks)).astype(np.int32)
    seq_len = np.array([96, 70, 33], dtype=np.int32)
    # one rotated segment per agent over blocks 1..2 (shift differs per agent)
    rope_off = np.array([0, 1, 2, 3], dtype=np.int32)
    rope_segs = np.array([[1, 2, 37, 0], [1, 2, -120, 0], [0, 1, 5, 0]], dtype=np.int32)
    idx, off = [], [0]
    for a in range(n_seq):
        pos = np.sort(rng.choice(seq_len[a], size=int(rng.integers(0, 12)), replace=False))
        idx.extend(pos.tolist())
        off.append(len(idx))
    idx = np.array(idx, dtype=np.int64)
    off = np.array(off, dtype=np.int64)
    kn = rng.standard_normal((len(idx), hkv, d))
    vn = rng.standard_normal((len(idx), hkv, d))
    return dict(k=k, v=v, table=table, seq_len=seq_len, rope_off=rope_off, rope_segs=rope_segs,
                idx=idx, off=off, kn=kn, vn=vn, B=B)


def test_restore_gives_the_refreshed_cache():
    """Applying the diffs and then restoring RoPE (the attention oracle's
    materialisation) yields the refreshed values at refreshed positions and
    the plain reused values elsewhere."""
    theta = 1e4
    for seed in range(6):
        f = _random_family(seed)
        r = OM.mirror_build(f["table"], f["idx"], f["off"], f["kn"], f["vn"], f["k"], f["v"], f["B"],
                            f["rope_off"], f["rope_segs"], theta)
        for a in range(f["table"].shape[0]):
            L = int(f["seq_len"][a])
            got_k, got_v = OA.materialise(a, L, f["k"], f["v"], f["table"], f["B"], r["diff_table"],
                                          r["dk"], r["dv"], f["rope_off"], f["rope_segs"], theta)
            plain_k, plain_v = OA.materialise(a, L, f["k"], f["v"], f["table"], f["B"], None, None, None,
                                              f["rope_off"], f["rope_segs"], theta)
            refreshed = {int(t): rr for rr, t in enumerate(f["idx"][f["off"][a]:f["off"][a + 1]], int(f["off"][a]))}
            for t in range(L):
                if t in refreshed:
                    assert np.allclose(got_k[t], f["kn"][refreshed[t]], rtol=0, atol=1e-12)
                    assert np.allclose(got_v[t], f["vn"][refreshed[t]], rtol=0, atol=1e-12)
                else:
                    assert np.allclose(got_k[t], plain_k[t], rtol=0, atol=1e-12)
                    assert np.allclose(got_v[t], plain_v[t], rtol=0, atol=1e-12)


def test_rotation_direction_matters():
    """Without taking K back to the master's frame the restore would not
    reproduce the refreshed K: the -delta step is pinned by the restore."""
    f = _random_family(1)
    theta = 1e4
    r = OM.mirror_build(f["table"], f["idx"], f["off"], f["kn"], f["vn"], f["k"], f["v"], f["B"],
                        f["rope_off"], f["rope_segs"], theta)
    a = 0
    got_k, _ = OA.materialise(a, int(f["seq_len"][a]), f["k"], f["v"], f["table"], f["B"], r["diff_table"],
                              r["dk"], r["dv"], f["rope_off"], f["rope_segs"], theta)
    # a position inside the rotated segment (blocks 1..2 of agent 0)
    rows = [rr for rr in range(f["off"][0], f["off"][1]) if 16 <= f["idx"][rr] < 48]
    assert rows
    rr = rows[0]
    assert np.allclose(got_k[f["idx"][rr]], f["kn"][rr], atol=1e-12)
    wrong = OR.rotate(f["kn"][rr], 2 * 37, theta)   # what the other direction would restore
    assert not np.allclose(got_k[f["idx"][rr]], wrong, atol=1e-6)


def test_dirty_ids_agent_major_then_block_order():
    for seed in range(6):
        f = _random_family(seed)
        r = OM.mirror_build(f["table"], f["idx"], f["off"], f["kn"], f["vn"], f["k"], f["v"], f["B"])
        n_seq, max_blocks = f["table"].shape
        keys = []
        for a in range(n_seq):
            keys.extend(a * max_blocks + t // f["B"] for t in f["idx"][f["off"][a]:f["off"][a + 1]])
        uniq = np.unique(np.array(keys, dtype=np.int64))
        expect = np.full(n_seq * max_blocks, -1, dtype=np.int32)
        expect[uniq] = np.arange(len(uniq))
        assert r["n_diff"] == len(uniq)
        assert np.array_equal(r["diff_table"].reshape(-1), expect)


def test_agent_without_refresh_has_no_diff():
    f = _random_family(2)
    off = f["off"].copy()
    # drop agent 1's positions
    keep = np.r_[np.arange(off[0], off[1]), np.arange(off[2], off[3])]
    idx, kn, vn = f["idx"][keep], f["kn"][keep], f["vn"][keep]
    n1 = off[2] - off[1]
    off2 = np.array([off[0], off[1], off[1], off[3] - n1])
    r = OM.mirror_build(f["table"], idx, off2, kn, vn, f["k"], f["v"], f["B"])
    assert (r["diff_table"][1] == -1).all()
