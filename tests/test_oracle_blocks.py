"""Pins of the block-lifetime oracle (INMS walkthrough §2.2 write_to_block,
§3.3 sequence destroy, §5.3 leaks): a hand example of the copy-on-write rule,
the reference-count invariant and leak freedom under random operation
sequences, and the isolation of the other referrers."""
import numpy as np

from oracle import blocks as OB


def test_hand_example_copy_on_write():
    # three sequences share physical block 0; capacity 5 -> free stack top is 1
    table = np.array([[0], [0], [0]], np.int32)
    seq_len = np.array([16, 16, 16])
    ref = np.array([3, 0, 0, 0, 0])
    slab = np.arange(5 * 4).reshape(5, 4)
    m = OB.BlockManager(table, seq_len, ref, 16, [slab])
    assert m.free == [4, 3, 2, 1]
    m.write_batch([0, 1, 2], [0, 0, 0])
    # the first two writers copy (blocks 1 and 2); the last one is alone and
    # writes in place
    assert m.table.tolist() == [[1], [2], [0]]
    assert m.ref.tolist() == [1, 1, 1, 0, 0]
    assert m.free == [4, 3]
    assert np.array_equal(m.slabs[0][1], slab[0]) and np.array_equal(m.slabs[0][2], slab[0])
    # a second write by sequence 0 is now in place
    m.write_batch([0], [0])
    assert m.table.tolist() == [[1], [2], [0]] and m.ref.tolist() == [1, 1, 1, 0, 0]
    # releasing 1 and 2 frees blocks 2 and 0, pushed so that 0 is on top
    m.release([1, 2])
    assert m.free == [4, 3, 2, 0]
    assert m.ref.tolist() == [0, 1, 0, 0, 0]
    assert (m.table[1:] == -1).all()
    assert not m.errors


def _random_manager(rng, n_seq=6, cap=40, B=16):
    """Sequences over a shared prefix of 3 blocks plus private blocks."""
    seq_len = rng.integers(1, 6 * B, size=n_seq)
    max_blocks = int(-(-seq_len.max() // B))
    table = np.full((n_seq, max_blocks), -1, np.int32)
    nxt = 3
    ref = np.zeros(cap, np.int64)
    for a in range(n_seq):
        for b in range(int(-(-seq_len[a] // B))):
            if b < 3 and (b + 1) * B <= seq_len[a]:
                p = b
            else:
                p = nxt
                nxt += 1
            table[a, b] = p
            ref[p] += 1
    slab = rng.standard_normal((cap, 3))
    return OB.BlockManager(table, seq_len, ref, B, [slab])


def _check_invariants(m):
    assert np.array_equal(m.ref, m.referenced_counts())
    referenced = {p for p in range(len(m.ref)) if m.ref[p] > 0}
    free = set(m.free)
    assert len(free) == len(m.free), "a block is on the free stack twice"
    assert not (free & referenced)
    assert free | referenced == set(range(len(m.ref))), "a block leaked"


def test_invariants_under_random_operations_and_no_leak():
    for seed in range(20):
        rng = np.random.default_rng(seed)
        m = _random_manager(rng)
        _check_invariants(m)
        alive = list(range(m.table.shape[0]))
        for _ in range(8):
            if rng.random() < 0.7 and alive:
                k = int(rng.integers(1, 5))
                seqs = rng.choice(alive, size=k)
                blocks = [int(rng.integers(0, m.n_blocks(a))) for a in seqs]
                m.write_batch(seqs, blocks)
            elif alive:
                out = [alive.pop(int(rng.integers(0, len(alive))))]
                m.release(out)
            _check_invariants(m)
        m.release(alive)
        _check_invariants(m)
        assert (m.ref == 0).all() and len(m.free) == len(m.ref)
        assert not m.errors


def test_copy_leaves_other_referrers_untouched():
    rng = np.random.default_rng(3)
    m = _random_manager(rng)
    before_tab = m.table.copy()
    view = {a: [m.slabs[0][m.table[a, b]].copy() for b in range(m.n_blocks(a))] for a in range(m.table.shape[0])}
    m.write_batch([0], [0])
    for a in range(1, m.table.shape[0]):
        assert np.array_equal(m.table[a], before_tab[a])
        for b in range(m.n_blocks(a)):
            assert np.array_equal(m.slabs[0][m.table[a, b]], view[a][b])
    # the writer sees the same contents in its private copy
    assert np.array_equal(m.slabs[0][m.table[0, 0]], view[0][0])


def test_private_block_written_in_place():
    table = np.array([[0, 1]], np.int32)
    m = OB.BlockManager(table, np.array([32]), np.array([1, 1, 0]), 16)
    m.write_batch([0, 0], [0, 1])
    assert m.table.tolist() == [[0, 1]] and m.free == [2]


def test_double_release_is_a_no_op_and_overrelease_is_an_error():
    m = OB.BlockManager(np.array([[0]], np.int32), np.array([16]), np.array([1, 0]), 16)
    m.release([0])
    m.release([0])
    assert not m.errors and m.free == [1, 0]
    bad = OB.BlockManager(np.array([[0], [0]], np.int32), np.array([16, 16]), np.array([1, 0]), 16)
    bad.release([0, 1])
    assert "refcount" in bad.errors


def test_copy_without_free_blocks_is_an_error():
    m = OB.BlockManager(np.array([[0], [0]], np.int32), np.array([16, 16]), np.array([2]), 16)
    m.write_batch([0], [0])
    assert "capacity" in m.errors and m.table.tolist() == [[0], [0]]


def test_write_to_an_unmapped_block_is_an_error():
    m = OB.BlockManager(np.array([[0, -1]], np.int32), np.array([16]), np.array([1, 0]), 16)
    m.write_batch([0], [1])
    assert "block_id" in m.errors and m.table.tolist() == [[0, -1]]
