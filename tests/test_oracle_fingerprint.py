"""Pins of oracle.fingerprint: CalcHash constants and structure, and the
dedup rule checked against a pairwise brute force on tiny inputs."""
import numpy as np
import pytest

from oracle import fingerprint as F
from golden_io import rows

MASK = (1 << 64) - 1


def test_constants_as_printed():
    g = {r[0]: int(r[1]) for r in rows("calchash_constants.txt")}
    assert F.FNV_OFFSET == g["offset_basis"]
    assert F.FNV_PRIME == g["prime"]


@pytest.mark.parametrize("seed", range(5))
def test_hash_unwinds_with_inverse_prime(seed):
    # The hash is a chain of (xor id, multiply by an odd prime mod 2^64)
    # steps; multiplying by the modular inverse of the prime and xoring the
    # same ids in reverse order must land exactly on the offset basis.  A
    # wrong constant, order of xor/multiply, word width or tag step fails.
    rng = np.random.default_rng(seed)
    toks = rng.integers(0, 2 ** 32, size=int(rng.integers(0, 40)), dtype=np.uint64)
    tag = int(rng.integers(0, 2 ** 32))
    h = F.calc_hash(toks, tag)
    inv = pow(F.FNV_PRIME, -1, 1 << 64)
    h = (h * inv) & MASK
    h ^= tag
    for t in toks[::-1]:
        h = (h * inv) & MASK
        h ^= int(t)
    assert h == F.FNV_OFFSET


def test_tag_and_token_sensitivity():
    toks = list(range(16))
    assert F.calc_hash(toks, 0) != F.calc_hash(toks, 1)
    assert F.calc_hash(toks, 0) != F.calc_hash(toks[::-1], 0)
    # ids are whole 32-bit words: values above 2^32 wrap as in the C cast
    assert F.calc_hash([5], 0) == F.calc_hash([5 + (1 << 32)], 0)


def test_find_match_length_stops_at_first_miss():
    C = 4
    a = list(range(100, 120))
    pool = {F.calc_hash(a[i:i + C], 0) for i in range(0, 20, C)}
    b = a[:12] + [7, 7, 7, 7] + a[16:]
    assert F.find_match_length(a, C, pool) == 20
    assert F.find_match_length(b, C, pool) == 12        # stops at the miss
    assert F.find_match_length(a[:10], C, pool) == 8    # trailing partial ignored


# ---------------------------------------------------------------------------
def brute_dedup(tokens, seq_off, tier, B, max_blocks, starts=None):
    """Pairwise restatement: slot (s,b) maps to the earliest slot (in scan
    order) it is equivalent to; ids are numbered by first occurrence."""
    n = len(seq_off) - 1
    slots = []
    for s in range(n):
        L = int(seq_off[s + 1] - seq_off[s])
        for b in range(-(-L // B)):
            slots.append((s, b))

    def info(s, b):
        L = int(seq_off[s + 1] - seq_off[s])
        full = (b + 1) * B <= L
        st = 0
        if starts is not None:
            st = max([0] + [x for x in starts[s] if x <= b])
        return full and int(tier[s]) != F.PRIVATE_TIER, st

    def equiv(s, b, s2, b2):
        sh1, st1 = info(s, b)
        sh2, st2 = info(s2, b2)
        if not (sh1 and sh2) or tier[s] != tier[s2] or b - st1 != b2 - st2:
            return False
        o1, o2 = int(seq_off[s]), int(seq_off[s2])
        for i in range((b - st1 + 1) * B):
            if tokens[o1 + st1 * B + i] != tokens[o2 + st2 * B + i]:
                return False
        return True

    rep = {}
    for i, (s, b) in enumerate(slots):
        rep[(s, b)] = (s, b)
        for j in range(i):
            if equiv(s, b, *slots[j]):
                rep[(s, b)] = slots[j]
                break
    ids = {}
    table = np.full((n, max_blocks), -1, dtype=np.int32)
    for (s, b) in slots:
        r = rep[(s, b)]
        if r == (s, b):
            ids[r] = len(ids)
        table[s, b] = ids[r]
    ref = np.bincount(table[table >= 0], minlength=len(ids)).astype(np.int32)
    return table, ref


def random_structure(seed, n=6, B=4, segments=False):
    rng = np.random.default_rng(seed)
    pieces = [rng.integers(0, 5, size=B * int(rng.integers(1, 4)), dtype=np.uint32) for _ in range(4)]
    seqs, starts = [], []
    for s in range(n):
        parts, st, nb = [], [], 0
        for _ in range(int(rng.integers(1, 5))):
            p = pieces[int(rng.integers(0, len(pieces)))]
            st.append(nb)
            parts.append(p)
            nb += len(p) // B
        tail = rng.integers(0, 5, size=int(rng.integers(0, B + 1)), dtype=np.uint32)
        seqs.append(np.concatenate(parts + [tail]))
        starts.append(st)
    off = np.concatenate([[0], np.cumsum([len(x) for x in seqs])]).astype(np.int64)
    toks = np.concatenate(seqs).astype(np.uint32)
    tier = rng.choice(np.array([0, 0, 1, F.PRIVATE_TIER], dtype=np.uint32), size=n)
    max_blocks = int(max(-(-len(x) // B) for x in seqs))
    return toks, off, tier, B, max_blocks, (starts if segments else None)


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("segments", [False, True])
def test_dedup_matches_bruteforce(seed, segments):
    toks, off, tier, B, mb, starts = random_structure(seed, segments=segments)
    s_off = s_flat = None
    if starts is not None:
        s_off = np.concatenate([[0], np.cumsum([len(x) for x in starts])]).astype(np.int64)
        s_flat = np.concatenate([np.asarray(x) for x in starts]).astype(np.int32)
    r = F.dedup(toks, off, tier, B, mb, s_off, s_flat)
    t2, ref2 = brute_dedup(toks, off, tier, B, mb, starts)
    np.testing.assert_array_equal(r["block_table"], t2)
    np.testing.assert_array_equal(r["refcount"], ref2)
    assert r["n_phys"] == len(ref2)
    assert r["refcount"].sum() == (r["block_table"] >= 0).sum()
    # owner = sequence of each id's first slot in scan order; reference CSR =
    # the slots holding each id, read off the flattened (sequence-major) table
    flat = t2.ravel()
    ref_off, ref_seq = F.references(r["block_table"], r["n_phys"])
    for p in range(r["n_phys"]):
        where = np.flatnonzero(flat == p)
        assert r["owner"][p] == where[0] // mb
        np.testing.assert_array_equal(ref_seq[ref_off[p]:ref_off[p + 1]], where // mb)
    np.testing.assert_array_equal(np.diff(ref_off), ref2)
    # fingerprints of full blocks are CalcHash of the block's tokens and tier
    for s in range(len(off) - 1):
        L = int(off[s + 1] - off[s])
        for b in range(L // B):
            assert r["fp"][s, b] == F.calc_hash(toks[off[s] + b * B: off[s] + (b + 1) * B], tier[s])


def test_block_granular_sharing_count():
    # 8 agents, a 10-block common prefix, 7 private blocks each: the shared
    # footprint formula at block granularity gives 10 + 8 x 7 physical blocks.
    rng = np.random.default_rng(1)
    B = 16
    prefix = rng.integers(0, 32000, size=10 * B, dtype=np.uint32)
    seqs = [np.concatenate([prefix, rng.integers(0, 32000, size=7 * B, dtype=np.uint32)]) for _ in range(8)]
    off = np.concatenate([[0], np.cumsum([len(x) for x in seqs])]).astype(np.int64)
    r = F.dedup(np.concatenate(seqs), off, None, B, 17)
    assert r["n_phys"] == 10 + 8 * 7
    assert list(r["refcount"][:10]) == [8] * 10
    assert (r["refcount"][10:] == 1).all()


def test_tier_isolation_and_private_tier():
    B = 4
    s = np.arange(12, dtype=np.uint32)
    toks = np.concatenate([s, s, s, s])
    off = np.array([0, 12, 24, 36, 48], dtype=np.int64)
    tier = np.array([0, 1, 0, F.PRIVATE_TIER], dtype=np.uint32)
    r = F.dedup(toks, off, tier, B, 3)
    t = r["block_table"]
    assert (t[0] == t[2]).all()               # same tokens, same tier: shared
    assert not np.intersect1d(t[0], t[1]).size  # other tier: never shared
    assert not np.intersect1d(t[3], t[0]).size  # PRIVATE tier never shared
    assert r["n_phys"] == 9


def test_divergence_ends_sharing():
    # Once two sequences diverge, later identical blocks are not shared in
    # prefix mode (sharing runs to the first divergence only).
    B = 2
    a = np.array([1, 2, 3, 4, 5, 6], np.uint32)
    b = np.array([1, 2, 9, 9, 5, 6], np.uint32)
    off = np.array([0, 6, 12], np.int64)
    r = F.dedup(np.concatenate([a, b]), off, None, B, 3)
    t = r["block_table"]
    assert t[0, 0] == t[1, 0] and t[0, 2] != t[1, 2]


def test_references_hand_example():
    # three sequences: a 1-block common prefix, a second block shared by the
    # first two, then private blocks; worked out by hand
    table = np.array([[0, 1, 2], [0, 1, 3], [0, 4, -1]], np.int32)
    off, seq = F.references(table, 5)
    assert off.tolist() == [0, 3, 5, 6, 7, 8]
    assert seq.tolist() == [0, 1, 2, 0, 1, 0, 1, 2]
    # a sequence that holds one block twice (a repeated segment) lists it twice
    off, seq = F.references(np.array([[0, 1, 0], [1, -1, -1]], np.int32), 2)
    assert off.tolist() == [0, 2, 4] and seq.tolist() == [0, 0, 0, 1]
