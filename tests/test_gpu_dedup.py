"""GPU fingerprint + dedup vs the oracle: bit-exact fingerprints, block
tables, refcounts, physical-block counts, owner sequences and the reference
lists of every physical block; pool statistics on the 7B workload."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from shared_paged_kv_gb300 import kvs as K
from shared_paged_kv_gb300 import workloads as W
from oracle import accounting as OA, fingerprint as OF
import harness as H


def check(w, flags=0, segments=True, tier=None, capacity=None):
    pool = H.bf16_pool(w, capacity=capacity, with_diff=False) if capacity is None else \
        K.kvs_pool_create(1, w.n_kv_heads, w.head_dim, w.block_tokens, K.KVS_DTYPE_BF16, capacity, w.n_seq,
                          [torch.zeros(16, dtype=torch.int16, device=H.DEV)],
                          [torch.zeros(16, dtype=torch.int16, device=H.DEV)])
    got = H.gpu_dedup(pool, w, flags=flags, segments=segments, tier=tier)
    t = w.tier if tier is None else tier
    so, sb = (w.seg_start_off, w.seg_start_blocks) if segments else (None, None)
    ref = OF.dedup(w.tokens, w.seq_off, t, w.block_tokens, w.max_blocks, so, sb)
    assert got["n_phys"] == ref["n_phys"]
    np.testing.assert_array_equal(got["block_table"], ref["block_table"])
    np.testing.assert_array_equal(got["refcount"], ref["refcount"])
    np.testing.assert_array_equal(got["fp"], ref["fp"])
    assert (got["refcount_full"][ref["n_phys"]:] == 0).all()
    n = ref["n_phys"]
    np.testing.assert_array_equal(got["owner"][:n], ref["owner"])
    assert (got["owner"][n:] == -1).all()
    r_off, r_seq = OF.references(ref["block_table"], n)
    np.testing.assert_array_equal(got["ref_off"][:n + 1], r_off)
    assert (got["ref_off"][n + 1:] == r_off[-1]).all()
    np.testing.assert_array_equal(got["ref_seq"][:r_off[-1]], r_seq)
    assert K.kvs_pool_check(pool) == 0
    got["pool"] = pool
    return got, ref


def test_tiny():
    got, ref = check(W.make_tiny())
    assert ref["n_phys"] == 16 + sum(-(-(l - 256) // 16) for l in W.make_tiny().seq_len)


def test_gqa_small_ragged():
    check(W.make_gqa_fanout(n_seq=7, prefix_tokens=200, priv_lo=1, priv_hi=90, hq=4, hkv=2, d=64))


def test_segments_allgather_small():
    w = W.make_allgather(n_seq=5, n_segs=7, priv_blocks_lo=2, priv_blocks_hi=6, hq=4, hkv=2, d=64, n_layers=1)
    got, ref = check(w)
    # every master segment is stored once: 7 segments x 8 blocks shared by 5 agents
    assert (ref["refcount"] == 5).sum() == 7 * 8
    check(w, segments=False)   # prefix hashing of the same tokens shares nothing


def test_reference_lists_take_both_buffers():
    # ref_off without ref_seq (or the reverse) is an argument error
    w = W.make_tiny()
    pool = H.bf16_pool(w, with_diff=False)
    cap = pool.desc.capacity_blocks
    tokens = torch.from_numpy(w.tokens.view(np.int32)).to(H.DEV)
    fp = torch.zeros(w.n_seq, w.max_blocks, dtype=torch.int64, device=H.DEV)
    table = torch.zeros(w.n_seq, w.max_blocks, dtype=torch.int32, device=H.DEV)
    refc = torch.zeros(cap, dtype=torch.int32, device=H.DEV)
    nphys = torch.zeros(1, dtype=torch.int32, device=H.DEV)
    ws = H.workspace(K.kvs_workspace_size(pool, K.KVS_OP_DEDUP, w.n_seq, w.max_blocks))
    ref_off = torch.zeros(cap + 1, dtype=torch.int64, device=H.DEV)
    ref_seq = torch.zeros(w.n_seq * w.max_blocks, dtype=torch.int32, device=H.DEV)
    for kw in (dict(ref_off=ref_off), dict(ref_seq=ref_seq)):
        with pytest.raises(K.KvsError) as e:
            K.kvs_fingerprint_dedup(pool, tokens, H.i64(w.seq_off), w.n_seq, None, None, None, fp, table,
                                    w.max_blocks, refc, nphys, ws, **kw)
        assert e.value.status == K.KVS_ERR_INVALID_ARG


def test_rerun_is_bit_identical():
    # the dedup has a fixed result for given inputs (no order from atomics
    # reaches the outputs): a second call on the same inputs gives the same bits
    w = W.make_allgather(n_seq=6, n_segs=9, priv_blocks_lo=1, priv_blocks_hi=7, hq=4, hkv=2, d=64, n_layers=1)
    pool = H.bf16_pool(w, with_diff=False)
    tier = np.array([0, 1, 0, W.PRIVATE_TIER, 1, 0], dtype=np.uint32)
    first = H.gpu_dedup(pool, w, tier=tier)
    second = H.gpu_dedup(pool, w, tier=tier)
    for k in ("fp", "block_table", "refcount_full", "owner", "ref_off", "ref_seq"):
        np.testing.assert_array_equal(first[k], second[k], err_msg=k)
    assert first["n_phys"] == second["n_phys"]


def test_tiers_and_private():
    w = W.make_gqa_fanout(n_seq=6, prefix_tokens=96, priv_lo=0, priv_hi=40, hq=4, hkv=2, d=64)
    tier = np.array([0, 1, 0, W.PRIVATE_TIER, 1, 0], dtype=np.uint32)
    check(w, tier=tier)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_collision_path_is_exact(seed):
    # 6-bit table keys force many hash collisions; the token compare and the
    # exact fallback must still give the oracle's result.
    rng = np.random.default_rng(seed)
    w = W.make_gqa_fanout(seed=seed, n_seq=6, prefix_tokens=int(rng.integers(16, 120)), priv_lo=0, priv_hi=70,
                          hq=4, hkv=2, d=64)
    check(w, flags=K.KVS_DEDUP_TEST_WEAK_KEYS)
    w2 = W.make_allgather(seed=seed, n_seq=4, n_segs=5, priv_blocks_lo=1, priv_blocks_hi=4, hq=4, hkv=2, d=64,
                          n_layers=1)
    check(w2, flags=K.KVS_DEDUP_TEST_WEAK_KEYS)


def test_empty_and_short_sequences():
    seqs = [np.arange(0, dtype=np.uint32), np.arange(5, dtype=np.uint32), np.arange(16, dtype=np.uint32),
            np.arange(40, dtype=np.uint32), np.arange(0, dtype=np.uint32)]
    off = np.concatenate([[0], np.cumsum([len(s) for s in seqs])]).astype(np.int64)
    w = W.Workload("edge", len(seqs), 2, 1, 64, 16, 1, 1e4, np.concatenate(seqs).astype(np.uint32), off,
                   np.zeros(len(seqs), np.uint32), 3, 8)
    got, ref = check(w)
    assert (got["block_table"][0] == -1).all() and (got["block_table"][4] == -1).all()


def test_pool_filled_exactly():
    # a pool whose capacity is exactly the number of physical blocks: no error
    w = W.make_gqa_fanout(n_seq=5, prefix_tokens=96, priv_lo=10, priv_hi=70, hq=4, hkv=2, d=64)
    n = OF.dedup(w.tokens, w.seq_off, w.tier, w.block_tokens, w.max_blocks)["n_phys"]
    got, ref = check(w, capacity=n)
    assert got["n_phys"] == n and (got["owner"] >= 0).all()


def test_too_long_sequence_is_flagged():
    w = W.make_gqa_fanout(n_seq=3, prefix_tokens=64, priv_lo=10, priv_hi=20, hq=4, hkv=2, d=64)
    w.max_blocks -= 1      # the longest sequence no longer fits its table row
    pool = H.bf16_pool(w, with_diff=False)
    H.gpu_dedup(pool, w)
    assert K.kvs_pool_check(pool) & K.KVS_DEVERR_SEQ_LEN


def test_capacity_overflow_is_flagged():
    w = W.make_gqa_fanout(n_seq=4, prefix_tokens=64, priv_lo=40, priv_hi=60, hq=4, hkv=2, d=64)
    pool = K.kvs_pool_create(1, 2, 64, 16, K.KVS_DTYPE_BF16, 5, 4,
                             [torch.zeros(5 * 2 * 16 * 64, dtype=torch.int16, device=H.DEV)],
                             [torch.zeros(5 * 2 * 16 * 64, dtype=torch.int16, device=H.DEV)])
    H.gpu_dedup(pool, w)
    assert K.kvs_pool_check(pool) & K.KVS_DEVERR_CAPACITY


@pytest.mark.parametrize("name", ["mha7b", "gqa_fanout", "allgather"])
def test_full_size(name):
    w = {"mha7b": W.make_mha7b, "gqa_fanout": W.make_gqa_fanout, "allgather": W.make_allgather}[name]()
    got, ref = check(w, capacity=w.capacity_blocks)
    if name == "mha7b":
        assert ref["n_phys"] == 614 + 8 * 410
        # pool statistics: INMS walkthrough §1.2 independent (n*L) against
        # shared ((1-p)*n + p)*L footprint, at block granularity (L = 1024
        # blocks, p = 614/1024); this pool holds one layer of 32 KV heads x 128
        st = K.kvs_pool_stats(got["pool"], got["refc_dev"], got["nphys_dev"])
        per_block = 2 * w.n_kv_heads * 16 * w.head_dim * 2
        assert st["unique_blocks"] == 3894 and st["shared_blocks"] == 614 and st["total_refs"] == 8 * 1024
        assert st["pool_bytes"] == round(OA.shared_bytes(8, 1024, per_block, 614 / 1024))
        assert st["dense_bytes"] == OA.independent_bytes(8, 1024, per_block)
