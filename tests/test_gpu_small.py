"""Small decode-attention calls (n_seq * num_kv_heads * max_blocks <= 2048,
query groups <= 8) run on the single-kernel path with no plan: one launch per
call.  Parity with the fp64 oracle at the attention tolerances, agreement with
the planned token-major path on the same pool, and the bound between the two
paths."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from shared_paged_kv_gb300 import kvs as K
from shared_paged_kv_gb300 import workloads as W
from oracle import attention as OA, fingerprint as OF
import harness as H

f32 = W.bf16_bits_to_f32
SMALL = 2048


def work(w):
    return w.n_seq * w.n_kv_heads * w.max_blocks


def oracle_out(w, pool, table, q_bits, seq_len=None):
    hst = pool.host[0]
    dk = f32(hst["dk"]) if "dk" in hst else None
    dv = f32(hst["dv"]) if "dv" in hst else None
    return OA.decode_attention(f32(q_bits), f32(hst["k"]), f32(hst["v"]), table,
                               w.seq_len if seq_len is None else seq_len, w.block_tokens, w.scale,
                               diff_table=w.diff_table, dk_pool=dk, dv_pool=dv, rope_off=w.rope_off,
                               rope_segs=w.rope_segs, theta=w.theta)


def both_paths(w, seq_len=None, expect_small=True):
    """The library's own choice (counted launches: one for the small path) and
    the planned path on the same pool, each against the oracle."""
    segs = w.seg_start_off is not None
    ref = OF.dedup(w.tokens, w.seq_off, w.tier, w.block_tokens, w.max_blocks,
                   w.seg_start_off if segs else None, w.seg_start_blocks if segs else None)
    pool = H.bf16_pool(w, path="auto")
    q_bits = w.q_layer(0)
    n0 = K.kvs_launch_count()
    auto = H.attn(pool, 0, q_bits, w, ref["block_table"], seq_len=seq_len)
    launches = K.kvs_launch_count() - n0
    assert (launches == 1) == expect_small, f"{launches} launches for work {work(w)}"
    exp = oracle_out(w, pool, ref["block_table"], q_bits, seq_len)
    H.assert_close_attn(auto, exp)
    K.kvs_pool_set_test_flags(pool, K.KVS_TEST_TOKEN_MAJOR)
    planned = H.attn(pool, 0, q_bits, w, ref["block_table"], seq_len=seq_len)
    H.assert_close_attn(planned, exp)
    H.assert_close_attn(auto, planned)
    assert K.kvs_pool_check(pool) == 0
    return auto, exp


def test_tiny_mirror_diffs_one_launch():
    w = W.make_tiny()
    assert work(w) <= SMALL
    both_paths(w)


def test_mha_group1_ragged():
    w = W.make_prefix_shared("mha_small", 3, 4, 4, 128, 1, 24 * 16, [16 * 16 + 5, 16 * 13, 16 * 17 + 11], seed=11)
    assert work(w) <= SMALL
    both_paths(w)


@pytest.mark.parametrize("hq,hkv,d", [(16, 2, 128), (16, 2, 64), (6, 2, 128)])
def test_gqa_groups_ragged(hq, hkv, d):
    w = W.make_gqa_fanout(n_seq=5, prefix_tokens=160, priv_lo=1, priv_hi=300, hq=hq, hkv=hkv, d=d)
    assert work(w) <= SMALL
    both_paths(w)


def test_rotation_and_diffs_group5():
    w = W.make_allgather(n_seq=4, n_segs=6, priv_blocks_lo=3, priv_blocks_hi=9, hq=10, hkv=2, n_layers=1)
    assert work(w) <= SMALL
    both_paths(w)


def test_one_chunk_rotation_and_diffs():
    # block tables of at most 32 blocks: one CTA per (sequence, KV head)
    # writes the output directly; here with rotated segments and mirror diffs
    w = W.make_allgather(n_seq=3, n_segs=2, priv_blocks_lo=1, priv_blocks_hi=4, hq=10, hkv=2, n_layers=1)
    assert w.max_blocks <= 32 and (w.diff_table >= 0).any() and w.rope_off is not None
    both_paths(w)


def test_edge_lengths_small_path():
    # empty context -> zeros; a single token; a block multiple and one past
    w = W.make_gqa_fanout(n_seq=5, prefix_tokens=64, priv_lo=40, priv_hi=90, hq=8, hkv=2, d=128)
    sl = w.seq_len.copy()
    sl[0], sl[1], sl[2], sl[3] = 0, 1, 64, 17
    got, _ = both_paths(w, seq_len=sl)
    assert np.all(got[0] == 0)


def test_bound_between_the_paths():
    # the largest small call and the next size up (one more block per row)
    w = W.make_prefix_shared("bound", 8, 8, 2, 128, 1, 16 * 64, [16 * 64] * 8, seed=5)
    assert work(w) <= SMALL
    both_paths(w, expect_small=True)
    w2 = W.make_prefix_shared("bound2", 8, 8, 2, 128, 1, 16 * 64, [16 * 65] * 8, seed=5)
    assert work(w2) > SMALL
    both_paths(w2, expect_small=False)
