"""GPU decode attention (bf16 pool, fused diff overlay and segment rotation)
vs the fp64 oracle: max|delta| <= 1e-2 and relative L2 <= 2e-3."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from shared_paged_kv_gb300 import kvs as K
from shared_paged_kv_gb300 import workloads as W
from oracle import attention as OA, fingerprint as OF
import harness as H

f32 = W.bf16_bits_to_f32


def oracle_out(w, pool, table, q_bits, layer=0, seq_len=None, diff=True, rope=True, agents=None, heads=None):
    hst = pool.host[layer]
    dk = f32(hst["dk"]) if diff and "dk" in hst else None
    dv = f32(hst["dv"]) if diff and "dv" in hst else None
    return OA.decode_attention(f32(q_bits), f32(hst["k"]), f32(hst["v"]), table,
                               w.seq_len if seq_len is None else seq_len, w.block_tokens, w.scale,
                               diff_table=w.diff_table if diff else None, dk_pool=dk, dv_pool=dv,
                               rope_off=w.rope_off if rope else None, rope_segs=w.rope_segs if rope else None,
                               theta=w.theta, agents=agents, heads=heads)


def run_case(w, diff=True, rope=True, seq_len=None):
    segs = w.seg_start_off is not None
    ref = OF.dedup(w.tokens, w.seq_off, w.tier, w.block_tokens, w.max_blocks,
                   w.seg_start_off if segs else None, w.seg_start_blocks if segs else None)
    pool = H.bf16_pool(w)
    q_bits = w.q_layer(0)
    got = H.attn(pool, 0, q_bits, w, ref["block_table"], seq_len=seq_len, diff=diff, rope=rope)
    exp = oracle_out(w, pool, ref["block_table"], q_bits, seq_len=seq_len, diff=diff, rope=rope)
    H.assert_close_attn(got, exp)
    assert K.kvs_pool_check(pool) == 0
    return got, exp


def test_tiny_with_mirror_diffs():
    run_case(W.make_tiny())


def test_tiny_without_diffs():
    run_case(W.make_tiny(), diff=False)


def test_mha_small_ragged():
    w = W.make_prefix_shared("mha_small", 3, 4, 4, 128, 1, 24 * 16, [16 * 16 + 5, 16 * 13, 16 * 17 + 11], seed=11)
    run_case(w)


def test_gqa_small_ragged():
    run_case(W.make_gqa_fanout(n_seq=5, prefix_tokens=256, priv_lo=30, priv_hi=300, hq=16, hkv=2, d=128))


def test_long_context_many_splits_separate_merge():
    # 2 sequences over a 24,000-token common prefix: about 2,500 blocks, 32-block
    # items, 79 chunks per sequence, so the separate merge walks three
    # 32-chunk windows of private and group-shared splits
    w = W.make_prefix_shared("long", 2, 4, 2, 64, 1, 24000, [16000 + 7, 9000], seed=21)
    run_case(w)


def test_many_sequences_multi_cta_plan():
    # 1,400 sequences in 700 groups of two over a 3-block common prefix: the
    # plan walks its groups with a grid-stride loop and compacts the item list
    # from many CTAs; some sequences hold only shared blocks
    rng = np.random.default_rng(5)
    w = W.make_prefix_shared("many", 1400, 8, 2, 64, 1, 48, rng.integers(0, 80, size=1400), seed=23)
    run_case(w)


@pytest.mark.parametrize("hq,hkv,d", [(10, 2, 128), (12, 2, 64), (14, 2, 128), (16, 2, 64)])
def test_wide_groups_two_column_tiles(hq, hkv, d):
    # 5 to 8 query heads per kv head: two 8-column tiles per warp, so 3 or 2
    # sequences share each tile over the common prefix (7 sequences: the last
    # group is partial); ragged private tails with mirror diffs off
    rng = np.random.default_rng(hq * 100 + d)
    w = W.make_prefix_shared("wide", 7, hq, hkv, d, 1, 20 * 16 + 3, rng.integers(1, 300, size=7), seed=hq + d)
    run_case(w)


def test_gqa_group16_d64():
    run_case(W.make_gqa_fanout(n_seq=3, prefix_tokens=100, priv_lo=1, priv_hi=200, hq=32, hkv=2, d=64))


def test_group12_d128_sixteen_row_kernel():
    # query groups of 9..16 heads take the 16-row (heads as M) kernel
    w = W.make_allgather(seed=5, n_seq=3, n_segs=4, priv_blocks_lo=2, priv_blocks_hi=7, hq=24, hkv=2, n_layers=1)
    run_case(w)


def test_allgather_small_rotation_and_diffs():
    w = W.make_allgather(n_seq=4, n_segs=6, priv_blocks_lo=3, priv_blocks_hi=9, hq=10, hkv=2, n_layers=1)
    run_case(w)
    run_case(w, rope=False)


def test_overlapping_rope_segments_last_entry_wins():
    # an extra entry for agent 0 covers the second half of its first shared
    # segment with another shift; where entries overlap, the last entry
    # covering a block applies (the oracle's rule and the plan's)
    import dataclasses
    w = W.make_allgather(n_seq=3, n_segs=4, priv_blocks_lo=2, priv_blocks_hi=5, hq=10, hkv=2, n_layers=1)
    ro, rs = w.rope_off.copy(), w.rope_segs.copy()
    fb, nb, dl, _ = rs[ro[0]]
    extra = np.array([[fb + nb // 2, nb - nb // 2, dl + 37, 0]], dtype=rs.dtype)
    rs2 = np.concatenate([rs[:ro[1]], extra, rs[ro[1]:]])
    ro2 = ro.copy()
    ro2[1:] += 1
    run_case(dataclasses.replace(w, rope_off=ro2, rope_segs=rs2))



def test_rotation_calls_repeat_on_one_pool():
    """Rotation calls on the wide tile: the token-major kernel takes its
    claims from a per-pool counter that the merge resets, so consecutive
    calls on one pool (two query sets, the first repeated) each match the
    oracle, and the repeated call is bit-identical."""
    w = W.make_allgather(seed=21, n_seq=6, n_segs=6, priv_blocks_lo=3, priv_blocks_hi=9, hq=10, hkv=2, n_layers=1)
    ref = OF.dedup(w.tokens, w.seq_off, w.tier, w.block_tokens, w.max_blocks, w.seg_start_off, w.seg_start_blocks)
    pool = H.bf16_pool(w)
    rng = np.random.default_rng(5)
    q1 = w.q_layer(0)
    q2 = W.f32_to_bf16_bits(rng.standard_normal(q1.shape).astype(np.float32))
    outs = []
    for q_bits in (q1, q2, q1):
        got = H.attn(pool, 0, q_bits, w, ref["block_table"])
        H.assert_close_attn(got, oracle_out(w, pool, ref["block_table"], q_bits))
        outs.append(got)
    assert np.array_equal(outs[0], outs[2])
    assert K.kvs_pool_check(pool) == 0


def test_rotation_calls_with_more_claims_than_tile_ctas():
    """260 agents at 40 query / 8 KV heads: 11 sharing groups x 8 KV heads
    give more wide-tile claims than the tile's CTAs (half of the SMs), so
    CTAs take several claims in turn, each with its own query tile, splits
    and tensor-memory epilogue; sampled agents match the oracle."""
    w = W.make_allgather(seed=31, n_seq=260, n_segs=3, priv_blocks_lo=1, priv_blocks_hi=3, hq=40, hkv=8, n_layers=1)
    ref = OF.dedup(w.tokens, w.seq_off, w.tier, w.block_tokens, w.max_blocks, w.seg_start_off, w.seg_start_blocks)
    pool = H.bf16_pool(w)
    q_bits = w.q_layer(0)
    got = H.attn(pool, 0, q_bits, w, ref["block_table"])
    agents = [0, 1, 24, 25, 130, 258, 259]
    exp = oracle_out(w, pool, ref["block_table"], q_bits, agents=agents)
    H.assert_close_attn(got[agents], exp[agents])
    assert K.kvs_pool_check(pool) == 0

def test_allgather_d64_rotation():
    w = W.make_allgather(seed=9, n_seq=3, n_segs=5, priv_blocks_lo=2, priv_blocks_hi=5, hq=4, hkv=2, d=64,
                         n_layers=1, theta=1e4)
    run_case(w)


@pytest.mark.parametrize("kind", ["gqa_wide", "allgather_rotation"])
def test_collective_call_equals_per_agent_calls(kind):
    # the collective call (shared blocks computed once for the group, on the
    # wide tile) against one call per agent on the same pool, where nothing is
    # shared: every agent's output agrees, and both match the oracle
    import dataclasses
    if kind == "gqa_wide":
        w = W.make_gqa_fanout(n_seq=6, prefix_tokens=300, priv_lo=20, priv_hi=200, hq=16, hkv=2, d=128)
    else:
        w = W.make_allgather(n_seq=4, n_segs=5, priv_blocks_lo=2, priv_blocks_hi=6, hq=10, hkv=2, n_layers=1)
    segs = w.seg_start_off is not None
    ref = OF.dedup(w.tokens, w.seq_off, w.tier, w.block_tokens, w.max_blocks,
                   w.seg_start_off if segs else None, w.seg_start_blocks if segs else None)
    pool = H.bf16_pool(w)
    q_bits = w.q_layer(0)
    together = H.attn(pool, 0, q_bits, w, ref["block_table"])
    exp = oracle_out(w, pool, ref["block_table"], q_bits)
    H.assert_close_attn(together, exp)
    for a in range(w.n_seq):
        ro = rs = None
        if w.rope_off is not None:
            rs = w.rope_segs[w.rope_off[a]:w.rope_off[a + 1]]
            ro = np.array([0, len(rs)], np.int32)
        w1 = dataclasses.replace(w, n_seq=1, seq_off=np.array([0, w.seq_len[a]], np.int64),
                                 diff_table=None if w.diff_table is None else w.diff_table[a:a + 1],
                                 rope_off=ro, rope_segs=rs)
        alone = H.attn(pool, 0, q_bits[a:a + 1], w1, ref["block_table"][a:a + 1])
        H.assert_close_attn(alone[0], exp[a])
        H.assert_close_attn(alone[0], together[a])
    assert K.kvs_pool_check(pool) == 0


@pytest.mark.parametrize("kind", ["tiny", "allgather_rotation"])
def test_fused_diff_overlay_equals_materialised_mirror(kind):
    # the same attention with every mirror-diff block materialised as a plain
    # block of its own (master + diff rounded to bf16, the agent's table
    # pointing at it, no diff table): the fused overlay agrees with it, and
    # each agrees with the oracle on its own values
    import dataclasses
    if kind == "tiny":
        w = W.make_tiny()
    else:
        w = W.make_allgather(n_seq=4, n_segs=6, priv_blocks_lo=3, priv_blocks_hi=9, hq=10, hkv=2, n_layers=1)
    segs = w.seg_start_off is not None
    ref = OF.dedup(w.tokens, w.seq_off, w.tier, w.block_tokens, w.max_blocks,
                   w.seg_start_off if segs else None, w.seg_start_blocks if segs else None)
    table = ref["block_table"]
    pool = H.bf16_pool(w)
    q_bits = w.q_layer(0)
    fused = H.attn(pool, 0, q_bits, w, table)
    H.assert_close_attn(fused, oracle_out(w, pool, table, q_bits))
    hst = pool.host[0]
    kb, vb, dkb, dvb = hst["k"], hst["v"], hst["dk"], hst["dv"]
    new_k, new_v = [kb], [vb]
    table_m = table.copy()
    nxt = kb.shape[0]
    for a in range(w.n_seq):
        for b in range(w.max_blocks):
            d = int(w.diff_table[a, b])
            if d < 0 or table[a, b] < 0:
                continue
            p = int(table[a, b])
            new_k.append(W.f32_to_bf16_bits(f32(kb[p]) + f32(dkb[d]))[None])
            new_v.append(W.f32_to_bf16_bits(f32(vb[p]) + f32(dvb[d]))[None])
            table_m[a, b] = nxt
            nxt += 1
    assert nxt > kb.shape[0], "the workload carries mirror diffs"
    km, vm = np.concatenate(new_k), np.concatenate(new_v)
    wm = dataclasses.replace(w, diff_table=None, diff_capacity_blocks=0, capacity_blocks=km.shape[0])
    pool_m = H.bf16_pool(wm, layers_np=[(km, vm)], with_diff=False)
    mat = H.attn(pool_m, 0, q_bits, wm, table_m)
    H.assert_close_attn(mat, oracle_out(wm, pool_m, table_m, q_bits))
    H.assert_close_attn(fused, mat)
    assert K.kvs_pool_check(pool) == 0 and K.kvs_pool_check(pool_m) == 0


def test_edge_lengths():
    # empty context -> zeros; a single token -> that token's V; exact block
    # multiples and one-past.
    w = W.make_gqa_fanout(n_seq=5, prefix_tokens=64, priv_lo=40, priv_hi=90, hq=8, hkv=2, d=128)
    sl = w.seq_len.copy()
    sl[0], sl[1], sl[2], sl[3] = 0, 1, 64, 17
    got, exp = run_case(w, seq_len=sl)
    assert np.all(got[0] == 0)


def test_shared_layout_equals_private_layout_on_gpu():
    # The same values in a deduplicated pool and in a fully private pool give
    # the same GPU output (and both match the oracle).
    w = W.make_gqa_fanout(n_seq=4, prefix_tokens=160, priv_lo=16, priv_hi=64, hq=8, hkv=2, d=128)
    ref = OF.dedup(w.tokens, w.seq_off, w.tier, w.block_tokens, w.max_blocks)
    pool = H.bf16_pool(w)
    q_bits = w.q_layer(0)
    o1 = H.attn(pool, 0, q_bits, w, ref["block_table"])
    tb = ref["block_table"]
    kb, vb = pool.host[0]["k"], pool.host[0]["v"]
    rows_k, rows_v, priv = [], [], np.full_like(tb, -1)
    for a in range(w.n_seq):
        for b in range(w.max_blocks):
            if tb[a, b] >= 0:
                priv[a, b] = len(rows_k)
                rows_k.append(kb[tb[a, b]])
                rows_v.append(vb[tb[a, b]])
    w2 = W.Workload(**{**w.__dict__, "capacity_blocks": len(rows_k)})
    pool2 = H.bf16_pool(w2, layers_np=[(np.stack(rows_k), np.stack(rows_v))])
    o2 = H.attn(pool2, 0, q_bits, w2, priv)
    # the deduplicated layout lets a group of sequences share one pass over a
    # common block, so only the fp32 summation order differs
    np.testing.assert_allclose(o1, o2, rtol=1e-5, atol=1e-6)
    exp = oracle_out(w, pool, ref["block_table"], q_bits)
    H.assert_close_attn(o1, exp)


def test_plan_reused_across_layers_and_mismatch_flagged():
    # one plan per step serves every layer; a call whose shapes do not match
    # the plan is reported on the device and writes nothing
    w = W.make_mha7b(n_seq=5, total_blocks=40, shared_blocks=25, n_layers=2, heads=4)
    ref = OF.dedup(w.tokens, w.seq_off, w.tier, w.block_tokens, w.max_blocks)
    pool = H.bf16_pool(w, n_layers=2)
    tb, sl = H.i32(ref["block_table"]), H.i32(w.seq_len)
    ws = H.workspace(K.kvs_workspace_size(pool, K.KVS_OP_DECODE_ATTN, w.n_seq, w.max_blocks, w.n_q_heads))
    K.kvs_decode_plan(pool, w.n_q_heads, tb, w.max_blocks, sl, w.n_seq, None, None, None, ws)
    for layer in range(2):
        q_bits = w.q_layer(layer)
        out = torch.full((w.n_seq, w.n_q_heads, w.head_dim), float("nan"), device=H.DEV)
        K.kvs_decode_attn_planned(pool, layer, H.bits_to_dev(q_bits), w.n_q_heads, tb, w.max_blocks, sl, w.n_seq,
                                  None, None, None, w.theta, w.scale, out, ws)
        torch.cuda.synchronize()
        exp = oracle_out(w, pool, ref["block_table"], q_bits, layer=layer)
        H.assert_close_attn(out.cpu().numpy().astype(np.float64), exp)
    assert K.kvs_pool_check(pool) == 0
    out = torch.full((w.n_seq - 1, w.n_q_heads, w.head_dim), 7.0, device=H.DEV)
    K.kvs_decode_attn_planned(pool, 0, H.bits_to_dev(w.q_layer(0)[:-1]), w.n_q_heads, tb, w.max_blocks, sl,
                              w.n_seq - 1, None, None, None, w.theta, w.scale, out, ws)
    assert K.kvs_pool_check(pool) & K.KVS_DEVERR_PLAN
    assert torch.all(out == 7.0)


def test_group_sharing_partial_groups_and_ragged_prefix_ends():
    # MHA (groups of 8): 11 sequences -> a full and a partial group; contexts
    # of different lengths end inside and after the shared prefix
    w = W.make_prefix_shared("mha_groups", 11, 2, 2, 128, 1, 30 * 16,
                             [0, 5, 16 * 3, 16 * 9 + 1, 7, 16 * 20, 16 * 2 + 15, 40, 16, 3, 16 * 6], seed=21)
    sl = w.seq_len.copy()
    sl[0] = 16 * 12          # ends inside the shared prefix
    sl[3] = 16 * 30          # exactly at its end
    run_case(w, seq_len=sl)


def test_bad_block_id_is_flagged_not_faulted():
    w = W.make_tiny()
    ref = OF.dedup(w.tokens, w.seq_off, w.tier, w.block_tokens, w.max_blocks)
    tb = ref["block_table"].copy()
    tb[1, 3] = w.capacity_blocks + 7
    pool = H.bf16_pool(w)
    H.attn(pool, 0, w.q_layer(0), w, tb)
    assert K.kvs_pool_check(pool) & K.KVS_DEVERR_BLOCK_ID
    assert K.kvs_pool_check(pool) == 0     # reading clears the word


def test_repeatable_bitwise():
    w = W.make_allgather(n_seq=4, n_segs=6, priv_blocks_lo=3, priv_blocks_hi=9, hq=10, hkv=2, n_layers=1)
    ref = OF.dedup(w.tokens, w.seq_off, w.tier, w.block_tokens, w.max_blocks, w.seg_start_off, w.seg_start_blocks)
    pool = H.bf16_pool(w)
    q = w.q_layer(0)
    a = H.attn(pool, 0, q, w, ref["block_table"])
    b = H.attn(pool, 0, q, w, ref["block_table"])
    np.testing.assert_array_equal(a, b)


# ---------------------------------------------------------------- full size ---
def full_size_all(w, layer_seed=0):
    """Full-size pool generated on the device by torch's seeded generator;
    the oracle recomputes every (agent, query head) output of the layer from
    a host copy of the slabs (input values only) and the two are compared
    element by element."""
    segs = w.seg_start_off is not None
    ref = OF.dedup(w.tokens, w.seq_off, w.tier, w.block_tokens, w.max_blocks,
                   w.seg_start_off if segs else None, w.seg_start_blocks if segs else None)
    cap = ref["n_phys"]
    g = torch.Generator(device=H.DEV).manual_seed(1234 + layer_seed)
    shape = (cap, w.n_kv_heads, w.block_tokens, w.head_dim)
    k = torch.randn(shape, generator=g, device=H.DEV).to(torch.bfloat16)
    v = torch.randn(shape, generator=g, device=H.DEV).to(torch.bfloat16)
    dks = dvs = None
    if w.diff_capacity_blocks:
        dshape = (w.diff_capacity_blocks,) + shape[1:]
        dks = [(0.1 * torch.randn(dshape, generator=g, device=H.DEV)).to(torch.bfloat16)]
        dvs = [(0.1 * torch.randn(dshape, generator=g, device=H.DEV)).to(torch.bfloat16)]
    pool = K.kvs_pool_create(1, w.n_kv_heads, w.head_dim, w.block_tokens, K.KVS_DTYPE_BF16, cap, w.n_seq,
                             [k.view(torch.int16)], [v.view(torch.int16)],
                             dk_layers=[x.view(torch.int16) for x in dks] if dks else None,
                             dv_layers=[x.view(torch.int16) for x in dvs] if dvs else None,
                             diff_capacity_blocks=w.diff_capacity_blocks)
    q_bits = w.q_layer(0)
    got = H.attn(pool, 0, q_bits, w, ref["block_table"])
    assert K.kvs_pool_check(pool) == 0
    assert np.isfinite(got).all()
    host = lambda t: t.float().cpu().numpy()
    exp = OA.decode_attention(f32(q_bits), host(k), host(v), ref["block_table"], w.seq_len, w.block_tokens,
                              w.scale, diff_table=w.diff_table, dk_pool=host(dks[0]) if dks else None,
                              dv_pool=host(dvs[0]) if dvs else None, rope_off=w.rope_off, rope_segs=w.rope_segs,
                              theta=w.theta)
    H.assert_close_attn(got, exp)
    for a in range(w.n_seq):      # and no agent hides a large local error
        H.assert_close_attn(got[a], exp[a])


def test_full_size_mha7b_every_pair():
    full_size_all(W.make_mha7b(n_layers=1))          # 8 agents x 32 heads


def test_full_size_gqa_fanout_every_pair():
    full_size_all(W.make_gqa_fanout(n_layers=1))     # 32 sequences x 16 heads


def test_full_size_allgather_every_pair():
    full_size_all(W.make_allgather(n_layers=1))      # 64 agents x 40 heads
