"""Shared chunks on the tensor cores (the wide tile: query group G >= 4,
head_dim 128, no rotation) vs the fp64 oracle, max|delta| <= 1e-2 and relative
L2 <= 2e-3, on tables built to reach its corners: groups whose members hold
different prefixes (the largest set of members with equal blocks shares, the
rest go private), contexts ending inside a shared prefix, chunks of several
128-token sub-tiles with row maxima that move between them, more shared work
items than SMs, and mirror diffs that take a block out of sharing."""
from types import SimpleNamespace

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from shared_paged_kv_gb300 import kvs as K
from shared_paged_kv_gb300 import workloads as W
from oracle import attention as OA
import harness as H
from test_gpu_attn import run_case

f32 = W.bf16_bits_to_f32


def table_case(table, seq_len, hq, hkv, kf, vf, seed):
    """Attention over an explicit block table and pool (float32 values,
    rounded to bf16) vs the oracle."""
    n, max_blocks = table.shape
    d = kf.shape[-1]
    kb, vb = W.f32_to_bf16_bits(kf), W.f32_to_bf16_bits(vf)
    rng = np.random.default_rng(seed)
    q_bits = W.f32_to_bf16_bits(rng.standard_normal((n, hq, d)).astype(np.float32))
    pool = K.kvs_pool_create(1, hkv, d, 16, K.KVS_DTYPE_BF16, kb.shape[0], n, [H.bits_to_dev(kb)],
                             [H.bits_to_dev(vb)])
    K.kvs_pool_set_test_flags(pool, K.KVS_TEST_TOKEN_MAJOR)   # the planned path, also for small calls
    w = SimpleNamespace(n_seq=n, n_q_heads=hq, head_dim=d, diff_table=None, rope_off=None, rope_segs=None,
                        max_blocks=max_blocks, theta=1e6, scale=1.0 / np.sqrt(d), seq_len=seq_len)
    got = H.attn(pool, 0, q_bits, w, table)
    exp = OA.decode_attention(f32(q_bits), f32(kb), f32(vb), table, seq_len, 16, w.scale)
    H.assert_close_attn(got, exp)
    assert K.kvs_pool_check(pool) == 0
    return got


def test_mixed_prefixes_largest_set_shares():
    """G = 4 (groups of 32 sequences), 40 sequences: prefix A (40 blocks) and
    prefix B (20 blocks, then private blocks).  Group 0 is mostly A, group 1
    mostly B; lengths end before, inside and after the prefixes, some in the
    middle of a block.  Keys of two A blocks are scaled up so the row maxima
    jump late in a chunk."""
    rng = np.random.default_rng(31)
    hq, hkv, d, n = 8, 2, 128, 40
    max_blocks = 64
    kinds = ["B" if (a >= 32 and a % 4 != 0) or (a < 32 and a % 3 == 1) else "A" for a in range(n)]
    seq_len = rng.integers(16 * 3, 16 * max_blocks + 1, size=n).astype(np.int32)
    seq_len[[0, 5, 33]] = [16 * 12 + 7, 16 * 40, 16 * 9 + 1]
    table = np.full((n, max_blocks), -1, np.int32)
    nxt = 60
    for a in range(n):
        nb = -(-int(seq_len[a]) // 16)
        for b in range(nb):
            if kinds[a] == "A" and b < 40:
                table[a, b] = b
            elif kinds[a] == "B" and b < 20:
                table[a, b] = 40 + b
            else:
                table[a, b] = nxt
                nxt += 1
    cap = nxt
    kf = rng.standard_normal((cap, hkv, 16, d)).astype(np.float32)
    vf = rng.standard_normal((cap, hkv, 16, d)).astype(np.float32)
    kf[[13, 30]] *= 4.0
    table_case(table, seq_len, hq, hkv, kf, vf, seed=32)


def test_group8_partial_overlap_between_sequences():
    """G = 8 (groups of 16): every sequence shares a different length of one
    prefix with the others, and pairs of sequences share a second-level
    branch, so the sharing sets change block by block."""
    rng = np.random.default_rng(41)
    hq, hkv, d, n = 16, 2, 128, 21
    max_blocks = 48
    table = np.full((n, max_blocks), -1, np.int32)
    seq_len = np.zeros(n, np.int32)
    nxt = 100
    for a in range(n):
        common = int(rng.integers(2, 30))
        for b in range(common):
            table[a, b] = b
        for b in range(common, common + 6):          # branch shared by the pair (a, a ^ 1)
            table[a, b] = 30 + (a // 2) * 6 + (b - common) if (a ^ 1) < n else nxt
            if (a ^ 1) >= n:
                nxt += 1
        tail = int(rng.integers(0, max_blocks - common - 6))
        for b in range(common + 6, common + 6 + tail):
            table[a, b] = nxt
            nxt += 1
        seq_len[a] = 16 * (common + 6 + tail) - int(rng.integers(0, 16))
    cap = nxt
    kf = rng.standard_normal((cap, hkv, 16, d)).astype(np.float32)
    vf = rng.standard_normal((cap, hkv, 16, d)).astype(np.float32)
    table_case(table, seq_len, hq, hkv, kf, vf, seed=42)


def test_long_prefix_several_subtiles_and_claims():
    """40 sequences (groups of 16) over a 9,000-token prefix: chunks of 16
    blocks (two sub-tiles each) and over 200 shared claims, more than the
    SMs, so CTAs take several claims and reload their query tile."""
    run_case(W.make_gqa_fanout(n_seq=40, prefix_tokens=9000, priv_lo=16, priv_hi=600, hq=16, hkv=2, d=128))


def test_diffs_take_blocks_out_of_sharing():
    """G = 5 (groups of 25 sequences) with mirror diffs on shared segment
    blocks and no rotation: a member with a diff computes that block
    privately; the others share it."""
    w = W.make_allgather(seed=12, n_seq=6, n_segs=6, priv_blocks_lo=3, priv_blocks_hi=9, hq=10, hkv=2,
                         n_layers=1)
    run_case(w, rope=False)


def test_repeatable_bitwise_with_wide_tile():
    w = W.make_gqa_fanout(n_seq=9, prefix_tokens=700, priv_lo=10, priv_hi=300, hq=16, hkv=2, d=128)
    a, _ = run_case(w)
    b, _ = run_case(w)
    assert np.array_equal(a, b)


def test_plan_routes_shared_chunks_to_the_wide_tile():
    """The plan header records the sharing-group size (16 sequences at G = 8)
    and a nonzero count of wide items for a shared prefix, and none when
    nothing is shared."""
    w = W.make_gqa_fanout(n_seq=20, prefix_tokens=512, priv_lo=16, priv_hi=200, hq=16, hkv=2, d=128)
    from oracle import fingerprint as OF
    ref = OF.dedup(w.tokens, w.seq_off, w.tier, w.block_tokens, w.max_blocks)
    pool = H.bf16_pool(w)
    nbytes = K.kvs_workspace_size(pool, K.KVS_OP_DECODE_ATTN, w.n_seq, w.max_blocks, w.n_q_heads)
    for table, expect_items in ((ref["block_table"], True),
                                (np.where(ref["block_table"] >= 0,
                                          np.arange(w.n_seq)[:, None] * w.max_blocks + np.arange(w.max_blocks),
                                          -1), False)):
        ws = H.workspace(nbytes)
        cap = pool.desc.capacity_blocks
        tb = np.where(table < cap, table, -1).astype(np.int32) if not expect_items else table
        K.kvs_decode_plan(pool, w.n_q_heads, H.i32(tb), w.max_blocks, H.i32(w.seq_len), w.n_seq, None, None,
                          None, ws)
        torch.cuda.synchronize()
        hdr = ws[:64].cpu().numpy().view(np.int32)
        assert hdr[7] == 16
        assert (hdr[8] > 0) == expect_items


def rope_case(table, seq_len, rope_off, rope_segs, hq, hkv, kf, vf, seed, diff_table=None, dkf=None, dvf=None):
    """Rotation call over an explicit table, segment list and pool vs the
    oracle (theta 1e6)."""
    n, max_blocks = table.shape
    d = kf.shape[-1]
    kb, vb = W.f32_to_bf16_bits(kf), W.f32_to_bf16_bits(vf)
    rng = np.random.default_rng(seed)
    q_bits = W.f32_to_bf16_bits(rng.standard_normal((n, hq, d)).astype(np.float32))
    kw = {}
    dkb = dvb = None
    if diff_table is not None:
        dkb, dvb = W.f32_to_bf16_bits(dkf), W.f32_to_bf16_bits(dvf)
        kw = dict(dk_layers=[H.bits_to_dev(dkb)], dv_layers=[H.bits_to_dev(dvb)], diff_capacity_blocks=dkb.shape[0])
    pool = K.kvs_pool_create(1, hkv, d, 16, K.KVS_DTYPE_BF16, kb.shape[0], n, [H.bits_to_dev(kb)],
                             [H.bits_to_dev(vb)], **kw)
    K.kvs_pool_set_test_flags(pool, K.KVS_TEST_TOKEN_MAJOR)   # the planned path, also for small calls
    w = SimpleNamespace(n_seq=n, n_q_heads=hq, head_dim=d, diff_table=diff_table, rope_off=rope_off,
                        rope_segs=rope_segs, max_blocks=max_blocks, theta=1e6, scale=1.0 / np.sqrt(d),
                        seq_len=seq_len)
    got = H.attn(pool, 0, q_bits, w, table)
    exp = OA.decode_attention(f32(q_bits), f32(kb), f32(vb), table, seq_len, 16, w.scale,
                              diff_table=diff_table, dk_pool=f32(dkb) if dkb is not None else None,
                              dv_pool=f32(dvb) if dvb is not None else None, rope_off=rope_off,
                              rope_segs=rope_segs, theta=1e6)
    H.assert_close_attn(got, exp)
    assert K.kvs_pool_check(pool) == 0
    return got


def test_rotation_runs_shared_across_positions_and_shifts():
    """G = 5 rotation call (groups of 25).  Three 8-block physical runs are
    placed by each of 9 members after a private prefix of its own length, in
    its own order and with its own shift: the tile shares each run across
    members at different logical positions.  Corners: a member holds one run
    twice (the first use is shared, the second private), a context ends
    inside a run (that run stays private), a mirror diff on one block keeps
    that member's run private, and two overlapping entries with equal shifts
    (only runs inside the last covering entry may be shared)."""
    rng = np.random.default_rng(61)
    hq, hkv, d, n = 10, 2, 128, 9
    runs = [np.arange(8) + 8 * j for j in range(3)]       # physical blocks 0..23
    nxt = 24
    rows, segs, lens = [], [], []
    for a in range(n):
        pre = int(rng.integers(0, 6))
        order = list(rng.permutation(3)) + ([1] if a == 2 else [])
        row = list(range(nxt, nxt + pre))
        nxt += pre
        sg = []
        if pre:
            sg.append([0, pre, int(rng.integers(-50, 50)), 0])
        for j in order:
            sg.append([len(row), 8, int(rng.integers(-3000, 3000)), 0])
            row += list(runs[j])
        if a == 4:   # equal-shift overlap: a later entry over the middle of the first two runs
            f0 = sg[1 if pre else 0][0]
            sg[1 if pre else 0][2] = sg[2 if pre else 1][2] = 777
            sg.append([f0 + 4, 8, 777, 0])
        tail = int(rng.integers(0, 4))
        row += list(range(nxt, nxt + tail))
        nxt += tail
        L = 16 * len(row)
        if a == 6:   # ends inside its last run: 5 of its 8 blocks, mid-block
            row = row[:len(row) - tail - 3]
            L = 16 * len(row) - 7
        rows.append(row)
        segs.append(sg)
        lens.append(L)
    max_blocks = max(len(r) for r in rows)
    table = np.full((n, max_blocks), -1, np.int32)
    for a, r in enumerate(rows):
        table[a, :len(r)] = r
    seq_len = np.array(lens, np.int32)
    rope_off = np.zeros(n + 1, np.int32)
    rope_off[1:] = np.cumsum([len(s) for s in segs])
    rope_segs = np.array([x for s in segs for x in s], np.int32).reshape(-1, 4)
    diff_table = np.full((n, max_blocks), -1, np.int32)
    diff_table[7, int(np.where(table[7] == 11)[0][0])] = 0   # member 7: a diff inside run 1
    cap = nxt
    kf = rng.standard_normal((cap, hkv, 16, d)).astype(np.float32)
    vf = rng.standard_normal((cap, hkv, 16, d)).astype(np.float32)
    dkf = 0.1 * rng.standard_normal((1, hkv, 16, d)).astype(np.float32)
    dvf = 0.1 * rng.standard_normal((1, hkv, 16, d)).astype(np.float32)
    rope_case(table, seq_len, rope_off, rope_segs, hq, hkv, kf, vf, seed=62, diff_table=diff_table, dkf=dkf,
              dvf=dvf)


def test_plan_routes_rotation_runs_to_the_wide_tile():
    """A rotation call with G = 5 (all-gather shape): the plan groups 25
    sequences and turns the shared 128-token segments into wide run items."""
    w = W.make_allgather(seed=13, n_seq=6, n_segs=6, priv_blocks_lo=3, priv_blocks_hi=9, hq=10, hkv=2, n_layers=1)
    from oracle import fingerprint as OF
    ref = OF.dedup(w.tokens, w.seq_off, w.tier, w.block_tokens, w.max_blocks, w.seg_start_off, w.seg_start_blocks)
    pool = H.bf16_pool(w)
    ws = H.workspace(K.kvs_workspace_size(pool, K.KVS_OP_DECODE_ATTN, w.n_seq, w.max_blocks, w.n_q_heads))
    K.kvs_decode_plan(pool, w.n_q_heads, H.i32(ref["block_table"]), w.max_blocks, H.i32(w.seq_len), w.n_seq,
                      H.i32(w.diff_table), H.i32(w.rope_off), H.i32(w.rope_segs), ws)
    torch.cuda.synchronize()
    hdr = ws[:64].cpu().numpy().view(np.int32)
    assert hdr[7] == 25
    assert hdr[8] >= 4   # most of the 6 segments are shared by at least two of the 6 agents
