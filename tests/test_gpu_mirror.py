"""GPU mirror construction (kvs_mirror_build) vs the oracle: diff tables and
ids bit-exact, diff rows within one bf16 ulp (plus the float32 rotation bound
on rotated K), untouched rows exactly zero; and the mirror it builds restores
the refreshed cache through the attention overlay."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from shared_paged_kv_gb300 import kvs as K
from shared_paged_kv_gb300 import workloads as W
from oracle import attention as OA, fingerprint as OF, mirror as OM
import harness as H

f32 = W.bf16_bits_to_f32


def bf16_ulp(x):
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126)))
    return 2.0 ** (e - 7)


def pair_norm(x):
    """Norm of each rotate-half pair (i, i + d/2), repeated on both halves."""
    h = x.shape[-1] // 2
    r = np.sqrt(x[..., :h] ** 2 + x[..., h:] ** 2)
    return np.concatenate([r, r], axis=-1)


def refresh_positions(w, rng, frac=0.2, tail=True, skip=()):
    """Per agent an ascending random subset of its positions (CSR); agents in
    skip refresh nothing."""
    idx, off = [], [0]
    for a in range(w.n_seq):
        L = 0 if a in skip else int(w.seq_len[a])
        n = max(0, int(frac * L))
        pos = set(rng.choice(L, size=n, replace=False).tolist()) if n else set()
        if tail and L > 0:
            pos.add(L - 1)   # a position in the (possibly partial) last block
        idx.extend(sorted(pos))
        off.append(len(idx))
    return np.array(idx, np.int32), np.array(off, np.int64)


def build_case(w, rng, rope=True, frac=0.2, diff_capacity=None, skip=()):
    ref = OF.dedup(w.tokens, w.seq_off, w.tier, w.block_tokens, w.max_blocks,
                   w.seg_start_off, w.seg_start_blocks)
    table = ref["block_table"]
    idx, off = refresh_positions(w, rng, frac, skip=skip)
    n_rows = len(idx)
    kn = W.f32_to_bf16_bits(rng.standard_normal((n_rows, w.n_kv_heads, w.head_dim)).astype(np.float32))
    vn = W.f32_to_bf16_bits(rng.standard_normal((n_rows, w.n_kv_heads, w.head_dim)).astype(np.float32))
    cap_d = diff_capacity if diff_capacity is not None else w.n_seq * w.max_blocks
    kb, vb = w.kv_layer(0)
    cap = w.capacity_blocks
    dz = np.zeros((max(cap_d, 1), w.n_kv_heads, w.block_tokens, w.head_dim), np.uint16)
    dk_t, dv_t = H.bits_to_dev(dz), H.bits_to_dev(dz)
    pool = K.kvs_pool_create(1, w.n_kv_heads, w.head_dim, w.block_tokens, K.KVS_DTYPE_BF16, cap, w.n_seq,
                             [H.bits_to_dev(kb)], [H.bits_to_dev(vb)], dk_layers=[dk_t], dv_layers=[dv_t],
                             diff_capacity_blocks=cap_d)
    use_rope = rope and w.rope_off is not None
    ro = H.i32(w.rope_off) if use_rope else None
    rs = H.i32(w.rope_segs) if use_rope else None
    diff_table = torch.full((w.n_seq, w.max_blocks), 7, dtype=torch.int32, device=H.DEV)
    n_diff = torch.zeros(1, dtype=torch.int32, device=H.DEV)
    ws = H.workspace(K.kvs_workspace_size(pool, K.KVS_OP_MIRROR, w.n_seq, w.max_blocks))
    K.kvs_mirror_build(pool, 0, H.i32(table), w.max_blocks, H.i32(w.seq_len), w.n_seq, H.i32(idx), H.i64(off),
                       H.bits_to_dev(kn), H.bits_to_dev(vn), ro, rs, w.theta, diff_table, n_diff, ws)
    torch.cuda.synchronize()
    exp = OM.mirror_build(table, idx, off, f32(kn), f32(vn), f32(kb), f32(vb), w.block_tokens,
                          w.rope_off if use_rope else None, w.rope_segs if use_rope else None, w.theta)
    got = dict(diff_table=diff_table.cpu().numpy(), n_diff=int(n_diff.item()),
               dk=f32(dk_t.cpu().numpy().view(np.uint16)).astype(np.float64),
               dv=f32(dv_t.cpu().numpy().view(np.uint16)).astype(np.float64))
    return dict(pool=pool, table=table, idx=idx, off=off, kn=kn, vn=vn, kb=kb, vb=vb, exp=exp, got=got,
                use_rope=use_rope, dk_t=dk_t, dv_t=dv_t, diff_table=diff_table)


def check_diffs(c, w):
    exp, got = c["exp"], c["got"]
    assert got["n_diff"] == exp["n_diff"]
    assert np.array_equal(got["diff_table"], exp["diff_table"])
    n = exp["n_diff"]
    B = w.block_tokens
    refreshed = np.zeros((n, B), bool)
    for a in range(w.n_seq):
        for r in range(int(c["off"][a]), int(c["off"][a + 1])):
            b, o = divmod(int(c["idx"][r]), B)
            refreshed[exp["diff_table"][a, b], o] = True
    gk = got["dk"][:n].transpose(0, 2, 1, 3)   # [id][row][h][d]
    gv = got["dv"][:n].transpose(0, 2, 1, 3)
    ek = exp["dk"].transpose(0, 2, 1, 3)
    ev = exp["dv"].transpose(0, 2, 1, 3)
    # untouched rows of dirty blocks are exactly zero
    assert not gk[~refreshed].any() and not gv[~refreshed].any()
    # refreshed rows: one bf16 ulp, plus the float32 rotation bound on K
    tol_k = bf16_ulp(ek[refreshed])
    if c["use_rope"]:
        rows = np.zeros(refreshed.shape, np.int64)
        for a in range(w.n_seq):
            for r in range(int(c["off"][a]), int(c["off"][a + 1])):
                b, o = divmod(int(c["idx"][r]), B)
                rows[exp["diff_table"][a, b], o] = r
        tol_k = tol_k + 2.0 ** -19 * pair_norm(f32(c["kn"])[rows[refreshed]].astype(np.float64))
    assert (np.abs(gk[refreshed] - ek[refreshed]) <= tol_k).all()
    assert (np.abs(gv[refreshed] - ev[refreshed]) <= bf16_ulp(ev[refreshed])).all()
    assert K.kvs_pool_check(c["pool"]) == 0


def test_small_family_with_rotation():
    w = W.make_allgather(n_seq=4, n_segs=6, priv_blocks_lo=3, priv_blocks_hi=9, hq=10, hkv=2, n_layers=1)
    c = build_case(w, np.random.default_rng(1))
    check_diffs(c, w)


def test_d64_without_rotation_and_an_agent_without_refresh():
    w = W.make_prefix_shared("mir64", 5, 4, 2, 64, 1, 7 * 16 + 5, [40, 0, 130, 17, 64], seed=31)
    rng = np.random.default_rng(2)
    c = build_case(w, rng, rope=False, frac=0.3, skip={1})
    assert (c["got"]["diff_table"][1] == -1).all()
    check_diffs(c, w)


def test_mirror_restores_through_attention():
    """GPU mirror -> GPU attention with the diff overlay equals the oracle's
    attention over master + diffs (the oracle's own diffs rounded to bf16,
    the stored format)."""
    w = W.make_allgather(seed=6, n_seq=3, n_segs=4, priv_blocks_lo=2, priv_blocks_hi=6, hq=10, hkv=2,
                         n_layers=1)
    c = build_case(w, np.random.default_rng(3), frac=0.15)
    exp = c["exp"]
    q_bits = w.q_layer(0)
    out = torch.zeros((w.n_seq, w.n_q_heads, w.head_dim), dtype=torch.float32, device=H.DEV)
    ws = H.workspace(K.kvs_workspace_size(c["pool"], K.KVS_OP_DECODE_ATTN, w.n_seq, w.max_blocks, w.n_q_heads))
    K.kvs_decode_attn(c["pool"], 0, H.bits_to_dev(q_bits), w.n_q_heads, H.i32(c["table"]), w.max_blocks,
                      H.i32(w.seq_len), w.n_seq, c["diff_table"], H.i32(w.rope_off), H.i32(w.rope_segs), w.theta,
                      w.scale, out, ws)
    torch.cuda.synchronize()
    dk16 = f32(W.f32_to_bf16_bits(exp["dk"].astype(np.float32))).astype(np.float64)
    dv16 = f32(W.f32_to_bf16_bits(exp["dv"].astype(np.float32))).astype(np.float64)
    ref = OA.decode_attention(f32(q_bits), f32(c["kb"]), f32(c["vb"]), c["table"], w.seq_len, w.block_tokens,
                              w.scale, diff_table=exp["diff_table"], dk_pool=dk16, dv_pool=dv16,
                              rope_off=w.rope_off, rope_segs=w.rope_segs, theta=w.theta)
    H.assert_close_attn(out.cpu().numpy().astype(np.float64), ref)
    assert K.kvs_pool_check(c["pool"]) == 0


def test_bad_positions_and_small_diff_capacity_are_flagged():
    w = W.make_prefix_shared("mirbad", 3, 4, 2, 128, 1, 3 * 16, [20, 40, 9], seed=41)
    rng = np.random.default_rng(4)
    ref = OF.dedup(w.tokens, w.seq_off, w.tier, w.block_tokens, w.max_blocks)
    table = ref["block_table"]
    # agent 1's list is out of order; agent 2 refreshes a position beyond its context
    idx = np.array([0, 30, 50, 5, 70], np.int32)
    off = np.array([0, 2, 4, 5], np.int64)
    kn = W.f32_to_bf16_bits(rng.standard_normal((5, 2, 128)).astype(np.float32))
    kb, vb = w.kv_layer(0)
    dz = np.zeros((2, 2, 16, 128), np.uint16)
    pool = K.kvs_pool_create(1, 2, 128, 16, K.KVS_DTYPE_BF16, w.capacity_blocks, w.n_seq,
                             [H.bits_to_dev(kb)], [H.bits_to_dev(vb)], dk_layers=[H.bits_to_dev(dz)],
                             dv_layers=[H.bits_to_dev(dz)], diff_capacity_blocks=2)
    diff_table = torch.zeros((w.n_seq, w.max_blocks), dtype=torch.int32, device=H.DEV)
    n_diff = torch.zeros(1, dtype=torch.int32, device=H.DEV)
    ws = H.workspace(K.kvs_workspace_size(pool, K.KVS_OP_MIRROR, w.n_seq, w.max_blocks))
    K.kvs_mirror_build(pool, 0, H.i32(table), w.max_blocks, H.i32(w.seq_len), w.n_seq, H.i32(idx), H.i64(off),
                       H.bits_to_dev(kn), H.bits_to_dev(kn), None, None, 1e4, diff_table, n_diff, ws)
    flags = K.kvs_pool_check(pool)
    assert flags & K.KVS_DEVERR_JOB
    # agent 0: blocks 0 and 1 dirty; agent 1: the in-order row 50 marks block 3,
    # its out-of-order row is dropped; 3 dirty blocks exceed a capacity of 2
    assert flags & K.KVS_DEVERR_DIFF_ID
    assert int(n_diff.item()) == 3


def test_full_size_allgather_mirror_sampled():
    """64 agents, each refreshing every row of 31 blocks among its 512 shared
    blocks (the all-gather round's mirror structure), with rotation."""
    w = W.make_allgather(n_layers=1)
    rng = np.random.default_rng(5)
    ref = OF.dedup(w.tokens, w.seq_off, w.tier, w.block_tokens, w.max_blocks,
                   w.seg_start_off, w.seg_start_blocks)
    table = ref["block_table"]
    idx, off = [], [0]
    for a in range(w.n_seq):
        fb = int(w.rope_segs[w.rope_off[a]][0])   # first shared block of the agent
        blocks = np.sort(rng.choice(512, size=31, replace=False)) + fb
        for b in blocks:
            idx.extend(range(int(b) * 16, int(b) * 16 + 16))
        off.append(len(idx))
    idx = np.array(idx, np.int32)
    off = np.array(off, np.int64)
    n_rows = len(idx)
    H_, D = w.n_kv_heads, w.head_dim
    gen = torch.Generator(device=H.DEV).manual_seed(9)
    cap = ref["n_phys"]
    k_t = torch.randn((cap, H_, 16, D), generator=gen, device=H.DEV, dtype=torch.bfloat16)
    v_t = torch.randn((cap, H_, 16, D), generator=gen, device=H.DEV, dtype=torch.bfloat16)
    kn_t = torch.randn((n_rows, H_, D), generator=gen, device=H.DEV, dtype=torch.bfloat16)
    vn_t = torch.randn((n_rows, H_, D), generator=gen, device=H.DEV, dtype=torch.bfloat16)
    cap_d = w.n_seq * 31
    dk_t = torch.zeros((cap_d, H_, 16, D), device=H.DEV, dtype=torch.bfloat16)
    dv_t = torch.zeros_like(dk_t)
    pool = K.kvs_pool_create(1, H_, D, 16, K.KVS_DTYPE_BF16, cap, w.n_seq, [k_t.view(torch.int16)],
                             [v_t.view(torch.int16)], dk_layers=[dk_t.view(torch.int16)],
                             dv_layers=[dv_t.view(torch.int16)], diff_capacity_blocks=cap_d)
    diff_table = torch.zeros((w.n_seq, w.max_blocks), dtype=torch.int32, device=H.DEV)
    n_diff = torch.zeros(1, dtype=torch.int32, device=H.DEV)
    ws = H.workspace(K.kvs_workspace_size(pool, K.KVS_OP_MIRROR, w.n_seq, w.max_blocks))
    K.kvs_mirror_build(pool, 0, H.i32(table), w.max_blocks, H.i32(w.seq_len), w.n_seq, H.i32(idx), H.i64(off),
                       kn_t.view(torch.int16), vn_t.view(torch.int16), H.i32(w.rope_off), H.i32(w.rope_segs),
                       w.theta, diff_table, n_diff, ws)
    torch.cuda.synchronize()
    assert K.kvs_pool_check(pool) == 0
    assert int(n_diff.item()) == cap_d
    # the diff table, by an independent count of dirty (agent, block) slots
    dt = diff_table.cpu().numpy()
    keys = np.unique(np.repeat(np.arange(w.n_seq), np.diff(off)) * w.max_blocks + idx // 16)
    expect = np.full(w.n_seq * w.max_blocks, -1, np.int32)
    expect[keys] = np.arange(len(keys))
    assert np.array_equal(dt.reshape(-1), expect)
    # sampled rows through the oracle, on host copies of the rows involved
    for r in rng.choice(n_rows, size=12, replace=False):
        a = int(np.searchsorted(off, r, side="right") - 1)
        b, o = divmod(int(idx[r]), 16)
        p = int(table[a, b])
        kn1 = kn_t[r].float().cpu().numpy()[None].astype(np.float64)
        vn1 = vn_t[r].float().cpu().numpy()[None].astype(np.float64)
        km = k_t[p].float().cpu().numpy().astype(np.float64)[None]
        vm = v_t[p].float().cpu().numpy().astype(np.float64)[None]
        one = OM.mirror_build(np.array([[0] * b + [0]], np.int32), np.array([idx[r]]), np.array([0, 1]),
                              kn1, vn1, km, vm, 16,
                              np.array([0, 1], np.int32),
                              np.array([[b, 1, int(OA.segment_delta_per_block(w.max_blocks, w.rope_off,
                                                                              w.rope_segs, a)[b]), 0]], np.int32),
                              w.theta)
        i = int(dt[a, b])
        gk = dk_t[i, :, o, :].float().cpu().numpy().astype(np.float64)
        gv = dv_t[i, :, o, :].float().cpu().numpy().astype(np.float64)
        ek, ev = one["dk"][0, :, o, :], one["dv"][0, :, o, :]
        assert (np.abs(gk - ek) <= bf16_ulp(ek) + 2.0 ** -19 * pair_norm(kn1[0])).all()
        assert (np.abs(gv - ev) <= bf16_ulp(ev)).all()
