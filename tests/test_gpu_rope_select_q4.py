"""GPU RoPE re-rotation, critical selection, Q4 quantiser and Q4 attention vs
the oracle."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from shared_paged_kv_gb300 import kvs as K
from shared_paged_kv_gb300 import workloads as W
from oracle import attention as OA, fingerprint as OF, q4 as OQ, rope as OR, select as OS
import harness as H

f32 = W.bf16_bits_to_f32


def bf16_ulp(x):
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126)))
    return 2.0 ** (e - 7)


def rope_tolerance(e):
    """One bf16 ulp of the fp64 result, plus 2^-19 of the norm of the rotated
    (i, i + d/2) pair: a rotation evaluated in float32 carries an absolute
    error proportional to the pair's size, which dominates the ulp when the
    result cancels to near zero."""
    h = e.shape[-1] // 2
    r = np.sqrt(e[..., :h] ** 2 + e[..., h:] ** 2)
    return bf16_ulp(e) + 2.0 ** -19 * np.concatenate([r, r], axis=-1)


# ---------------------------------------------------------------- RoPE ----
def rope_case(w, check_rows=None, device_values=False, edit_jobs=None):
    ref = OF.dedup(w.tokens, w.seq_off, w.tier, w.block_tokens, w.max_blocks, w.seg_start_off, w.seg_start_blocks)
    n_phys = ref["n_phys"]
    jobs, dst_table, n_dst = W.rope_jobs_for(w, first_free_block=n_phys)
    if edit_jobs is not None:
        jobs = edit_jobs(jobs)
    cap = n_phys + n_dst
    if device_values:
        # full size: K drawn by torch's seeded generator on the device
        gen = torch.Generator(device=H.DEV).manual_seed(5)
        k = torch.randn((cap, w.n_kv_heads, w.block_tokens, w.head_dim), generator=gen, device=H.DEV)
        k = k.to(torch.bfloat16).view(torch.int16)
        v = torch.zeros(16, dtype=torch.int16, device=H.DEV)
        pool = K.kvs_pool_create(1, w.n_kv_heads, w.head_dim, w.block_tokens, K.KVS_DTYPE_BF16, cap, w.n_seq, [k], [v])
        kdev = k
    else:
        pool = H.bf16_pool(w, capacity=cap, with_diff=False)
        kdev = pool.dev["k"][0]
    before = kdev[:n_phys].clone()
    sel = jobs if check_rows is None else jobs[check_rows]
    sel = sel[sel[:, 4] > 0]
    K.kvs_rope_rerotate(pool, 0, H.i32(jobs), len(jobs), int(jobs[:, 4].max()), w.theta,
                        H.i32(ref["block_table"]), H.i32(dst_table), w.max_blocks)
    torch.cuda.synchronize()
    assert K.kvs_pool_check(pool) == 0
    assert torch.equal(kdev[:n_phys], before)          # sources untouched
    # compact copy of the blocks the checked jobs touch, tables remapped
    B = w.block_tokens
    src_ids, dst_ids = set(), set()
    for (sr, st0, dr, dt0, n, _, _, _) in sel:
        src_ids.update(int(x) for x in ref["block_table"][sr, st0 // B:(st0 + n - 1) // B + 1])
        dst_ids.update(int(x) for x in dst_table[dr, dt0 // B:(dt0 + n - 1) // B + 1])
    src_ids, dst_ids = sorted(src_ids), sorted(dst_ids)
    remap = {b: i for i, b in enumerate(src_ids + dst_ids)}
    idx = torch.tensor(src_ids, device=H.DEV)
    src = np.zeros((len(remap),) + tuple(kdev.shape[1:]), np.float64)
    src[:len(src_ids)] = H.dev_bits_to_f64(kdev[idx])
    rt = np.vectorize(lambda b: remap.get(int(b), -1))
    exp, written = OR.rerotate_jobs(src, sel, rt(ref["block_table"]), rt(dst_table), B, w.theta)
    pd = np.array([dst_ids[p - len(src_ids)] for p, _ in written])
    pc = np.array([p for p, _ in written])
    od = np.array([o for _, o in written])
    got = H.dev_bits_to_f64(kdev[torch.from_numpy(pd).to(H.DEV), :, torch.from_numpy(od).to(H.DEV), :])
    e = exp[pc, :, od, :]
    assert (np.abs(got - e) <= rope_tolerance(e)).all(), f"max err {np.abs(got - e).max()}"
    return len(written)


def test_rope_small():
    rope_case(W.make_allgather(n_seq=4, n_segs=6, priv_blocks_lo=2, priv_blocks_hi=6, hq=8, hkv=2, n_layers=1))


def test_rope_small_d64_theta1e4():
    rope_case(W.make_allgather(seed=3, n_seq=3, n_segs=5, priv_blocks_lo=2, priv_blocks_hi=6, hq=4, hkv=2, d=64,
                               n_layers=1, theta=1e4))


def test_rope_ragged_jobs():
    """Jobs that start and end inside blocks, with lengths that are not a
    multiple of the tokens a warp step covers, an empty job, and five KV
    heads (a head batch that does not divide them)."""
    def ragged(jobs):
        out = jobs.copy()
        for i in range(len(out)):
            o = (7 * i) % 13
            n = int(out[i, 4]) - o - (i % 5)
            out[i, 1] += o; out[i, 3] += o; out[i, 5] += o; out[i, 6] += o
            out[i, 4] = max(n, 0) if i != 3 else 0
        return out
    n = rope_case(W.make_allgather(seed=4, n_seq=4, n_segs=6, priv_blocks_lo=2, priv_blocks_hi=6, hq=10, hkv=5,
                                   n_layers=1), edit_jobs=ragged)
    assert n > 0


def test_rope_bad_jobs_are_flagged():
    """A token range past the block table, an unmapped destination block and
    a shift of 2^18 each set their device error flag; nothing faults and the
    pool's blocks are not written."""
    w = W.make_allgather(n_seq=2, n_segs=2, priv_blocks_lo=2, priv_blocks_hi=3, hq=8, hkv=2, n_layers=1)
    ref = OF.dedup(w.tokens, w.seq_off, w.tier, w.block_tokens, w.max_blocks, w.seg_start_off, w.seg_start_blocks)
    n_phys = ref["n_phys"]
    jobs, dst_table, n_dst = W.rope_jobs_for(w, first_free_block=n_phys)
    pool = H.bf16_pool(w, capacity=n_phys + n_dst, with_diff=False)
    kdev = pool.dev["k"][0]
    lim = w.max_blocks * w.block_tokens
    cases = [
        (dict(col=3, val=lim - 8), K.KVS_DEVERR_JOB),            # runs past the table
        (dict(col=2, val=1, unmap=True), K.KVS_DEVERR_BLOCK_ID),  # destination row without blocks
        (dict(col=6, val=None), K.KVS_DEVERR_ROPE_RANGE),         # shift 2^18
    ]
    for edit, flag in cases:
        j = jobs[:1].copy()
        dt = dst_table.copy()
        if edit["col"] == 6:
            j[0, 6] = j[0, 5] + (1 << 18)
        else:
            j[0, edit["col"]] = edit["val"]
        if edit.get("unmap"):
            dt[1, :] = -1
        before = kdev.clone()
        K.kvs_rope_rerotate(pool, 0, H.i32(j), 1, int(j[0, 4]), w.theta, H.i32(ref["block_table"]), H.i32(dt),
                            w.max_blocks)
        torch.cuda.synchronize()
        assert K.kvs_pool_check(pool) & flag
        if flag != K.KVS_DEVERR_JOB:
            assert torch.equal(kdev, before)


def test_rope_full_size_sampled_jobs():
    w = W.make_allgather(n_layers=1)
    rng = np.random.default_rng(0)
    n = rope_case(w, check_rows=np.sort(rng.choice(w.n_seq * 64, size=24, replace=False)), device_values=True)
    assert n == 24 * 128


# ----------------------------------------------------------- selection ----
def select_case(kc_bits, kn_bits, off, ratio, max_rows):
    n = len(off) - 1
    row_elems = kc_bits.shape[1]
    ws = H.workspace(4 * n * max_rows)
    idx = torch.full((int(off[-1]) + 1,), -7, dtype=torch.int32, device=H.DEV)
    idx_off = torch.zeros(n + 1, dtype=torch.int64, device=H.DEV)
    K.kvs_select_critical(H.bits_to_dev(kc_bits), H.bits_to_dev(kn_bits), H.i64(off), n, max_rows, row_elems,
                          ratio, idx, idx_off, ws)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), idx_off.cpu().numpy()


check_selection = H.check_selection


def test_select_small():
    rows = [37, 1, 0, 200, 64]
    kc, kn, off = W.selection_inputs(1, len(rows), rows, 64)
    gi, go = select_case(kc, kn, off, 0.15, 256)
    check_selection(kc, kn, off, 0.15, gi, go)


def test_select_max_rows_and_malformed_offsets():
    # one agent at the 65,536-row limit
    kc, kn, off = W.selection_inputs(3, 1, [65536], 64)
    gi, go = select_case(kc, kn, off, 0.01, 65536)
    check_selection(kc, kn, off, 0.01, gi, go)
    # offsets that decrease (that agent selects nothing) and overlap (an agent
    # whose rows start inside its predecessor's): the oracle's slices of the
    # same offsets define both
    kc, kn, _ = W.selection_inputs(4, 3, [100, 50, 150], 64)
    off2 = np.array([0, 100, 50, 200], np.int64)
    gi, go = select_case(kc, kn, off2, 0.2, 150)
    assert go[2] == go[1]
    check_selection(kc, kn, off2, 0.2, gi, go)


def test_select_ties_and_ratio_edges():
    rows = [10, 10]
    kc = np.zeros((20, 16), np.uint16)
    kn = np.full((20, 16), 0x3F80, np.uint16)          # every score equal
    off = np.array([0, 10, 20], np.int64)
    gi, go = select_case(kc, kn, off, 0.35, 10)
    assert list(gi[go[0]:go[1]]) == [0, 1, 2, 3]        # ceil(3.5) lowest positions
    for r in (0.0, 1.0):
        gi, go = select_case(kc, kn, off, r, 10)
        assert go[-1] == (0 if r == 0 else 20)


def test_select_full_size():
    # 64 agents x 8192 shared positions x (8 KV heads x 128 dims); inputs drawn
    # on the device by torch's seeded generator, oracle on sampled agents.
    n, rows, E = 64, 8192, 1024
    gen = torch.Generator(device=H.DEV).manual_seed(11)
    kc = torch.randn((n * rows, E), generator=gen, device=H.DEV)
    sig = 0.05 + 0.45 * torch.rand((n * rows, 1), generator=gen, device=H.DEV)
    kn = (kc + torch.randn((n * rows, E), generator=gen, device=H.DEV) * sig).to(torch.bfloat16)
    kc = kc.to(torch.bfloat16)
    off = np.arange(n + 1, dtype=np.int64) * rows
    ws = H.workspace(4 * n * rows)
    idx = torch.full((n * rows,), -7, dtype=torch.int32, device=H.DEV)
    idx_off = torch.zeros(n + 1, dtype=torch.int64, device=H.DEV)
    K.kvs_select_critical(kc.view(torch.int16), kn.view(torch.int16), H.i64(off), n, rows, E, 0.15, idx, idx_off, ws)
    torch.cuda.synchronize()
    gi, go = idx.cpu().numpy(), idx_off.cpu().numpy()
    np.testing.assert_array_equal(go, np.arange(n + 1) * 1229)
    for a in (0, 17, 63):
        kcb = kc[a * rows:(a + 1) * rows].view(torch.int16).cpu().numpy().view(np.uint16)
        knb = kn[a * rows:(a + 1) * rows].view(torch.int16).cpu().numpy().view(np.uint16)
        sub_i = gi[go[a]:go[a + 1]]
        check_selection(kcb, knb, np.array([0, rows], np.int64), 0.15, sub_i, np.array([0, len(sub_i)], np.int64))


# ------------------------------------------------------------------ Q4 ----
def q4_pool(w, cap, n_layers=1):
    ks = [torch.zeros(cap * w.n_kv_heads * w.block_tokens * 64, dtype=torch.uint8, device=H.DEV) for _ in range(n_layers)]
    vs = [torch.zeros_like(ks[0]) for _ in range(n_layers)]
    ksb = [torch.zeros(cap * w.n_kv_heads * w.block_tokens * 4, dtype=torch.float16, device=H.DEV) for _ in range(n_layers)]
    vsb = [torch.zeros_like(ksb[0]) for _ in range(n_layers)]
    nd = w.diff_capacity_blocks
    dks = dvs = None
    if nd:
        # mirror diffs per 16-token sub-block, from the workload's seeded values
        dks, dvs = [], []
        for l in range(n_layers):
            db, dvb = w.diff_layer(l)
            dks.append(H.bits_to_dev(db))
            dvs.append(H.bits_to_dev(dvb))
    pool = K.kvs_pool_create(n_layers, w.n_kv_heads, 128, w.block_tokens, K.KVS_DTYPE_Q4G64, cap, w.n_seq,
                             ks, vs, ksb, vsb, dk_layers=dks, dv_layers=dvs, diff_capacity_blocks=nd)
    pool.q4 = (ks, vs, ksb, vsb)
    pool.diffs = (dks, dvs)
    return pool


def q4_case(w, sample_agents=None, q_pow2=0, gpu_diff_table=None, expect_flags=0, repeat=False):
    """Source bf16 K/V per physical block -> GPU quantiser; the oracle
    quantises the same source values itself and must match bit for bit; then
    Q4 attention vs the oracle on its dequantised values.  q_pow2 multiplies
    the query by 2^q_pow2 (exact in bf16) and the score scale by 2^-q_pow2.
    repeat: a second call on the same inputs must give the same bits."""
    ref = OF.dedup(w.tokens, w.seq_off, w.tier, w.block_tokens, w.max_blocks)
    cap = ref["n_phys"]
    g = torch.Generator(device=H.DEV).manual_seed(77)
    shape = (cap, w.n_kv_heads, w.block_tokens, 128)
    ksrc = torch.randn(shape, generator=g, device=H.DEV).to(torch.bfloat16)
    vsrc = torch.randn(shape, generator=g, device=H.DEV).to(torch.bfloat16)
    pool = q4_pool(w, cap)
    K.kvs_quantize_q4(pool, 0, ksrc.view(torch.int16), vsrc.view(torch.int16),
                      H.i32(np.arange(cap)), cap)
    q_bits = w.q_layer(0)
    scale = w.scale
    if q_pow2:
        q_bits = W.f32_to_bf16_bits(f32(q_bits) * np.float32(2.0 ** q_pow2))
        scale = w.scale * 2.0 ** -q_pow2
    n = w.n_seq
    out = torch.full((n, w.n_q_heads, 128), float("nan"), dtype=torch.float32, device=H.DEV)
    ws = H.workspace(K.kvs_workspace_size(pool, K.KVS_OP_DECODE_ATTN_Q4, n, w.max_blocks, w.n_q_heads))
    gdt = w.diff_table if gpu_diff_table is None else gpu_diff_table
    dt = H.i32(gdt) if gdt is not None else None
    K.kvs_decode_attn_q4(pool, 0, H.bits_to_dev(q_bits), w.n_q_heads, H.i32(ref["block_table"]), w.max_blocks,
                         H.i32(w.seq_len), n, scale, out, ws, diff_table=dt)
    torch.cuda.synchronize()
    assert K.kvs_pool_check(pool) == expect_flags
    got = out.cpu().numpy().astype(np.float64)
    if repeat:
        out2 = torch.full_like(out, float("nan"))
        K.kvs_decode_attn_q4(pool, 0, H.bits_to_dev(q_bits), w.n_q_heads, H.i32(ref["block_table"]), w.max_blocks,
                             H.i32(w.seq_len), n, scale, out2, ws, diff_table=dt)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int32), out2.view(torch.int32))
    ks, vs, ksb, vsb = pool.q4
    agents = range(n) if sample_agents is None else sample_agents
    blocks = sorted({int(b) for a in agents for b in ref["block_table"][a] if b >= 0})
    kcod = ks[0].view(cap, w.n_kv_heads, w.block_tokens, 64).cpu().numpy()
    vcod = vs[0].view(cap, w.n_kv_heads, w.block_tokens, 64).cpu().numpy()
    ksbh = ksb[0].view(cap, w.n_kv_heads, w.block_tokens, 2, 2).cpu().numpy()
    vsbh = vsb[0].view(cap, w.n_kv_heads, w.block_tokens, 2, 2).cpu().numpy()
    ks_src = ksrc.float().cpu().numpy()
    vs_src = vsrc.float().cpu().numpy()
    kd = np.zeros(shape, np.float64)
    vd = np.zeros(shape, np.float64)
    for b in blocks:
        c_k, sb_k = OQ.quantize(ks_src[b])
        c_v, sb_v = OQ.quantize(vs_src[b])
        np.testing.assert_array_equal(kcod[b], c_k)
        np.testing.assert_array_equal(vcod[b], c_v)
        np.testing.assert_array_equal(ksbh[b].view(np.uint16), sb_k.view(np.uint16))
        np.testing.assert_array_equal(vsbh[b].view(np.uint16), sb_v.view(np.uint16))
        kd[b] = OQ.dequantize(c_k, sb_k)
        vd[b] = OQ.dequantize(c_v, sb_v)
    dk_h = dv_h = None
    if w.diff_table is not None:
        dk_h, dv_h = (f32(x.cpu().numpy().view(np.uint16)) for x in (pool.diffs[0][0], pool.diffs[1][0]))
    exp = OA.decode_attention(f32(q_bits), kd, vd, ref["block_table"], w.seq_len, w.block_tokens, scale,
                              agents=agents, diff_table=w.diff_table, dk_pool=dk_h, dv_pool=dv_h,
                              diff_block_tokens=w.diff_block_tokens or None)
    sel = list(agents)
    H.assert_close_attn(got[sel], exp[sel])


def test_q4_small_ragged():
    w = W.make_q4(n_seq=3, ctx=700, hq=8, hkv=2)
    w2 = W.Workload(**{**w.__dict__})
    lens = np.array([700, 256, 513], np.int64)
    toks = np.concatenate([w.tokens[:700], w.tokens[700:956], w.tokens[1400:1913]])
    w2.tokens = toks
    w2.seq_off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    q4_case(w2)


def test_q4_group8():
    q4_case(W.make_q4(n_seq=2, ctx=600, hq=16, hkv=2))


def test_q4_query_outside_fp16_range():
    # the Q4 kernel multiplies in fp16: a bf16 query above 65504, or one deep
    # in fp16's subnormal range, must still give the oracle's attention
    w = W.make_q4(n_seq=2, ctx=600, hq=8, hkv=2)
    q_big = W.f32_to_bf16_bits(f32(w.q_layer(0)) * np.float32(2.0 ** 15))
    assert np.abs(f32(q_big)).max() > 65504.0
    q4_case(w, q_pow2=15)
    q4_case(w, q_pow2=-22)


def test_q4_diff_table_needs_diff_slabs():
    # a diff table on a Q4 pool created without mirror-diff slabs is an
    # argument error, raised before any launch
    w = W.make_q4(n_seq=2, ctx=300, hq=8, hkv=2)
    pool = q4_pool(w, 8)
    n = w.n_seq
    out = torch.zeros((n, w.n_q_heads, 128), dtype=torch.float32, device=H.DEV)
    ws = H.workspace(K.kvs_workspace_size(pool, K.KVS_OP_DECODE_ATTN_Q4, n, w.max_blocks, w.n_q_heads))
    dt = H.i32(np.full((n, w.max_blocks * 16), -1, np.int32))
    with pytest.raises(K.KvsError) as e:
        K.kvs_decode_attn_q4(pool, 0, H.bits_to_dev(w.q_layer(0)), w.n_q_heads,
                             H.i32(np.zeros((n, w.max_blocks), np.int32)), w.max_blocks, H.i32(w.seq_len), n,
                             w.scale, out, ws, diff_table=dt)
    assert e.value.status == K.KVS_ERR_INVALID_ARG


def test_q4_full_size_every_pair():
    q4_case(W.make_q4(n_layers=1))       # 12 agents x 32 heads


def test_q4_mirror_small_ragged():
    # mirror diffs on 16-token sub-blocks of Q4 masters, ragged lengths (the
    # last block partial, a dirty sub-block past the end of a sequence's
    # tokens) and a query group of 4
    w = W.make_q4_mirror(n_seq=3, ctx=700, hq=8, hkv=2, diff_frac=0.2)
    lens = np.array([700, 256, 513], np.int64)
    toks = np.concatenate([w.tokens[:700], w.tokens[700:956], w.tokens[1400:1913]])
    import dataclasses
    w2 = dataclasses.replace(w, tokens=toks, seq_off=np.concatenate([[0], np.cumsum(lens)]).astype(np.int64))
    q4_case(w2, repeat=True)


def test_q4_mirror_group8():
    q4_case(W.make_q4_mirror(n_seq=2, ctx=600, hq=16, hkv=2, diff_frac=0.3))


def test_q4_edge_lengths_with_and_without_diffs():
    # empty context (zeros), one token, exactly one block, a partial second block
    import dataclasses
    for frac in (0.0, 0.25):
        w = W.make_q4(n_seq=4, ctx=300, hq=8, hkv=2, diff_frac=frac)
        lens = np.array([0, 1, 256, 300], np.int64)
        toks = np.concatenate([w.tokens[300:301], w.tokens[600:856], w.tokens[900:1200]])
        q4_case(dataclasses.replace(w, tokens=toks, seq_off=np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)))


def test_q4_bad_diff_id_is_flagged_and_ignored():
    # an id beyond the diff capacity sets KVS_DEVERR_DIFF_ID and that
    # sub-block is read as the master alone (the oracle with the entry at -1)
    w = W.make_q4_mirror(n_seq=2, ctx=512, hq=8, hkv=2, diff_frac=0.1)
    a, sb = np.argwhere(w.diff_table >= 0)[0]
    bad = w.diff_table.copy()
    bad[a, sb] = w.diff_capacity_blocks + 5
    import dataclasses
    ok = w.diff_table.copy()
    ok[a, sb] = -1
    q4_case(dataclasses.replace(w, diff_table=ok), gpu_diff_table=bad, expect_flags=K.KVS_DEVERR_DIFF_ID)


def test_q4_mirror_full_size_every_pair():
    # the Q4 configuration with 31 dirty 16-token sub-blocks of 512 per agent
    q4_case(W.make_q4_mirror(n_layers=1))
