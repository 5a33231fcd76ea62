"""Helpers shared by the GPU parity tests: move seeded workload inputs to the
device, call the C-ABI entry points, and compare against the oracle."""
import numpy as np
import torch

from shared_paged_kv_gb300 import kvs as K
from shared_paged_kv_gb300 import workloads as W
from oracle import select as OS

DEV = torch.device("cuda:0")

ATOL = 1e-2      # max |delta| for attention outputs from bf16 inputs
RTOL_L2 = 2e-3   # relative L2 error for attention outputs


def bits_to_dev(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(DEV)


def i32(x) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32)).to(DEV)


def i64(x) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.int64)).to(DEV)


def dev_bits_to_f64(t: torch.Tensor) -> np.ndarray:
    return W.bf16_bits_to_f32(t.cpu().numpy().view(np.uint16)).astype(np.float64)


def workspace(nbytes: int) -> torch.Tensor:
    return torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=DEV)


def gpu_dedup(pool, w: W.Workload, flags: int = 0, segments: bool = True, tier=None):
    tokens = torch.from_numpy(w.tokens.view(np.int32)).to(DEV)
    seq_off = i64(w.seq_off)
    tier_t = None
    tier_np = w.tier if tier is None else tier
    if tier is not None or (w.tier != 0).any():
        tier_t = torch.from_numpy(np.ascontiguousarray(tier_np, dtype=np.uint32).view(np.int32)).to(DEV)
    seg_off = seg_blocks = None
    if segments and w.seg_start_off is not None:
        seg_off = i64(w.seg_start_off)
        seg_blocks = i32(w.seg_start_blocks)
    fp = torch.zeros(w.n_seq, w.max_blocks, dtype=torch.int64, device=DEV)
    table = torch.zeros(w.n_seq, w.max_blocks, dtype=torch.int32, device=DEV)
    cap = pool.desc.capacity_blocks
    refc = torch.zeros(cap, dtype=torch.int32, device=DEV)
    nphys = torch.zeros(1, dtype=torch.int32, device=DEV)
    owner = torch.full((cap,), -7, dtype=torch.int32, device=DEV)
    ref_off = torch.full((cap + 1,), -7, dtype=torch.int64, device=DEV)
    ref_seq = torch.full((max(w.n_seq * w.max_blocks, 1),), -7, dtype=torch.int32, device=DEV)
    ws = workspace(K.kvs_workspace_size(pool, K.KVS_OP_DEDUP, w.n_seq, w.max_blocks))
    K.kvs_fingerprint_dedup(pool, tokens, seq_off, w.n_seq, tier_t, seg_off, seg_blocks, fp, table,
                            w.max_blocks, refc, nphys, ws, flags=flags, owner_seq=owner, ref_off=ref_off,
                            ref_seq=ref_seq)
    torch.cuda.synchronize()
    n = int(nphys.item())
    return dict(fp=fp.cpu().numpy().view(np.uint64), block_table=table.cpu().numpy(),
                refcount=refc.cpu().numpy()[:n], refcount_full=refc.cpu().numpy(), n_phys=n,
                owner=owner.cpu().numpy(), ref_off=ref_off.cpu().numpy(), ref_seq=ref_seq.cpu().numpy(),
                refc_dev=refc, nphys_dev=nphys)


def bf16_pool(w: W.Workload, n_layers: int = 1, capacity=None, with_diff: bool = None, layers_np=None,
              path: str = "token_major"):
    """Pool of n_layers bf16 slabs filled from the workload's seeded values.
    path "token_major" makes every attention call on it take the planned
    token-major path (KVS_TEST_TOKEN_MAJOR), also for small calls, which the
    library would otherwise run on the single-kernel path; "auto" keeps the
    library's own choice."""
    cap = capacity or w.capacity_blocks
    ks, vs, dks, dvs = [], [], [], []
    host = []
    for l in range(n_layers):
        kb, vb = w.kv_layer(l) if layers_np is None else layers_np[l]
        if kb.shape[0] < cap:
            pad = np.zeros((cap - kb.shape[0],) + kb.shape[1:], np.uint16)
            kb, vb = np.concatenate([kb, pad]), np.concatenate([vb, pad])
        ks.append(bits_to_dev(kb))
        vs.append(bits_to_dev(vb))
        ent = {"k": kb, "v": vb}
        if with_diff if with_diff is not None else w.diff_capacity_blocks > 0:
            db, dvb = w.diff_layer(l)
            dks.append(bits_to_dev(db))
            dvs.append(bits_to_dev(dvb))
            ent.update(dk=db, dv=dvb)
        host.append(ent)
    use_diff = len(dks) > 0
    pool = K.kvs_pool_create(n_layers, w.n_kv_heads, w.head_dim, w.block_tokens, K.KVS_DTYPE_BF16, cap,
                             w.n_seq, ks, vs, dk_layers=dks if use_diff else None,
                             dv_layers=dvs if use_diff else None,
                             diff_capacity_blocks=w.diff_capacity_blocks if use_diff else 0)
    pool.host = host
    pool.dev = dict(k=ks, v=vs, dk=dks, dv=dvs)
    if path == "token_major":
        K.kvs_pool_set_test_flags(pool, K.KVS_TEST_TOKEN_MAJOR)
    return pool


def attn(pool, layer, q_bits, w: W.Workload, table, seq_len=None, diff=True, rope=True, n_seq=None):
    n = w.n_seq if n_seq is None else n_seq
    q = bits_to_dev(q_bits)
    sl = i32(w.seq_len if seq_len is None else seq_len)
    tb = i32(table)
    dt = i32(w.diff_table) if (diff and w.diff_table is not None) else None
    ro = rs = None
    if rope and w.rope_off is not None:
        ro = i32(w.rope_off)
        rs = i32(w.rope_segs)
    out = torch.full((n, w.n_q_heads, w.head_dim), float("nan"), dtype=torch.float32, device=DEV)
    ws = workspace(K.kvs_workspace_size(pool, K.KVS_OP_DECODE_ATTN, n, w.max_blocks, w.n_q_heads))
    K.kvs_decode_attn(pool, layer, q, w.n_q_heads, tb, w.max_blocks, sl, n, dt, ro, rs, w.theta, w.scale, out, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64)


def assert_close_attn(got, exp, atol=ATOL, rtol=RTOL_L2):
    assert np.isfinite(got).all(), "non-finite attention output"
    err = np.abs(got - exp).max()
    rel = np.linalg.norm(got - exp) / max(np.linalg.norm(exp), 1e-30)
    assert err <= atol and rel <= rtol, f"max|d|={err:.3e} relL2={rel:.3e}"
    return err, rel


def check_selection(kc_bits, kn_bits, off, ratio, gi, go):
    """A GPU selection (positions gi, offsets go) against the oracle: offsets
    equal, positions ascending, and the position sets equal except for ties
    within 1e-5 of the k-th score (relative to that score once it exceeds 1:
    the GPU sums row_elems squared differences in float32, whose rounding
    error is relative to the sum)."""
    f32 = W.bf16_bits_to_f32
    ridx, roff, sc = OS.select_critical(f32(kc_bits), f32(kn_bits), off, ratio)
    np.testing.assert_array_equal(go, roff)
    for a in range(len(off) - 1):
        g = set(gi[go[a]:go[a + 1]].tolist())
        r = set(ridx[roff[a]:roff[a + 1]].tolist())
        assert list(gi[go[a]:go[a + 1]]) == sorted(g)
        if g != r:
            s = sc[off[a]:off[a + 1]]
            kth = np.sort(s)[::-1][len(r) - 1]
            for t in g ^ r:
                assert abs(s[t] - kth) <= 1e-5 * max(1.0, kth), (a, t, s[t], kth)
