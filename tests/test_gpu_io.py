"""GPU block export / import (packed block records, the persistent-pool
round trip of the Q4 page) and Q4 attention over shared blocks."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from shared_paged_kv_gb300 import kvs as K
from shared_paged_kv_gb300 import workloads as W
from oracle import attention as OA, fingerprint as OF, q4 as OQ
import harness as H

f32 = W.bf16_bits_to_f32


def q4_layers(cap, hkv, layers, seed):
    g = torch.Generator(device=H.DEV).manual_seed(seed)
    codes = [torch.randint(0, 256, (cap, hkv, 256, 64), generator=g, device=H.DEV, dtype=torch.int32).to(torch.uint8)
             for _ in range(2 * layers)]
    sbs = [torch.randn((cap, hkv, 256, 4), generator=g, device=H.DEV).to(torch.float16) for _ in range(2 * layers)]
    return codes, sbs


def test_q4_export_layout_and_import_round_trip():
    cap, hkv, layers = 12, 2, 2
    codes, sbs = q4_layers(cap, hkv, layers, 5)
    pool = K.kvs_pool_create(layers, hkv, 128, 256, K.KVS_DTYPE_Q4G64, cap, 4, codes[0::2], codes[1::2],
                             sbs[0::2], sbs[1::2])
    rec = K.kvs_pool_block_bytes(pool)
    per_layer = 2 * hkv * 256 * 64 + 2 * hkv * 256 * 8
    assert rec == layers * per_layer
    blocks = np.array([3, 0, 5], np.int32)
    packed = torch.zeros(len(blocks) * rec, dtype=torch.uint8, device=H.DEV)
    K.kvs_pool_export(pool, H.i32(blocks), len(blocks), packed)
    torch.cuda.synchronize()
    # the record layout, from host copies of the slabs: per layer K codes,
    # V codes, K scale/bias, V scale/bias
    host = []
    for b in blocks:
        for l in range(layers):
            host += [codes[2 * l][b].cpu().numpy().tobytes(), codes[2 * l + 1][b].cpu().numpy().tobytes(),
                     sbs[2 * l][b].cpu().numpy().tobytes(), sbs[2 * l + 1][b].cpu().numpy().tobytes()]
    assert packed.cpu().numpy().tobytes() == b"".join(host)
    # import into other blocks: identical contents
    dst = np.array([7, 9, 11], np.int32)
    K.kvs_pool_import(pool, H.i32(dst), len(dst), packed)
    torch.cuda.synchronize()
    for s, d in zip(blocks, dst):
        for t in codes + sbs:
            assert torch.equal(t[d], t[s])
    assert K.kvs_pool_check(pool) == 0


def test_bf16_round_trip_and_bad_block():
    cap, hkv, layers, d = 10, 4, 3, 64
    g = torch.Generator(device=H.DEV).manual_seed(6)
    ks = [torch.randn((cap, hkv, 16, d), generator=g, device=H.DEV).to(torch.bfloat16).view(torch.int16)
          for _ in range(layers)]
    vs = [torch.randn((cap, hkv, 16, d), generator=g, device=H.DEV).to(torch.bfloat16).view(torch.int16)
          for _ in range(layers)]
    pool = K.kvs_pool_create(layers, hkv, d, 16, K.KVS_DTYPE_BF16, cap, 4, ks, vs)
    rec = K.kvs_pool_block_bytes(pool)
    assert rec == layers * 2 * hkv * 16 * d * 2
    packed = torch.zeros(2 * rec, dtype=torch.uint8, device=H.DEV)
    K.kvs_pool_export(pool, H.i32([1, 2]), 2, packed)
    K.kvs_pool_import(pool, H.i32([8, 9]), 2, packed)
    torch.cuda.synchronize()
    for t in ks + vs:
        assert torch.equal(t[8], t[1]) and torch.equal(t[9], t[2])
    K.kvs_pool_export(pool, H.i32([1, 99]), 2, packed)
    assert K.kvs_pool_check(pool) & K.KVS_DEVERR_BLOCK_ID
    with pytest.raises(K.KvsError):
        K.kvs_pool_export(pool, H.i32([1, 2, 3]), 3, packed)   # buffer too small


def test_q4_attention_over_shared_and_imported_blocks():
    """Four agents over a 3-block (768-token) common prefix of 256-token Q4
    blocks: attention equals the oracle on the dequantised codes, and is
    unchanged, bit for bit, after the blocks are exported and imported into
    other physical blocks and the tables redirected."""
    w = W.make_prefix_shared("q4sh", 4, 8, 2, 128, 1, 768, [100, 300, 0, 513], seed=51, block=256)
    ref = OF.dedup(w.tokens, w.seq_off, w.tier, w.block_tokens, w.max_blocks)
    table = ref["block_table"]
    n_phys = ref["n_phys"]
    assert n_phys < int(sum(-(-int(l) // 256) for l in w.seq_len))   # the prefix blocks are shared
    cap = 2 * n_phys
    g = torch.Generator(device=H.DEV).manual_seed(52)
    shape = (cap, w.n_kv_heads, 256, 128)
    ksrc = torch.randn(shape, generator=g, device=H.DEV).to(torch.bfloat16)
    vsrc = torch.randn(shape, generator=g, device=H.DEV).to(torch.bfloat16)
    codes = [torch.zeros((cap, w.n_kv_heads, 256, 64), dtype=torch.uint8, device=H.DEV) for _ in range(2)]
    sbs = [torch.zeros((cap, w.n_kv_heads, 256, 4), dtype=torch.float16, device=H.DEV) for _ in range(2)]
    pool = K.kvs_pool_create(1, w.n_kv_heads, 128, 256, K.KVS_DTYPE_Q4G64, cap, w.n_seq, [codes[0]], [codes[1]],
                             [sbs[0]], [sbs[1]])
    K.kvs_quantize_q4(pool, 0, ksrc.view(torch.int16), vsrc.view(torch.int16), H.i32(np.arange(n_phys)), n_phys)
    q_bits = w.q_layer(0)

    def attend(tab):
        out = torch.zeros((w.n_seq, w.n_q_heads, 128), dtype=torch.float32, device=H.DEV)
        ws = H.workspace(K.kvs_workspace_size(pool, K.KVS_OP_DECODE_ATTN_Q4, w.n_seq, w.max_blocks, w.n_q_heads))
        K.kvs_decode_attn_q4(pool, 0, H.bits_to_dev(q_bits), w.n_q_heads, H.i32(tab), w.max_blocks,
                             H.i32(w.seq_len), w.n_seq, w.scale, out, ws)
        torch.cuda.synchronize()
        return out

    out = attend(table)
    # oracle on the oracle's own quantisation of the same source values
    kd, vd = [], []
    for src in (ksrc, vsrc):
        x = src[:n_phys].float().cpu().numpy().astype(np.float32)
        c, sb = OQ.quantize(x)
        (kd if src is ksrc else vd).append(OQ.dequantize(c, sb))
    exp = OA.decode_attention(f32(q_bits), kd[0], vd[0], table, w.seq_len, 256, w.scale)
    H.assert_close_attn(out.cpu().numpy().astype(np.float64), exp)
    # export -> import into the upper half of the pool, redirect the tables
    rec = K.kvs_pool_block_bytes(pool)
    packed = torch.zeros(n_phys * rec, dtype=torch.uint8, device=H.DEV)
    K.kvs_pool_export(pool, H.i32(np.arange(n_phys)), n_phys, packed)
    K.kvs_pool_import(pool, H.i32(np.arange(n_phys) + n_phys), n_phys, packed)
    moved = np.where(table >= 0, table + n_phys, table).astype(np.int32)
    assert torch.equal(attend(moved), out)
    assert K.kvs_pool_check(pool) == 0
