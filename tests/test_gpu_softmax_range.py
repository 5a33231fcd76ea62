"""Online-softmax rescale events vs the fp64 oracle (max|delta| <= 1e-2,
relative L2 <= 2e-3).  Keys are built so that a block's scores sit on a level
set by its physical id, with levels that jump by up to ~60 (log2 units of P)
between consecutive blocks, up and down, plus a jitter inside each block.
The attention kernels keep a column's reference point until a score exceeds
it by 2^8, so within one item some blocks take the lazy path (P up to 2^8, no
rescale) and others reduce the maxima and rescale; the small steps make P
climb towards 2^8 across several blocks before a rescale.  Every path of the
call runs: the planned token-major path (with the tensor-core tile for the
shared prefix where the group allows it) and the single-kernel small-call
path."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from types import SimpleNamespace

from shared_paged_kv_gb300 import kvs as K
from shared_paged_kv_gb300 import workloads as W
from oracle import attention as OA
import harness as H

f32 = W.bf16_bits_to_f32


def crafted_pool(n_phys, hkv, d, step, seed):
    """K = level(phys) + jitter(token) + small noise; V standard normal."""
    rng = np.random.default_rng(seed)
    level = ((np.arange(n_phys) * 5) % 11).astype(np.float32) * step
    jit = rng.uniform(0.0, 1.0, size=(n_phys, hkv, 16, 1)).astype(np.float32) * step
    kf = rng.standard_normal((n_phys, hkv, 16, d)).astype(np.float32) * 0.05 + level[:, None, None, None] + jit
    vf = rng.standard_normal((n_phys, hkv, 16, d)).astype(np.float32)
    return kf, vf


def shared_tables(n_seq, prefix_blocks, priv_blocks):
    """Block tables over a common prefix (physical ids 0..prefix-1) and
    private tails (fresh ids), padded with -1."""
    max_blocks = prefix_blocks + max(priv_blocks)
    table = np.full((n_seq, max_blocks), -1, np.int32)
    nxt = prefix_blocks
    for a, nb in enumerate(priv_blocks):
        table[a, :prefix_blocks] = np.arange(prefix_blocks)
        table[a, prefix_blocks:prefix_blocks + nb] = np.arange(nxt, nxt + nb)
        nxt += nb
    return table, nxt


def run(table, seq_len, hq, hkv, d, step, seed, path):
    n, max_blocks = table.shape
    n_phys = int(table.max()) + 1
    kf, vf = crafted_pool(n_phys, hkv, d, step, seed)
    kb, vb = W.f32_to_bf16_bits(kf), W.f32_to_bf16_bits(vf)
    rng = np.random.default_rng(seed + 1)
    # q close to +1 or -1 per head: scores follow the key levels up for some
    # heads and down for others
    sign = np.where(np.arange(hq) % 2 == 0, 1.0, -1.0).astype(np.float32)
    qf = sign[None, :, None] * (1.0 + 0.05 * rng.standard_normal((n, hq, d)).astype(np.float32))
    q_bits = W.f32_to_bf16_bits(qf)
    pool = K.kvs_pool_create(1, hkv, d, 16, K.KVS_DTYPE_BF16, n_phys, n, [H.bits_to_dev(kb)], [H.bits_to_dev(vb)])
    if path == "token_major":
        K.kvs_pool_set_test_flags(pool, K.KVS_TEST_TOKEN_MAJOR)
    w = SimpleNamespace(n_seq=n, n_q_heads=hq, head_dim=d, diff_table=None, rope_off=None, rope_segs=None,
                        max_blocks=max_blocks, theta=1e6, scale=1.0 / np.sqrt(d), seq_len=seq_len)
    n0 = K.kvs_launch_count()
    got = H.attn(pool, 0, q_bits, w, table)
    launches = K.kvs_launch_count() - n0
    exp = OA.decode_attention(f32(q_bits), f32(kb), f32(vb), table, seq_len, 16, w.scale)
    H.assert_close_attn(got, exp)
    assert K.kvs_pool_check(pool) == 0
    return launches


@pytest.mark.parametrize("path", ["token_major", "auto"])
@pytest.mark.parametrize("step", [0.4, 0.06])
@pytest.mark.parametrize("hq,hkv,d", [(2, 2, 128), (8, 2, 64), (16, 2, 128)])
def test_score_levels_jump_between_blocks(hq, hkv, d, step, path):
    # three sequences over a 24-block prefix with 9, 30 and 41 private blocks
    # (ragged last blocks): long enough for several items per sequence on the
    # planned path, and small enough (3 x 2 x 65 blocks) for the small-call path
    table, _ = shared_tables(3, 24, [9, 30, 41])
    seq_len = np.array([33 * 16 - 5, 54 * 16, 65 * 16 - 11], np.int32)
    launches = run(table, seq_len, hq, hkv, d, step, seed=hq * 10 + d + int(step * 100), path=path)
    if path == "auto":
        assert launches == 1   # the single-kernel path


@pytest.mark.parametrize("step", [0.4, 0.06])
def test_score_levels_long_items_planned(step):
    # 8 sequences x 160 blocks (a 96-block prefix): the planned path with
    # many-block items and the separate split merge over dozens of splits
    table, _ = shared_tables(8, 96, [64, 50, 64, 7, 33, 64, 20, 1])
    seq_len = (np.array([160, 146, 160, 103, 129, 160, 116, 97]) * 16).astype(np.int32)
    run(table, seq_len, 4, 4, 128, step, seed=77, path="auto")
