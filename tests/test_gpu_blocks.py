"""GPU block lifetime (kvs_blocks_init_free, kvs_block_write, kvs_seq_release)
vs the sequential oracle: tables, reference counts, the free stack and the
copied block contents bit-exact after every operation of random sequences."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from shared_paged_kv_gb300 import kvs as K
from oracle import blocks as OB, fingerprint as OF
from shared_paged_kv_gb300 import workloads as W
import harness as H


class GpuBlocks:
    """Device state mirrored from a table / seq_len / refcount triple."""

    def __init__(self, pool, table, seq_len, ref):
        self.pool = pool
        self.cap = pool.desc.capacity_blocks
        self.table = H.i32(table)
        self.seq_len = H.i32(seq_len)
        self.ref = H.i32(ref)
        self.free = torch.zeros(self.cap, dtype=torch.int32, device=H.DEV)
        self.n_free = torch.zeros(1, dtype=torch.int32, device=H.DEV)
        n_items = max(table.shape[0], 64)
        self.ws = H.workspace(K.kvs_workspace_size(pool, K.KVS_OP_BLOCKS, n_items, 0))
        self.n_seq, self.max_blocks = table.shape
        K.kvs_blocks_init_free(pool, self.ref, self.free, self.n_free, self.ws)

    def write(self, seqs, blocks):
        K.kvs_block_write(self.pool, self.table, self.max_blocks, self.n_seq, H.i32(seqs), H.i32(blocks), len(seqs),
                          self.ref, self.free, self.n_free, self.ws)

    def release(self, seqs):
        K.kvs_seq_release(self.pool, self.table, self.max_blocks, self.seq_len, self.n_seq, H.i32(seqs), len(seqs),
                          self.ref, self.free, self.n_free, self.ws)

    def compare(self, m):
        torch.cuda.synchronize()
        assert np.array_equal(self.table.cpu().numpy(), m.table)
        assert np.array_equal(self.ref.cpu().numpy(), m.ref.astype(np.int32))
        n = int(self.n_free.item())
        assert n == len(m.free)
        assert self.free[:n].cpu().numpy().tolist() == m.free


def _random_tables(rng, n_seq=6, B=16, shared=3):
    seq_len = rng.integers(1, 6 * B, size=n_seq).astype(np.int32)
    max_blocks = int(-(-seq_len.max() // B))
    table = np.full((n_seq, max_blocks), -1, np.int32)
    nxt = shared
    for a in range(n_seq):
        for b in range(int(-(-seq_len[a] // B))):
            if b < shared and (b + 1) * B <= seq_len[a]:
                table[a, b] = b
            else:
                table[a, b] = nxt
                nxt += 1
    ref = np.bincount(table[table >= 0], minlength=40).astype(np.int32)
    return table, seq_len, ref


def _bf16_pool(rng, cap, layers=2, hkv=2, d=64):
    ks = [torch.from_numpy(rng.integers(0, 65535, size=(cap, hkv, 16, d), dtype=np.uint16).view(np.int16)).to(H.DEV)
          for _ in range(layers)]
    vs = [torch.from_numpy(rng.integers(0, 65535, size=(cap, hkv, 16, d), dtype=np.uint16).view(np.int16)).to(H.DEV)
          for _ in range(layers)]
    pool = K.kvs_pool_create(layers, hkv, d, 16, K.KVS_DTYPE_BF16, cap, 64, ks, vs)
    return pool, ks, vs


def test_random_operation_sequences_match_the_oracle():
    for seed in range(12):
        rng = np.random.default_rng(seed)
        table, seq_len, ref = _random_tables(rng)
        cap = len(ref)
        pool, ks, vs = _bf16_pool(rng, cap)
        host = [t.cpu().numpy() for t in ks + vs]
        m = OB.BlockManager(table, seq_len, ref, 16, host)
        g = GpuBlocks(pool, table, seq_len, ref)
        g.compare(m)
        alive = list(range(table.shape[0]))
        for _ in range(10):
            if rng.random() < 0.7 and alive:
                k = int(rng.integers(1, 6))
                seqs = rng.choice(alive, size=k).astype(np.int32)
                blocks = np.array([int(rng.integers(0, m.n_blocks(a))) for a in seqs], np.int32)
                m.write_batch(seqs, blocks)
                g.write(seqs, blocks)
            elif alive:
                out = [alive.pop(int(rng.integers(0, len(alive))))]
                m.release(out)
                g.release(np.array(out, np.int32))
            g.compare(m)
            for s_dev, s_host in zip(ks + vs, m.slabs):
                assert np.array_equal(s_dev.cpu().numpy(), s_host)
        m.release(alive)
        g.release(np.array(alive, np.int32))
        g.compare(m)
        assert int(g.n_free.item()) == cap and not m.errors
        assert K.kvs_pool_check(pool) == 0


def test_duplicate_writes_in_one_batch_and_duplicate_release():
    rng = np.random.default_rng(7)
    table = np.array([[0, 3], [0, 4], [0, 5]], np.int32)
    seq_len = np.array([32, 32, 32], np.int32)
    ref = np.bincount(table.reshape(-1), minlength=9).astype(np.int32)
    pool, ks, vs = _bf16_pool(rng, 9, layers=1)
    m = OB.BlockManager(table, seq_len, ref, 16, [t.cpu().numpy() for t in ks + vs])
    g = GpuBlocks(pool, table, seq_len, ref)
    seqs = np.array([1, 1, 2, 0, 2], np.int32)
    blocks = np.array([0, 0, 0, 0, 1], np.int32)
    m.write_batch(seqs, blocks)
    g.write(seqs, blocks)
    g.compare(m)
    m.release([2, 2])
    g.release(np.array([2, 2], np.int32))
    g.compare(m)
    assert K.kvs_pool_check(pool) == 0


def test_q4_pool_copies_codes_and_scale_bias():
    rng = np.random.default_rng(8)
    cap, hkv = 6, 2
    codes = [torch.from_numpy(rng.integers(0, 255, size=(cap, hkv, 256, 64), dtype=np.uint8)).to(H.DEV) for _ in range(2)]
    sbs = [torch.from_numpy(rng.standard_normal((cap, hkv, 256, 4)).astype(np.float16)).to(H.DEV) for _ in range(2)]
    pool = K.kvs_pool_create(1, hkv, 128, 256, K.KVS_DTYPE_Q4G64, cap, 4, [codes[0]], [codes[1]], [sbs[0]], [sbs[1]])
    table = np.array([[0], [0]], np.int32)
    g = GpuBlocks(pool, table, np.array([256, 256], np.int32), np.array([2, 0, 0, 0, 0, 0], np.int32))
    g.write(np.array([0], np.int32), np.array([0], np.int32))
    torch.cuda.synchronize()
    new = int(g.table[0, 0].item())
    assert new == 1
    for t in codes + sbs:
        assert torch.equal(t[new], t[0])
    assert K.kvs_pool_check(pool) == 0


def test_empty_stack_and_overrelease_are_flagged():
    rng = np.random.default_rng(9)
    pool, ks, vs = _bf16_pool(rng, 2, layers=1)
    table = np.array([[0], [0]], np.int32)
    g = GpuBlocks(pool, table, np.array([16, 16], np.int32), np.array([2, 1], np.int32))   # block 1 in use elsewhere
    g.write(np.array([0], np.int32), np.array([0], np.int32))
    torch.cuda.synchronize()
    assert g.table.cpu().numpy().tolist() == [[0], [0]]
    assert K.kvs_pool_check(pool) & K.KVS_DEVERR_CAPACITY
    bad = GpuBlocks(pool, table, np.array([16, 16], np.int32), np.array([1, 0], np.int32))
    bad.release(np.array([0, 1], np.int32))
    assert K.kvs_pool_check(pool) & K.KVS_DEVERR_REFCOUNT


def test_full_size_mha7b_copy_burst_and_release():
    """The 7B-MHA tables from GPU dedup (614 shared + 8 x 410 private blocks,
    32 layers of 32 heads): every agent writes into the last shared block (7
    copies of 4 MiB each), then every agent is released."""
    w = W.make_mha7b(n_layers=1)
    ref_o = OF.dedup(w.tokens, w.seq_off, w.tier, w.block_tokens, w.max_blocks)
    cap = ref_o["n_phys"] + 16
    layers, hkv, d = 32, 32, 128
    ks = [torch.zeros((cap, hkv, 16, d), dtype=torch.int16, device=H.DEV) for _ in range(layers)]
    vs = [torch.zeros_like(ks[0]) for _ in range(layers)]
    gen = torch.Generator(device=H.DEV).manual_seed(3)
    for t in ks + vs:
        t[613].copy_(torch.randint(-30000, 30000, (hkv, 16, d), generator=gen, device=H.DEV, dtype=torch.int16))
    pool = K.kvs_pool_create(layers, hkv, d, 16, K.KVS_DTYPE_BF16, cap, w.n_seq, ks, vs)
    refc = np.zeros(cap, np.int32)
    refc[:ref_o["n_phys"]] = ref_o["refcount"]
    m = OB.BlockManager(ref_o["block_table"], w.seq_len, refc, 16)
    g = GpuBlocks(pool, ref_o["block_table"], w.seq_len, refc)
    seqs = np.arange(w.n_seq, dtype=np.int32)
    blocks = np.full(w.n_seq, 613, np.int32)
    m.write_batch(seqs, blocks)
    g.write(seqs, blocks)
    g.compare(m)
    for a in range(w.n_seq - 1):
        new = int(m.table[a, 613])
        for t in (ks[0], vs[17], ks[31]):
            assert torch.equal(t[new], t[613])
    m.release(seqs)
    g.release(seqs)
    g.compare(m)
    assert int(g.n_free.item()) == cap and K.kvs_pool_check(pool) == 0
