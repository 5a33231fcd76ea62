"""GPU block-granular MemDecay eviction scoring vs the fp64 oracle: block
scores within float32 rounding, victim sets exact except for blocks whose
scores tie (within 1e-5 relative) with the k-th lowest, victims ascending."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from shared_paged_kv_gb300 import kvs as K
from oracle import evict as OE
import harness as H

INIT = [100.0, 10.0, 5.0, 2.0, 1.0]          # the post's suggested initial scores (§5.2)
DECAY = [0.0, 0.0092, 0.02, 0.05, 0.1]


def memdecay_inputs(rng, n_seq, max_blocks, B=16, lo=None):
    """Token metadata with the post's region layout: a system prompt at the
    start, scattered key decisions and tool summaries, a recent-dialogue tail,
    ordinary context elsewhere; created = position, access counts ~ Poisson."""
    T = max_blocks * B
    lo = lo if lo is not None else B
    seq_len = rng.integers(lo, T + 1, size=n_seq).astype(np.int32)
    region = np.full((n_seq, T), 4, np.uint8)
    for a in range(n_seq):
        L = int(seq_len[a])
        region[a, :min(L, 64)] = 0
        region[a, rng.random(T) < 0.03] = 1
        region[a, rng.random(T) < 0.05] = 2
        region[a, max(0, L - 256):L] = 3
    created = np.tile(np.arange(T, dtype=np.int32), (n_seq, 1))
    access = rng.poisson(1.5, size=(n_seq, T)).astype(np.int32)
    return seq_len, region, created, access


def run(region, created, access, seq_len, max_blocks, k, step, B=16):
    n_seq = len(seq_len)
    d16 = torch.zeros(16, dtype=torch.int16, device=H.DEV)
    pool = K.kvs_pool_create(1, 1, 64, B, K.KVS_DTYPE_BF16, 1, 1, [d16], [d16])
    scores = torch.zeros((n_seq, max_blocks), dtype=torch.float32, device=H.DEV)
    victims = torch.full((max(1, int(sum(k))),), -7, dtype=torch.int32, device=H.DEV)
    voff = torch.zeros(n_seq + 1, dtype=torch.int64, device=H.DEV)
    K.kvs_evict_score(pool, torch.from_numpy(region).to(H.DEV), H.i32(created), H.i32(access), H.i32(seq_len),
                      n_seq, max_blocks, INIT, DECAY, step, H.i32(k), scores, victims, voff)
    torch.cuda.synchronize()
    return pool, scores.cpu().numpy(), victims.cpu().numpy(), voff.cpu().numpy()


def check(region, created, access, seq_len, max_blocks, k, step, B=16):
    pool, gs, gv, goff = run(region, created, access, seq_len, max_blocks, k, step, B)
    es = OE.block_scores(region, created, access, seq_len, INIT, DECAY, step, B)
    fin = np.isfinite(es)
    assert np.array_equal(np.isfinite(gs), fin)
    assert (np.abs(gs[fin] - es[fin]) <= 1e-5 * np.abs(es[fin]) + 1e-30).all()
    ev, eoff = OE.victims(es, seq_len, k, B)
    assert np.array_equal(goff, eoff)
    for a in range(len(seq_len)):
        got = gv[goff[a]:goff[a + 1]].tolist()
        exp = ev[eoff[a]:eoff[a + 1]].tolist()
        assert got == sorted(got)
        if got == exp or not exp:
            continue
        # the sets may differ only inside the tie band around the k-th score
        sk = max(es[a, b] for b in exp)
        tol = 1e-5 * sk + 1e-30
        for b in set(got) - set(exp):
            assert es[a, b] <= sk + tol
        for b in set(exp) - set(got):
            assert es[a, b] >= sk - tol
    return pool


def test_small_random():
    rng = np.random.default_rng(0)
    for trial in range(5):
        seq_len, region, created, access = memdecay_inputs(rng, 5, 12)
        nb = -(-seq_len // 16)
        k = np.array([int(rng.integers(0, b + 1)) for b in nb], np.int32)
        pool = check(region, created, access, seq_len, 12, k, step=12 * 16 + 7)
        assert K.kvs_pool_check(pool) == 0


def test_k_beyond_blocks_and_zero():
    rng = np.random.default_rng(1)
    seq_len, region, created, access = memdecay_inputs(rng, 3, 6)
    k = np.array([0, 100, 2], np.int32)
    check(region, created, access, seq_len, 6, k, step=200)


def test_many_ties_from_underflow():
    """Old ordinary-context tokens decay to zero in float32: the ties at zero
    resolve to the lower block indices."""
    rng = np.random.default_rng(2)
    seq_len, region, created, access = memdecay_inputs(rng, 4, 40, lo=40 * 16)
    k = np.full(4, 25, np.int32)
    check(region, created, access, seq_len, 40, k, step=40 * 16 + 5000)


def test_full_size_64_agents_16k_tokens():
    rng = np.random.default_rng(3)
    seq_len, region, created, access = memdecay_inputs(rng, 64, 1024, lo=12000)
    nb = -(-seq_len // 16)
    k = (nb // 4).astype(np.int32)
    check(region, created, access, seq_len, 1024, k, step=16384 + 10)


def test_bad_region_is_flagged():
    rng = np.random.default_rng(4)
    seq_len, region, created, access = memdecay_inputs(rng, 2, 4)
    region[1, 0] = 9
    pool, *_ = run(region, created, access, seq_len, 4, np.array([1, 1], np.int32), step=100)
    assert K.kvs_pool_check(pool) & K.KVS_DEVERR_JOB
