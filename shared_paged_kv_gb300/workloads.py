"""Seeded synthetic workloads for the shared paged KV hot path.

This module only draws random inputs and lays them out; it performs none of
the method's arithmetic (no hashing, no deduplication, no rotation, no
quantisation, no attention).  It is the one module that both the CUDA path
(bench, GPU tests) and the CPU oracle (tests) take their inputs from.

Workload shapes follow the five synthetic configurations of the build:

* ``tiny``       4 agents, Hq 8 / Hkv 2, d 64, block 16; a 256-token shared
                 prefix plus 64..128 private tokens each; 2 mirror-diff blocks
                 per agent with diffs ~N(0, 0.1).
* ``mha7b``      8 agents x 16384 tokens, Hq = Hkv = 32, d 128, block 16;
                 614 shared prefix blocks (60 % of 1024) + 410 private blocks.
* ``gqa_fanout`` 32 sequences, Hq 16 / Hkv 2, d 128; a 4096-token system
                 prefix + 512..2048 private tokens each.
* ``allgather``  64 agents, Hq 40 / Hkv 8, d 128, theta 1e6; private history
                 of 16*U{64..384} tokens followed by 64 shared 128-token
                 segments in a per-agent random order; 31 diff blocks per
                 agent among its 512 segment blocks.
* ``q4``         12 agents x 8192 tokens, Hq 32 / Hkv 8, d 128, 256-token
                 blocks; values ~N(0, 1) before 4-bit quantisation.

Every ``make_*`` function takes scale-down knobs so the tests can run the same
structure at sizes the CPU oracle finishes in seconds.

bf16 values are produced from float32 samples by round-to-nearest-even and are
carried as ``uint16`` bit patterns.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

PRIVATE_TIER = 0xFFFFFFFF


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((u >> 16) & 1) + np.uint32(0x7FFF)
    out = ((u + rounding) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass
class Workload:
    name: str
    n_seq: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    block_tokens: int
    n_layers: int
    theta: float
    # token ids of every sequence, concatenated; seq_off is the CSR offset
    tokens: np.ndarray            # uint32 [total_tokens]
    seq_off: np.ndarray           # int64  [n_seq + 1]
    tier: np.ndarray              # uint32 [n_seq]
    max_blocks: int               # block-table row length
    capacity_blocks: int          # physical blocks per layer slab (upper bound)
    # segment-based hashing boundaries (block indices where a hashed segment
    # starts; block 0 always starts one).  None = plain prefix hashing.
    seg_start_off: Optional[np.ndarray] = None     # int64 [n_seq + 1]
    seg_start_blocks: Optional[np.ndarray] = None  # int32 [n_starts]
    # query-side RoPE shifts per agent: CSR over (first_block, n_blocks, delta)
    rope_off: Optional[np.ndarray] = None          # int32 [n_seq + 1]
    rope_segs: Optional[np.ndarray] = None         # int32 [n_segs, 4]
    # mirror diffs: diff_table[a, b] = diff block id or -1
    diff_table: Optional[np.ndarray] = None        # int32 [n_seq, max_blocks * block_tokens / diff_block_tokens]
    diff_capacity_blocks: int = 0
    seed: int = 0
    # tokens per mirror-diff block (0: the pool's block size; Q4 pools keep
    # their diffs per 16-token sub-block of a 256-token block)
    diff_block_tokens: int = 0

    @property
    def seq_len(self) -> np.ndarray:
        return np.diff(self.seq_off).astype(np.int32)

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def scale(self) -> float:
        return float(1.0 / np.sqrt(self.head_dim))

    # ---- per-layer values -------------------------------------------------
    def _rng(self, layer: int, what: int) -> np.random.Generator:
        return np.random.default_rng([self.seed, 1000 + layer, what])

    def kv_layer(self, layer: int):
        """bf16 bits of the K and V slabs of one layer: [cap][Hkv][B][d]."""
        shape = (self.capacity_blocks, self.n_kv_heads, self.block_tokens, self.head_dim)
        k = self._rng(layer, 1).standard_normal(shape, dtype=np.float32)
        v = self._rng(layer, 2).standard_normal(shape, dtype=np.float32)
        return f32_to_bf16_bits(k), f32_to_bf16_bits(v)

    def diff_layer(self, layer: int, sigma: float = 0.1):
        """bf16 bits of the mirror-diff K and V slabs: [diff_cap][Hkv][B][d]."""
        shape = (max(self.diff_capacity_blocks, 0), self.n_kv_heads, self.diff_block_tokens or self.block_tokens,
                 self.head_dim)
        dk = self._rng(layer, 3).standard_normal(shape, dtype=np.float32) * np.float32(sigma)
        dv = self._rng(layer, 4).standard_normal(shape, dtype=np.float32) * np.float32(sigma)
        return f32_to_bf16_bits(dk), f32_to_bf16_bits(dv)

    def q_layer(self, layer: int):
        """bf16 bits of the decode queries: [n_seq][Hq][d]."""
        shape = (self.n_seq, self.n_q_heads, self.head_dim)
        return f32_to_bf16_bits(self._rng(layer, 5).standard_normal(shape, dtype=np.float32))


def _csr(lists):
    off = np.zeros(len(lists) + 1, dtype=np.int64)
    for i, l in enumerate(lists):
        off[i + 1] = off[i] + len(l)
    flat = np.concatenate([np.asarray(l) for l in lists]) if lists else np.zeros(0)
    return off, flat


def make_tiny(seed: int = 0) -> Workload:
    """4 agents; 256-token shared prefix (ids U[0,32000), seed 0) + 64..128
    private tokens; 2 diff blocks per agent among its 16 shared blocks."""
    B, n = 16, 4
    rng = np.random.default_rng(seed)
    prefix = rng.integers(0, 32000, size=256, dtype=np.uint32)
    seqs, diff_rows = [], []
    for a in range(n):
        priv_len = int(rng.integers(64, 129))
        seqs.append(np.concatenate([prefix, rng.integers(0, 32000, size=priv_len, dtype=np.uint32)]))
    off, toks = _csr(seqs)
    lens = np.diff(off)
    max_blocks = int(-(-lens.max() // B))
    cap = int(sum(-(-l // B) for l in lens))
    diff_table = np.full((n, max_blocks), -1, dtype=np.int32)
    nd = 0
    for a in range(n):
        for b in sorted(rng.choice(16, size=2, replace=False)):
            diff_table[a, b] = nd
            nd += 1
    return Workload("tiny", n, 8, 2, 64, B, 1, 1e4, toks.astype(np.uint32), off,
                    np.zeros(n, np.uint32), max_blocks, cap, diff_table=diff_table,
                    diff_capacity_blocks=nd, seed=seed)


def make_prefix_shared(name: str, n_seq: int, hq: int, hkv: int, d: int, n_layers: int,
                       shared_tokens: int, private_lens, seed: int, block: int = 16) -> Workload:
    """n_seq sequences = one common prefix of shared_tokens ids + private ids."""
    rng = np.random.default_rng(seed)
    prefix = rng.integers(0, 32000, size=shared_tokens, dtype=np.uint32)
    seqs = [np.concatenate([prefix, rng.integers(0, 32000, size=int(pl), dtype=np.uint32)])
            for pl in private_lens]
    off, toks = _csr(seqs)
    lens = np.diff(off)
    max_blocks = int(-(-lens.max() // block))
    cap = int(-(-shared_tokens // block) + sum(-(-int(l) // block) for l in lens))
    return Workload(name, n_seq, hq, hkv, d, block, n_layers, 1e4, toks.astype(np.uint32), off,
                    np.zeros(n_seq, np.uint32), max_blocks, cap, seed=seed)


def make_mha7b(seed: int = 2, n_seq: int = 8, total_blocks: int = 1024, shared_blocks: int = 614,
               n_layers: int = 32, heads: int = 32, d: int = 128) -> Workload:
    """8 agents x 16384 tokens, 32 = 32 heads, d 128, 60 % shared prefix."""
    B = 16
    priv = [(total_blocks - shared_blocks) * B] * n_seq
    return make_prefix_shared("mha7b", n_seq, heads, heads, d, n_layers, shared_blocks * B, priv, seed)


def make_gqa_fanout(seed: int = 3, n_seq: int = 32, prefix_tokens: int = 4096,
                    priv_lo: int = 512, priv_hi: int = 2048, n_layers: int = 28,
                    hq: int = 16, hkv: int = 2, d: int = 128) -> Workload:
    """32 sequences sharing a 4096-token prefix + U{512..2048} private tokens."""
    rng = np.random.default_rng([seed, 7])
    priv = rng.integers(priv_lo, priv_hi + 1, size=n_seq)
    return make_prefix_shared("gqa_fanout", n_seq, hq, hkv, d, n_layers, prefix_tokens, priv, seed)


def make_allgather(seed: int = 4, n_seq: int = 64, n_segs: int = 64, seg_tokens: int = 128,
                   priv_blocks_lo: int = 64, priv_blocks_hi: int = 384, diff_frac: float = 0.06,
                   n_layers: int = 48, hq: int = 40, hkv: int = 8, d: int = 128,
                   theta: float = 1e6) -> Workload:
    """All-gather round: private history then n_segs shared segments in a
    per-agent random order.  Master segment j is taken to sit at source
    position seg_tokens*j; in agent a it sits at P_a + seg_tokens*pi_a(j)."""
    B = 16
    assert seg_tokens % B == 0
    rng = np.random.default_rng(seed)
    seg_ids = [rng.integers(0, 32000, size=seg_tokens, dtype=np.uint32) for _ in range(n_segs)]
    seqs, starts, rope = [], [], []
    blocks_per_seg = seg_tokens // B
    n_diff_per_agent = int(round(diff_frac * n_segs * blocks_per_seg))
    for a in range(n_seq):
        p_a = B * int(rng.integers(priv_blocks_lo, priv_blocks_hi + 1))
        order = rng.permutation(n_segs)          # order[k] = segment placed in slot k
        parts = [rng.integers(0, 32000, size=p_a, dtype=np.uint32)]
        st = [0]
        rr = []
        for slot, j in enumerate(order):
            parts.append(seg_ids[j])
            first_block = (p_a + seg_tokens * slot) // B
            st.append(first_block)
            dst_pos = p_a + seg_tokens * slot
            src_pos = seg_tokens * int(j)
            rr.append((first_block, blocks_per_seg, dst_pos - src_pos, 0))
        seqs.append(np.concatenate(parts))
        starts.append(st)
        rope.append(rr)
    off, toks = _csr(seqs)
    lens = np.diff(off)
    max_blocks = int(-(-lens.max() // B))
    cap = int(sum(-(-int(l) // B) for l in lens))
    s_off, s_flat = _csr(starts)
    r_off, _ = _csr(rope)
    r_flat = np.array([x for rr in rope for x in rr], dtype=np.int32).reshape(-1, 4)
    diff_table = np.full((n_seq, max_blocks), -1, dtype=np.int32)
    nd = 0
    for a in range(n_seq):
        p_blocks = int(lens[a] // B) - n_segs * blocks_per_seg
        seg_blocks = np.arange(p_blocks, p_blocks + n_segs * blocks_per_seg)
        for b in np.sort(rng.choice(seg_blocks, size=n_diff_per_agent, replace=False)):
            diff_table[a, b] = nd
            nd += 1
    return Workload("allgather", n_seq, hq, hkv, d, B, n_layers, theta, toks.astype(np.uint32), off,
                    np.zeros(n_seq, np.uint32), max_blocks, cap,
                    seg_start_off=s_off, seg_start_blocks=s_flat.astype(np.int32),
                    rope_off=r_off.astype(np.int32), rope_segs=r_flat,
                    diff_table=diff_table, diff_capacity_blocks=nd, seed=seed)


def make_q4(seed: int = 5, n_seq: int = 12, ctx: int = 8192, n_layers: int = 32,
            hq: int = 32, hkv: int = 8, d: int = 128, block: int = 256, diff_frac: float = 0.0,
            diff_block: int = 16) -> Workload:
    """12 agents x 8192 tokens, no sharing, 256-token blocks (Q4 pool).  With
    diff_frac > 0, each agent gets round(diff_frac * its diff_block-token
    sub-blocks) mirror-diff sub-blocks, chosen uniformly (the all-gather
    round's 31 of 512 at 6 %), with diffs ~N(0, 0.1)."""
    rng = np.random.default_rng(seed)
    seqs = [rng.integers(0, 32000, size=ctx, dtype=np.uint32) for _ in range(n_seq)]
    off, toks = _csr(seqs)
    lens = np.diff(off)
    max_blocks = int(-(-lens.max() // block))
    cap = int(sum(-(-int(l) // block) for l in lens))
    diff_table, nd = None, 0
    if diff_frac > 0:
        per = block // diff_block
        diff_table = np.full((n_seq, max_blocks * per), -1, dtype=np.int32)
        for a in range(n_seq):
            n_sub = -(-int(lens[a]) // diff_block)
            for sb in np.sort(rng.choice(n_sub, size=int(round(diff_frac * n_sub)), replace=False)):
                diff_table[a, sb] = nd
                nd += 1
    return Workload("q4_mirror" if diff_frac > 0 else "q4", n_seq, hq, hkv, d, block, n_layers, 1e4,
                    toks.astype(np.uint32), off, np.full(n_seq, PRIVATE_TIER, np.uint32), max_blocks, cap,
                    diff_table=diff_table, diff_capacity_blocks=nd, seed=seed,
                    diff_block_tokens=diff_block if diff_frac > 0 else 0)


def make_q4_mirror(**kw) -> Workload:
    """The Q4 configuration with mirror diffs on 6 % of every agent's 16-token
    sub-blocks (31 of 512)."""
    kw.setdefault("diff_frac", 0.06)
    return make_q4(**kw)


def selection_inputs(seed: int, n_agents: int, rows_per_agent, row_elems: int,
                     sigma_lo: float = 0.05, sigma_hi: float = 0.5):
    """K_cached ~N(0,1) and K_new = K_cached + N(0, sigma_t^2) per position,
    sigma_t ~ U(sigma_lo, sigma_hi); both as bf16 bits [rows][row_elems]."""
    rng = np.random.default_rng([seed, 99])
    rows = np.asarray(rows_per_agent, dtype=np.int64)
    off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int64)
    total = int(off[-1])
    kc = rng.standard_normal((total, row_elems), dtype=np.float32)
    sig = rng.uniform(sigma_lo, sigma_hi, size=(total, 1)).astype(np.float32)
    kn = kc + rng.standard_normal((total, row_elems), dtype=np.float32) * sig
    return f32_to_bf16_bits(kc), f32_to_bf16_bits(kn), off


def rope_jobs_for(w: Workload, first_free_block: int, src_row: int = 0):
    """Re-rotation jobs that materialise every shared segment of every agent
    from the master copy into fresh private blocks at the agent's positions.

    The master of segment j is its occurrence in block-table row ``src_row``
    (whose segment positions are read from ``w.rope_segs``).  Destination
    blocks are numbered from ``first_free_block`` upward.  Returns
    ``(jobs, dst_table, n_dst_blocks)``: jobs are int32 rows (src_row,
    src_tok0, dst_row, dst_tok0, n_tok, src_pos, dst_pos, 0) and dst_table is
    int32 [n_seq][max_blocks] with -1 outside the segments."""
    assert w.rope_segs is not None
    B = w.block_tokens
    r_off = w.rope_off
    by_src = {}
    for (fb, nb, delta, _) in w.rope_segs[r_off[src_row]:r_off[src_row + 1]]:
        by_src[fb * B - delta] = fb * B     # master position -> token offset in row src_row
    jobs = []
    dst_table = np.full((w.n_seq, w.max_blocks), -1, dtype=np.int32)
    nxt = first_free_block
    for a in range(w.n_seq):
        for (fb, nb, delta, _) in w.rope_segs[r_off[a]:r_off[a + 1]]:
            dst_pos = fb * B
            src_pos = dst_pos - delta
            dst_table[a, fb:fb + nb] = np.arange(nxt, nxt + nb, dtype=np.int32)
            nxt += nb
            jobs.append((src_row, by_src[src_pos], a, dst_pos, nb * B, src_pos, dst_pos, 0))
    return np.array(jobs, dtype=np.int32).reshape(-1, 8), dst_table, nxt - first_free_block
