"""KV-cache accounting, written out from the pages' closed forms.

* Per-token KV bytes = layers x 2 (K and V) x kv_heads x head_dim x dtype
  bytes — shared-memory KV pool post, §1.1 (worked case 28x2x2x128x2 = 28672 B).
  The INMS walkthrough §1.2 prices a 7B model the same way (2 x 4096 x 2 B per
  layer x 32 layers = 512 KiB per token).
* Independent vs shared footprint: n*L*s against ((1-p)*n + p)*L*s — INMS
  walkthrough §1.2 (and its §4.1 three-agent re-run).
* Break-even / duplicate bytes = prefix tokens x concurrency x bytes per token
  — shared-memory KV pool post §1.2 and §5.1.
* Q4 footprint ratio against fp16 for group-g codes with fp16 scale and bias —
  Q4 edge paper summary §2.1 (ratio 0.281).
"""
from __future__ import annotations


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, dtype_bytes: int) -> int:
    return layers * 2 * kv_heads * head_dim * dtype_bytes


def independent_bytes(n_agents: int, seq_len: int, bytes_per_token: float) -> float:
    return n_agents * seq_len * bytes_per_token


def shared_bytes(n_agents: int, seq_len: int, bytes_per_token: float, common_frac: float) -> float:
    return ((1.0 - common_frac) * n_agents + common_frac) * seq_len * bytes_per_token


def duplicate_prefix_bytes(prefix_tokens: int, copies: int, bytes_per_token: float) -> float:
    return prefix_tokens * copies * bytes_per_token


def q4_ratio(bits: int = 4, group: int = 64, scale_bits: int = 16, bias_bits: int = 16,
             ref_bits: int = 16) -> float:
    """Bits per element of a group-quantised code (code + amortised scale and
    bias) over the reference element width."""
    return (bits + (scale_bits + bias_bits) / group) / ref_bits


def block_granular_phys_blocks(n_agents: int, shared_blocks: int, private_blocks: int) -> int:
    """Physical blocks when a common prefix of shared_blocks full blocks is
    stored once and every agent keeps private_blocks of its own (the shared
    formula of INMS §1.2 at block granularity)."""
    return shared_blocks + n_agents * private_blocks
