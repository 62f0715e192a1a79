"""Algorithmic byte and flop counts for MLA attention over an FP8 latent cache.

These are the roofline numerators: bytes every launch must move at least once and the
multiply-adds the definition needs, independent of how a kernel tiles the work.

* A cached position is 576 e4m3 bytes ("Scaling Kimi K3 on AMD Instinct MI355X", section
  "缓存可复用，还要能一致地恢复": 24 MLA layers x 142,000 positions x 576 bytes is about
  1.96 GB per GPU, about 245 MB once position-sharded eight ways).
* Per visible (query row, key) pair the contraction is 576 multiply-adds for the score
  and 512 for the value, i.e. 2 * (576 + 512) flops.
"""
from __future__ import annotations

D = 576
DV = 512
FLOPS_PER_PAIR = 2 * (D + DV)


def kv_cache_bytes(positions: int, layers: int = 1, shards: int = 1) -> float:
    """Latent cache bytes for `positions` cached tokens over `layers` layers, divided
    evenly across `shards` position shards."""
    return positions * layers * D / shards


def decode_bytes(seq_lens, n_q: int, H: int, page_size: int = 64) -> int:
    """Bytes a decode/verify call must move: every cached row once, the queries (bf16),
    the outputs (bf16), the LSE (fp32), the lengths and the page-table entries read."""
    lens = [int(x) for x in seq_lens]
    rows = len(lens) * n_q * H
    pages = sum((L + page_size - 1) // page_size for L in lens)
    return sum(lens) * D + rows * (D * 2 + DV * 2 + 4) + 4 * len(lens) + 4 * pages


def visible_pairs(seq_lens, n_q: int, H: int) -> int:
    """Number of (query row, visible key) pairs: query j of sequence b sees
    L_b - n_q + j + 1 keys."""
    total = 0
    for L in seq_lens:
        L = int(L)
        for j in range(n_q):
            total += max(0, L - n_q + j + 1)
    return total * H


def attention_flops(seq_lens, n_q: int, H: int) -> int:
    return visible_pairs(seq_lens, n_q, H) * FLOPS_PER_PAIR


def prefill_bytes(T: int, H: int, L: int) -> int:
    """Queries + cache rows + outputs + LSE of one causal prefill chunk."""
    return T * H * D * 2 + L * D + T * H * DV * 2 + T * H * 4


# MHA (non-absorbed) form: per head, keys of 128 up-projected + 64 RoPE dims, values of 128
# ("MI355X Kimi K2.5 vLLM AITER 7x speedup", section "PR #35850 修复了什么": K and V share
# one latent, which the MHA form expands per head).
MHA_QK = 192
MHA_V = 128
MHA_FLOPS_PER_PAIR = 2 * (MHA_QK + MHA_V)


def mha_attention_flops(T: int, L: int, H: int) -> int:
    """Score and value flops of the MHA-form causal prefill: T new positions, the last T
    of L cached, H heads."""
    return visible_pairs([L], T, H) * MHA_FLOPS_PER_PAIR


def mha_projection_flops(L: int, H: int) -> int:
    """The up-projection of L cached latent rows (512 wide) to H heads x (128 + 128)."""
    return 2 * L * DV * H * (128 + MHA_V)
