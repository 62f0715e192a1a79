"""Seeded synthetic inputs for MLA attention over a paged FP8-e4m3 latent KV cache.

This module only draws inputs: it holds none of the attention arithmetic, and both
the CUDA path and the float64 oracle consume exactly what it returns.

Shapes follow the pages on MLA serving: every cached position is one row of 576
FP8 bytes (read here as a 512-wide latent followed by a 64-wide RoPE part), the
cache is paged, and query heads per rank are 8, 12 or 16
("Scaling Kimi K3 on AMD Instinct MI355X", sections "缓存可复用，还要能一致地恢复"
and "并行度必须适配真正的形状"; "MI355X Kimi K2.5 vLLM AITER 7x speedup",
section "PR #35850 修复了什么").

Recipe (fixed draw order, one CPU ``torch.Generator`` seeded per workload):
  1. sequence lengths (``seq_lens`` include the ``n_q`` new positions),
  2. a random permutation of physical pool pages (identity for a contiguous cache),
  3. queries ``q ~ N(0, 1)`` rounded to bfloat16, layout ``[B][n_q][H][576]``,
  4. latent rows ``x ~ N(0, 1)`` in float32, one per logical cache slot (whole pages,
     so slots past ``seq_lens[b]`` in a sequence's last page hold valid codes too),
     quantised with one per-tensor scale ``kv_scale = amax / 448`` as
     ``e4m3_rne(clamp(x * inv, -448, 448))``, ``inv = 1 / kv_scale`` and the product
     both rounded to binary32 (the cache-append kernel quantises new rows the same
     way). The clamp comes first because the product can round a hair above 448 and
     the float8 cast does not saturate.
``sm_scale`` is ``1 / sqrt(192)`` for every workload.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

D = 576  # bytes (= e4m3 codes) per cached position
DV = 512  # latent width; V is the first DV codes of a row
PAGE = 64  # positions per page
SM_SCALE = 1.0 / math.sqrt(192.0)


@dataclasses.dataclass
class MlaInputs:
    """One seeded workload, all tensors on the CPU.

    pool        uint8  [num_pages, page_size, 576]  e4m3 codes
    page_table  int32  [B, max_pages]               physical page per logical page, -1 unused
    seq_lens    int32  [B]                          cached positions per sequence (incl. n_q new)
    q           bfloat16 [B, n_q, H, 576]
    kv_scale    float  dequantised value = e4m3(code) * kv_scale
    sm_scale    float
    """

    name: str
    pool: torch.Tensor
    page_table: torch.Tensor
    seq_lens: torch.Tensor
    q: torch.Tensor
    kv_scale: float
    sm_scale: float
    page_size: int

    @property
    def B(self) -> int:
        return int(self.q.shape[0])

    @property
    def n_q(self) -> int:
        return int(self.q.shape[1])

    @property
    def H(self) -> int:
        return int(self.q.shape[2])

    def kv_bytes_touched(self) -> int:
        """Bytes of cache rows the attention must read once: sum of seq_lens * 576."""
        return int(self.seq_lens.to(torch.int64).sum().item()) * D


def quantize_e4m3(x: torch.Tensor, scale: float) -> torch.Tensor:
    """float32 -> e4m3fn codes (uint8): x * (1 / scale), the reciprocal and the product
    rounded to binary32, clamped to +-448, then rounded to nearest even."""
    inv = torch.tensor(1.0, dtype=torch.float32) / torch.tensor(scale, dtype=torch.float32)
    y = (x.float() * inv).clamp_(-448.0, 448.0)
    return y.to(torch.float8_e4m3fn).view(torch.uint8)


def _latent_codes(n_rows: int, g: torch.Generator, chunk: int = 1 << 16):
    """Draw n_rows x 576 N(0,1) values and quantise them with scale = amax / 448.

    Two passes over the same generator state keep peak host memory small: the
    first finds amax, the second replays the identical draws and quantises them.
    """
    state = g.get_state()
    amax = 0.0
    done = 0
    while done < n_rows:
        n = min(chunk, n_rows - done)
        x = torch.randn(n, D, generator=g, dtype=torch.float32)
        amax = max(amax, float(x.abs().max().item()))
        done += n
    g.set_state(state)
    scale = amax / 448.0
    codes = torch.empty(n_rows, D, dtype=torch.uint8)
    done = 0
    while done < n_rows:
        n = min(chunk, n_rows - done)
        x = torch.randn(n, D, generator=g, dtype=torch.float32)
        codes[done:done + n] = quantize_e4m3(x, scale)
        done += n
    return codes, float(scale)


def make_inputs(
    name: str,
    seq_lens: Sequence[int] | None = None,
    *,
    H: int,
    n_q: int = 1,
    B: Optional[int] = None,
    len_range: Optional[tuple[int, int]] = None,
    page_size: int = PAGE,
    contiguous: bool = False,
    seed: int = 0,
    sm_scale: float = SM_SCALE,
) -> MlaInputs:
    """Build one workload. Either ``seq_lens`` or (``B``, ``len_range``) is given;
    ``len_range`` draws lengths uniformly from the closed interval."""
    g = torch.Generator().manual_seed(seed)
    # 1. lengths
    if seq_lens is None:
        assert B is not None and len_range is not None
        lo, hi = len_range
        lens = torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64)
    else:
        lens = torch.tensor(list(seq_lens), dtype=torch.int64)
    B = int(lens.numel())
    pages_per_seq = [(int(L) + page_size - 1) // page_size for L in lens.tolist()]
    total_pages = sum(pages_per_seq)
    max_pages = max(1, max(pages_per_seq) if pages_per_seq else 1)
    # 2. physical page permutation
    if contiguous:
        perm = torch.arange(total_pages, dtype=torch.int64)
    else:
        perm = torch.randperm(total_pages, generator=g)
    page_table = torch.full((B, max_pages), -1, dtype=torch.int32)
    logical = 0
    for b, np_ in enumerate(pages_per_seq):
        page_table[b, :np_] = perm[logical:logical + np_].to(torch.int32)
        logical += np_
    # 3. queries
    q = torch.randn(B, n_q, H, D, generator=g, dtype=torch.float32).to(torch.bfloat16)
    # 4. latent rows in logical order, then scattered into the pool
    codes, kv_scale = _latent_codes(total_pages * page_size, g)
    codes = codes.view(total_pages, page_size, D)
    pool = torch.empty_like(codes)
    pool[perm] = codes
    return MlaInputs(
        name=name,
        pool=pool,
        page_table=page_table,
        seq_lens=lens.to(torch.int32),
        q=q,
        kv_scale=kv_scale,
        sm_scale=float(sm_scale),
        page_size=page_size,
    )


# --- the five named workloads ---------------------------------------------------

def tiny_decode(seed: int = 0) -> MlaInputs:
    """Batch 1, 12 heads, 1 query, 1024 cached positions, contiguous cache."""
    return make_inputs("tiny_decode_b1_h12_l1024", [1024], H=12, n_q=1, contiguous=True, seed=seed)


def batched_paged_decode(seed: int = 0) -> MlaInputs:
    """Batch 32, 12 heads, 1 query, lengths uniform in [4096, 16384], random pages."""
    return make_inputs("batched_paged_decode_b32_h12_l4k-16k", None, H=12, n_q=1, B=32,
                       len_range=(4096, 16384), seed=seed)


def long_history_decode(H: int = 12, seed: int = 0) -> MlaInputs:
    """Batch 1, one query, 142,000 cached positions, H in {8, 12, 16}."""
    return make_inputs(f"long_history_decode_b1_h{H}_l142000", [142000], H=H, n_q=1, seed=seed)


def spec_verify(seed: int = 0) -> MlaInputs:
    """Batch 8, 12 heads, 4 verify positions on a 32,768 prefix (32,772 cached)."""
    return make_inputs("spec_verify_b8_h12_q4_l32772", [32768 + 4] * 8, H=12, n_q=4, seed=seed)


def causal_prefill(T: int = 8192, prefix: int = 32768, H: int = 12, seed: int = 0) -> MlaInputs:
    """One sequence: a T-token chunk on a `prefix`-token cached history, causal."""
    return make_inputs(f"causal_prefill_t{T}_p{prefix}_h{H}", [prefix + T], H=H, n_q=T, seed=seed)


@dataclasses.dataclass
class MhaInputs:
    """One MHA-form (non-absorbed) prefill workload of one sequence, all on the CPU.

    cache   MlaInputs with B = 1 and n_q = T: the paged latent cache (its absorbed q is
            not used by the MHA form)
    q       bfloat16 [T][H][192]   per head: 128 no-RoPE dims, then the 64 RoPE dims
    w_ukv   bfloat16 [512][H][256] per head: W_UK (columns 0..127) then W_UV (128..255);
            key h of position n = [latent_n @ W_UK_h ; rope_n], value = latent_n @ W_UV_h
    """

    cache: MlaInputs
    q: torch.Tensor
    w_ukv: torch.Tensor

    @property
    def T(self) -> int:
        return int(self.q.shape[0])

    @property
    def H(self) -> int:
        return int(self.q.shape[1])


QK_NOPE = 128  # up-projected key dims per head
QK_ROPE = 64   # RoPE dims (shared by the heads)
V_HEAD = 128   # up-projected value dims per head


def mha_prefill_inputs(T: int, prefix: int, H: int = 12, seed: int = 0,
                       page_size: int = PAGE) -> MhaInputs:
    """The cache as ``make_inputs`` draws it (one sequence of prefix + T positions), then,
    from a second generator seeded ``seed + 1``: q ~ N(0, 1) [T][H][192] and
    w_ukv ~ N(0, 1/512) [512][H][256] (so up-projected keys and values have unit variance
    like the RoPE part), each rounded to bfloat16. The pages give no weights; these are
    synthetic stand-ins."""
    cache = make_inputs(f"mha_prefill_t{T}_p{prefix}_h{H}", [prefix + T], H=H, n_q=T,
                        page_size=page_size, seed=seed)
    g = torch.Generator().manual_seed(seed + 1)
    q = torch.randn(T, H, QK_NOPE + QK_ROPE, generator=g).to(torch.bfloat16)
    w = (torch.randn(DV, H, QK_NOPE + V_HEAD, generator=g) / math.sqrt(DV)).to(torch.bfloat16)
    return MhaInputs(cache=cache, q=q, w_ukv=w)


def mha_prefill(T: int = 8192, prefix: int = 32768, H: int = 12, seed: int = 0) -> MhaInputs:
    """The causal prefill chunk of the named workload (T new positions on a prefix) in the
    MHA form."""
    return mha_prefill_inputs(T, prefix, H, seed)


# --- inputs with a wide dynamic range --------------------------------------------
#
# N(0, 1) queries and keys give scores that spread over about 1.7 nats, so almost every
# weight sits within a few binades of its row's largest one. The inputs below reach the
# cases that spread does not: one dominant key over a long, flat tail (an "attention
# sink"), weights that fall off over tens of nats, and query rows whose entries span many
# binades. They only set codes and query entries; the scores follow from the definition.

E4M3_CODE_448 = 0x7E  # +448, the largest finite e4m3 value
ROPE0 = DV            # first of the 64 RoPE dims (512..575)


def _set_rope_block(inp: MlaInputs, b: int, positions: torch.Tensor, k: torch.Tensor) -> None:
    """Rows `positions` of sequence b: RoPE dims 512 .. 512 + k - 1 hold +448, the rest of
    the 64 RoPE dims hold 0 (k per position, 0..64)."""
    pages = inp.page_table[b, (positions // inp.page_size).long()].long()
    offs = (positions % inp.page_size).long()
    dims = torch.arange(64)
    block = torch.where(dims[None, :] < k[:, None], E4M3_CODE_448, 0).to(torch.uint8)
    inp.pool[pages, offs, ROPE0:] = block


def _ramp_query(inp: MlaInputs, nats_per_dim, spread) -> None:
    """Queries whose score against a row with k RoPE dims at +448 (the rest 0) is
    k x nats_per_dim[h] plus a random part: RoPE dims = nats_per_dim[h] / (448 kv_scale
    sm_scale), dims 0..511 = spread[h] x (the N(0, 1) draw already there), rounded to bf16."""
    H = inp.H
    q = inp.q.float()
    for h in range(H):
        a = float(nats_per_dim[h]) / (448.0 * inp.kv_scale * inp.sm_scale)
        q[:, :, h, ROPE0:] = a
        q[:, :, h, :ROPE0] *= float(spread[h])
    inp.q = q.to(torch.bfloat16)


SINK_GAPS = (4.0, 6.0, 8.0, 10.0, 12.0, 16.0)


def attention_sink(L: int = 142000, H: int = 12, n_q: int = 1, B: int = 1, seed: int = 0,
                   sink_at: Optional[int] = None) -> MlaInputs:
    """One key per sequence (position `sink_at`, default L // 3, visible to every new
    position) stands about gap nats above a tail of L - 1 keys. Head h takes gap
    SINK_GAPS[h % 6]; even heads have an exactly flat tail (every other key scores 0),
    odd heads add the N(0, 1) query draw scaled by 1/2 on dims 0..511 (a tail spread of
    about 0.9 nats). Values (dims 0..511) stay the usual N(0, 1) latent."""
    inp = make_inputs(f"attention_sink_b{B}_h{H}_q{n_q}_l{L}", [L] * B, H=H, n_q=n_q, seed=seed)
    at = L // 3 if sink_at is None else sink_at
    pos = torch.arange(L)
    for b in range(B):
        _set_rope_block(inp, b, pos, torch.where(pos == at, 64, 0))
    gaps = [SINK_GAPS[h % len(SINK_GAPS)] / 64.0 for h in range(H)]
    _ramp_query(inp, gaps, [0.0 if h % 2 == 0 else 0.5 for h in range(H)])
    return inp


def graded_tail(L: int = 142000, H: int = 12, n_q: int = 1, nats: float = 30.0,
                seed: int = 0) -> MlaInputs:
    """Scores that fall off linearly over `nats` nats from the first key to the last, in
    65 equal steps (key n has round(64 (1 - n / L)) RoPE dims at +448); even heads have no
    other score component, odd heads add the N(0, 1) query draw scaled by 1/2."""
    inp = make_inputs(f"graded_tail_h{H}_q{n_q}_l{L}", [L], H=H, n_q=n_q, seed=seed)
    pos = torch.arange(L)
    k = torch.round(64.0 * (1.0 - pos.double() / L)).long()
    _set_rope_block(inp, 0, pos, k)
    _ramp_query(inp, [nats / 64.0] * H, [0.0 if h % 2 == 0 else 0.5 for h in range(H)])
    return inp


def wide_range_query(lens: Sequence[int], H: int = 12, n_q: int = 1, binades: float = 20.0,
                     big: Optional[float] = 4096.0, seed: int = 0) -> MlaInputs:
    """Query rows whose entries span `binades` binades: |q_d| = 2^-u with u uniform in
    [0, binades), random sign (bf16). With `big`, one entry of every odd row is set to
    `big` (2^12 by default: all the row's other entries then sit below 2^-12 of it)."""
    inp = make_inputs(f"wide_range_query_h{H}_q{n_q}", list(lens), H=H, n_q=n_q, seed=seed)
    g = torch.Generator().manual_seed(seed + 7)
    B = inp.B
    u = torch.rand(B, n_q, H, D, generator=g, dtype=torch.float64) * binades
    sign = torch.where(torch.rand(B, n_q, H, D, generator=g) < 0.5, -1.0, 1.0).double()
    q = sign * torch.exp2(-u)
    rows = q.view(-1, D)
    at = torch.randint(0, D, (rows.shape[0],), generator=g)
    if big is not None:
        for r in range(1, rows.shape[0], 2):
            rows[r, int(at[r])] = float(big)
    inp.q = q.to(torch.bfloat16)
    return inp


WORKLOADS = {
    "tiny_decode": tiny_decode,
    "batched_paged_decode": batched_paged_decode,
    "long_history_decode": long_history_decode,
    "spec_verify": spec_verify,
    "causal_prefill": causal_prefill,
}
