"""Decode-context parallelism (DCP) over the paged latent cache.

Every rank holds a contiguous, page-aligned shard of each sequence's positions and attends
to that shard alone; the shards' outputs, kept in float32 with their log-sum-exp, are
gathered and combined by ``mla_merge_lse`` into attention over the whole sequence ("Scaling
Kimi K3 on AMD Instinct MI355X: Matching NVIDIA HGX B300 Throughput per GPU on AgentX",
section "缓存可复用，还要能一致地恢复": under DCP each rank keeps part of the positions and the
partial results are combined through their normalisation statistics).

A rank's shard is a view of the shared page table (its pages, its shard length); nothing of
the pool is copied. With n_q new positions (speculative verify) the new positions are the
sequence's last n_q, so the shard that holds them (the final shard, made to hold at least
n_q positions) is the only one a causal mask reaches. Every other shard is wholly visible
to every new position: it runs with the causal limit moved past its end
(``mla_verify_f32_shard``, visible_shift = n_q - 1), so its pages are read once for all n_q
positions. A rank therefore contributes two partials per row when n_q > 1 (the final-shard
call and the whole-shard call); the one that does not apply to a sequence has no key,
lse = -inf and weight 0 in the merge.

``shard_plan`` and ``shard_views`` are host logic (``rank_views`` wraps the views as caches);
``rank_partials`` runs the rank's attention through ``mla_verify_f32``; ``gather_partials`` is the all-gather (in host memory
over a ``torch.distributed`` group, or a stack of the ranks' results when one process plays
every rank); ``merge_partials`` is ``mla_merge_lse``.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence, Tuple

import numpy as np
import torch

from . import MLA_DV, KVCache, mla_merge_lse, mla_verify_f32


@dataclasses.dataclass
class Shard:
    """One rank's part of every sequence (numpy int64 / bool arrays of length B)."""

    rank: int
    world: int
    n_q: int
    first_page: np.ndarray  # first logical page of the shard
    num_pages: np.ndarray   # pages in the shard
    length: np.ndarray      # positions in the shard
    final: np.ndarray       # the shard holds the sequence's last position

    @property
    def parts(self) -> int:
        """Partials this rank contributes per query row."""
        return 1 if self.n_q == 1 else 2


def shard_plan(seq_lens: Sequence[int], page_size: int, world: int, n_q: int = 1) -> List[Shard]:
    """Cut each sequence's pages into `world` contiguous ranges, rank r taking pages
    [r * P / world, (r + 1) * P / world) of the P pages; when the last non-empty range holds
    fewer than n_q positions its start moves back one page (page_size >= n_q), so the n_q new
    positions share one shard."""
    if world < 1 or page_size < 1 or n_q < 1 or page_size < n_q:
        raise ValueError("world >= 1, page_size >= n_q >= 1")
    L = np.asarray(seq_lens, dtype=np.int64).reshape(-1)
    if (L < 0).any() or ((L > 0) & (L < n_q)).any():
        raise ValueError("a non-empty sequence holds at least its n_q new positions")
    pages = (L + page_size - 1) // page_size
    bounds = (np.arange(world + 1, dtype=np.int64)[:, None] * pages[None, :]) // world
    last = np.full(L.shape, -1, dtype=np.int64)
    for b in range(L.shape[0]):
        if L[b] == 0:
            continue
        last[b] = max(r for r in range(world) if bounds[r + 1, b] > bounds[r, b])
        if L[b] - bounds[last[b], b] * page_size < n_q:
            moved = bounds[last[b], b] - 1
            bounds[: last[b] + 1, b] = np.minimum(bounds[: last[b] + 1, b], moved)
    shards = []
    for r in range(world):
        first = bounds[r].copy()
        num = bounds[r + 1] - bounds[r]
        length = np.clip(L - first * page_size, 0, num * page_size)
        shards.append(Shard(r, world, n_q, first, num, length, (last == r) & (L > 0)))
    return shards


def shard_views(page_table: torch.Tensor, shard: Shard):
    """The rank's page-table views, on page_table's device.

    Returns [(page_table, seq_lens, visible_shift), ...], one entry per partial, each over
    the B sequences with n_q rows: for n_q == 1 the shard itself (shift 0); for n_q > 1
    first the final shards, causally masked (shift 0, other sequences empty), then every
    other shard seen whole by every new position (shift n_q - 1, final ones empty)."""
    dev = page_table.device
    B = page_table.shape[0]
    width = max(1, int(shard.num_pages.max()) if B else 1)
    cols = torch.arange(width, dtype=torch.int64)
    first = torch.from_numpy(shard.first_page)
    idx = (first[:, None] + cols[None, :]).clamp_(max=page_table.shape[1] - 1)
    used = cols[None, :] < torch.from_numpy(shard.num_pages)[:, None]
    pt = torch.where(used, torch.gather(page_table.cpu().to(torch.int64), 1, idx),
                     torch.full_like(idx, -1)).to(torch.int32)
    length = torch.from_numpy(shard.length).to(torch.int32)
    pt = pt.contiguous().to(dev)
    if shard.n_q == 1:
        return [(pt, length.to(dev), 0)]
    final = torch.from_numpy(shard.final)
    lens_final = torch.where(final, length, torch.zeros_like(length))
    lens_rest = torch.where(final, torch.zeros_like(length), length)
    return [(pt, lens_final.to(dev), 0), (pt, lens_rest.to(dev), shard.n_q - 1)]


def rank_views(kv: KVCache, shard: Shard):
    """The rank's attention calls as [(KVCache view, visible_shift)], on kv's device."""
    return [(KVCache(kv.pool, pt, lens, kv.kv_scale), shift)
            for pt, lens, shift in shard_views(kv.page_table, shard)]


def rank_partials(views, q: torch.Tensor, sm_scale: float,
                  part_out: Optional[torch.Tensor] = None,
                  part_lse: Optional[torch.Tensor] = None, stream=None):
    """This rank's partials from its views (rank_views): part_out [parts, B, n_q, H, 512]
    float32 and part_lse [parts, B, n_q, H], each the normalised attention over the shard."""
    B, n_q, H = q.shape[0], q.shape[1], q.shape[2]
    P = len(views)
    if P != (1 if n_q == 1 else 2):
        raise ValueError("views do not match q's n_q")
    if part_out is None:
        part_out = torch.empty(P, B, n_q, H, MLA_DV, dtype=torch.float32, device=q.device)
    if part_lse is None:
        part_lse = torch.empty(P, B, n_q, H, dtype=torch.float32, device=q.device)
    for i, (view, shift) in enumerate(views):
        if view.seq_lens.shape[0] != B:
            raise ValueError("views do not match q's batch")
        mla_verify_f32(view, q, sm_scale, out=part_out[i], lse=part_lse[i], stream=stream,
                       visible_shift=shift)
    return part_out, part_lse


def gather_partials(part_out: torch.Tensor, part_lse: torch.Tensor, group=None):
    """All-gather every rank's partials in host memory over `group` (any backend that moves
    CPU tensors, e.g. gloo), in rank order. Returns ([world * parts, ...] out, lse) on the
    device of the inputs."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    host_out = part_out.detach().to("cpu")
    host_lse = part_lse.detach().to("cpu")
    outs = [torch.empty_like(host_out) for _ in range(world)]
    lses = [torch.empty_like(host_lse) for _ in range(world)]
    dist.all_gather(outs, host_out, group=group)
    dist.all_gather(lses, host_lse, group=group)
    return (torch.cat(outs, 0).to(part_out.device), torch.cat(lses, 0).to(part_lse.device))


def merge_partials(part_out: torch.Tensor, part_lse: torch.Tensor, stream=None):
    """[S, B, n_q, H, 512] float32 partials and [S, B, n_q, H] lse -> (out [B, n_q, H, 512]
    bf16, lse [B, n_q, H]) through mla_merge_lse."""
    S = part_out.shape[0]
    shape = part_lse.shape[1:]
    R = int(np.prod(shape))
    out, lse = mla_merge_lse(part_out.reshape(S, R, MLA_DV).contiguous(),
                             part_lse.reshape(S, R).contiguous(), stream=stream)
    return out.view(*shape, MLA_DV), lse.view(*shape)


def dcp_attention(kv: KVCache, q: torch.Tensor, sm_scale: float, world: int,
                  group=None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Attention of q over kv computed as `world` DCP shards and merged.

    With a process group, this process is rank `group.rank()` of `world`: it attends to its
    own shard and all-gathers the partials in host memory. Without one, this process plays
    every rank in turn on its device (the shards' attention calls are independent launches)
    and the gather is a stack in device memory."""
    B, n_q, H = q.shape[0], q.shape[1], q.shape[2]
    plan = shard_plan(kv.seq_lens.cpu().tolist(), kv.pool.shape[1], world, n_q)
    P = plan[0].parts
    if group is not None:
        import torch.distributed as dist
        mine = plan[dist.get_rank(group)]
        po, pl = rank_partials(rank_views(kv, mine), q, sm_scale, stream=stream)
        po, pl = gather_partials(po, pl, group)
    else:
        po = torch.empty(world * P, B, n_q, H, MLA_DV, dtype=torch.float32, device=q.device)
        pl = torch.empty(world * P, B, n_q, H, dtype=torch.float32, device=q.device)
        for r, sh in enumerate(plan):
            rank_partials(rank_views(kv, sh), q, sm_scale, po[r * P:(r + 1) * P],
                          pl[r * P:(r + 1) * P], stream=stream)
    return merge_partials(po, pl, stream=stream)
