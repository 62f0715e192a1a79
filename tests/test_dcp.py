"""Decode-context parallelism: the host logic, on the CPU.

The shard plan must cut every sequence into disjoint page-aligned pieces that cover it,
with the new positions in one shard. Computing each shard's views with the oracle and
merging them with the oracle's merge must reproduce the oracle's attention over the whole
sequence (this checks the causal split: the final shard masked, the others seen whole).
The gather runs as two gloo ranks in separate processes."""
import dataclasses
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from mla_latent_kv_attention_gb300 import dcp
from mla_latent_kv_attention_gb300 import workloads as W


@pytest.mark.parametrize("world", [1, 2, 3, 8])
@pytest.mark.parametrize("n_q", [1, 2, 4])
def test_shard_plan_covers_each_sequence(world, n_q):
    g = np.random.default_rng(world * 10 + n_q)
    for page in (16, 64):
        lens = [0, n_q, page, page + 1, 2 * page + n_q - 1] + list(g.integers(n_q, 40 * page, 20))
        plan = dcp.shard_plan(lens, page, world, n_q)
        assert len(plan) == world
        for b, L in enumerate(lens):
            covered = np.zeros(L, dtype=int)
            finals = 0
            prev_end = 0
            for sh in plan:
                start = sh.first_page[b] * page
                n = sh.length[b]
                assert 0 <= n <= sh.num_pages[b] * page
                if n:
                    assert start == prev_end  # contiguous, in rank order
                    prev_end = start + n
                covered[start:start + n] += 1
                if sh.final[b]:
                    finals += 1
                    assert start + n == L and n >= n_q
            assert (covered == 1).all()
            assert finals == (1 if L > 0 else 0)


def _view_inputs(inp, pt, lens, shift):
    """The oracle's form of a view: causal as defined (shift 0), or, for a shard every new
    position sees whole (shift n_q - 1), each new position as a one-position query over the
    whole shard."""
    if shift == 0:
        return dataclasses.replace(inp, page_table=pt, seq_lens=lens)
    assert shift == inp.n_q - 1
    q = inp.q.reshape(inp.B * inp.n_q, 1, inp.H, inp.q.shape[-1])
    return dataclasses.replace(inp, page_table=pt.repeat_interleave(inp.n_q, dim=0),
                               seq_lens=lens.repeat_interleave(inp.n_q), q=q)


def _oracle_partials(inp, shard):
    outs, lses = [], []
    for pt, lens, shift in dcp.shard_views(inp.page_table, shard):
        o, l = oracle.attention(_view_inputs(inp, pt, lens, shift))
        outs.append(o.reshape(inp.B, inp.n_q, inp.H, -1))
        lses.append(l.reshape(inp.B, inp.n_q, inp.H))
    return np.stack(outs), np.stack(lses)


def _merge_and_check(inp, po, pl):
    S = po.shape[0]
    out, lse = oracle.merge_lse(po.reshape(S, -1, po.shape[-1]), pl.reshape(S, -1))
    ref_out, ref_lse = oracle.attention(inp)
    assert np.allclose(out.reshape(ref_out.shape), ref_out, rtol=0, atol=1e-12)
    fin = ~np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse.reshape(ref_lse.shape)), ~fin)
    assert np.allclose(lse.reshape(ref_lse.shape)[fin], ref_lse[fin], rtol=1e-13, atol=0)


@pytest.mark.parametrize("world", [2, 3, 8])
@pytest.mark.parametrize("n_q", [1, 4])
def test_sharded_oracle_merges_to_full_attention(world, n_q):
    inp = W.make_inputs("dcp", [0, 5, 64, 129, 700, 1000], H=4, n_q=n_q, seed=world + n_q)
    plan = dcp.shard_plan(inp.seq_lens.tolist(), inp.page_size, world, n_q)
    parts = [_oracle_partials(inp, sh) for sh in plan]
    po = np.concatenate([p[0] for p in parts])
    pl = np.concatenate([p[1] for p in parts])
    _merge_and_check(inp, po, pl)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _gloo_rank(rank, world, port, n_q, result):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        inp = W.make_inputs("dcp", [4, 200, 513, 1000], H=2, n_q=n_q, seed=11)
        plan = dcp.shard_plan(inp.seq_lens.tolist(), inp.page_size, world, n_q)
        po, pl = _oracle_partials(inp, plan[rank])
        go, gl = dcp.gather_partials(torch.from_numpy(po), torch.from_numpy(pl))
        assert go.shape[0] == world * plan[rank].parts
        _merge_and_check(inp, go.numpy(), gl.numpy())
        result[rank] = 1
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("n_q", [1, 4])
def test_gather_over_two_gloo_ranks(n_q):
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    result = manager.dict()
    mp.start_processes(_gloo_rank, args=(2, _free_port(), n_q, result), nprocs=2, join=True,
                       start_method="spawn")
    assert dict(result) == {0: 1, 1: 1}
