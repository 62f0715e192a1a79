"""Wide dynamic range against the float64 oracle, through the C ABI.

N(0, 1) queries and keys keep every weight within a few binades of its row's largest,
so these cases are built to leave that regime (workloads in ``workloads.py``):

* an attention sink: one key 4 to 16 nats above a tail of 141,999 keys, the tail exactly
  flat (even heads) or spread by about 0.9 nats (odd heads): the tail's total weight is
  comparable to the sink's while each tail weight is 2^-6 to 2^-23 of it;
* a graded tail: scores falling linearly over 30 nats from the first key to the last;
* query rows whose entries span 20 binades, in some cases with one entry 2^12 above
  the rest.

Each runs through decode (8, 12 and 16 heads: one launch of 16 rows or fewer), verify (48
rows a unit, or 32) and prefill (48 rows a unit) at the tolerances of tests/parity.py.
"""
import numpy as np
import pytest
import torch

import mla_latent_kv_attention_gb300 as mla
import oracle
from mla_latent_kv_attention_gb300 import workloads as W
from tests.parity import compare

pytestmark = pytest.mark.gpu

DEV = "cuda"


def run(inp):
    kv = mla.KVCache.from_inputs(inp, DEV)
    q = inp.q.to(DEV)
    ws = mla.workspace(mla.MLA_OP_DECODE if inp.n_q == 1 else mla.MLA_OP_VERIFY, inp.B, inp.H,
                       inp.n_q, DEV)
    if inp.n_q == 1:
        out, lse = mla.mla_decode(kv, q[:, 0].contiguous(), inp.sm_scale, ws=ws)
        out, lse = out[:, None], lse[:, None]
    else:
        out, lse = mla.mla_verify(kv, q, inp.sm_scale, ws=ws)
    torch.cuda.synchronize()
    assert mla.mla_read_status(ws) == 0
    return out, lse


def run_prefill(inp):
    kv = mla.KVCache.from_inputs(inp, DEV)
    out, lse = mla.mla_prefill(kv, inp.q[0].to(DEV).contiguous(), inp.sm_scale)
    torch.cuda.synchronize()
    return out[None], lse[None]


def check_full(inp, what):
    out, lse = run(inp)
    ref_out, ref_lse = oracle.attention(inp)
    return compare(out, lse, ref_out, ref_lse, what)


def check_prefill_rows(inp, what, n_random=8, seed=0):
    out, lse = run_prefill(inp)
    T, H = inp.n_q, inp.H
    g = np.random.default_rng(seed)
    pos = [0, 1, T // 2, T - 2, T - 1] + [int(x) for x in g.integers(2, T - 2, n_random)]
    rows = np.array([(0, j, h) for j in pos for h in range(H)], dtype=np.int32)
    ref_out, ref_lse = oracle.attention_rows(inp, rows)
    idx = (rows[:, 0], rows[:, 1], rows[:, 2])
    return compare(out.cpu()[idx], lse.cpu()[idx], ref_out, ref_lse, what)


@pytest.mark.parametrize("H", [8, 12, 16])
def test_attention_sink_decode(H):
    check_full(W.attention_sink(L=142000, H=H), f"attention sink, decode H={H}")


@pytest.mark.parametrize("H,n_q", [(12, 4), (16, 2)])
def test_attention_sink_verify(H, n_q):
    check_full(W.attention_sink(L=142000, H=H, n_q=n_q, B=2, seed=1),
               f"attention sink, verify H={H} n_q={n_q}")


def test_attention_sink_split_across_sequences():
    """Several sequences in one call: the sink sits in a different split for each."""
    inp = W.attention_sink(L=40000, H=12, B=6, seed=2)
    check_full(inp, "attention sink, 6 sequences")


def test_attention_sink_prefill():
    inp = W.attention_sink(L=50000, H=12, n_q=512, seed=3)
    check_prefill_rows(inp, "attention sink, prefill")


def test_graded_tail_decode():
    check_full(W.graded_tail(L=142000, H=12), "graded tail, decode")


def test_graded_tail_verify():
    check_full(W.graded_tail(L=142000, H=12, n_q=4, seed=4), "graded tail, verify")


def test_graded_tail_prefill():
    check_prefill_rows(W.graded_tail(L=20000, H=12, n_q=384, seed=5), "graded tail, prefill")


@pytest.mark.parametrize("n_q", [1, 4])
def test_wide_range_query(n_q):
    """Query entries over 20 binades, every odd row with one entry 2^12 above the rest.
    Those rows' scores spread over hundreds of nats, so their output is one value row (or
    a few) and its bf16 rounding alone is 1.9e-3 to 2.1e-3 relative on such inputs, at
    the tolerance itself; the float32-output entry point (the same kernel and the same
    query split) is compared, so what is measured is the split."""
    inp = W.wide_range_query([3000, 700, 64, 9000], H=12, n_q=n_q, seed=6 + n_q)
    kv = mla.KVCache.from_inputs(inp, DEV)
    out, lse = mla.mla_verify_f32(kv, inp.q.to(DEV), inp.sm_scale)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.attention(inp)
    compare(out, lse, ref_out, ref_lse, f"wide-range query rows, float32 out, n_q={n_q}")


@pytest.mark.parametrize("n_q", [1, 4])
def test_wide_range_query_bf16(n_q):
    """Query entries over 20 binades (no dominant entry), bf16 outputs."""
    inp = W.wide_range_query([3000, 700, 64, 9000], H=12, n_q=n_q, big=None, seed=16 + n_q)
    check_full(inp, f"wide-range query rows, n_q={n_q}")


def test_wide_range_query_prefill():
    inp = W.wide_range_query([1024 + 256], H=12, n_q=256, big=None, seed=9)
    out, lse = run_prefill(inp)
    ref_out, ref_lse = oracle.attention(inp)
    compare(out, lse, ref_out, ref_lse, "wide-range query rows, prefill")
