"""The float32-output attention call and the decode-context-parallel harness on the GPU.

mla_verify_f32 against the oracle, and against mla_verify: the same arithmetic, so the
bf16 rounding of its float32 output must equal the bf16 output bit for bit. The DCP
harness (every rank played in turn on this GPU, partials merged by mla_merge_lse) against
the oracle's attention over the whole sequence."""
import numpy as np
import pytest
import torch

import mla_latent_kv_attention_gb300 as mla
import oracle
from mla_latent_kv_attention_gb300 import dcp
from mla_latent_kv_attention_gb300 import workloads as W
from tests.parity import compare

pytestmark = pytest.mark.gpu

DEV = "cuda"

CASES = [
    ([1], 12, 1),
    ([0, 63, 129, 1000], 16, 1),
    ([2000, 4, 257], 12, 4),
    ([513, 77], 8, 2),
    ([20000] * 3, 12, 1),  # long enough to be split over several CTAs
    ([3000, 700], 16, 4),  # 64 rows a sequence: two launches over halves of the heads
]


@pytest.mark.parametrize("lens,H,n_q", CASES)
def test_verify_f32_matches_oracle_and_bf16_path(lens, H, n_q):
    inp = W.make_inputs("f32", lens, H=H, n_q=n_q, seed=len(lens) + H)
    kv = mla.KVCache.from_inputs(inp, DEV)
    q = inp.q.to(DEV)
    out32, lse32 = mla.mla_verify_f32(kv, q, inp.sm_scale)
    out16, lse16 = mla.mla_verify(kv, q, inp.sm_scale)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.attention(inp)
    compare(out32, lse32, ref_out, ref_lse, "verify_f32")
    assert torch.equal(out32.to(torch.bfloat16).view(torch.int16), out16.view(torch.int16))
    assert torch.equal(lse32, lse16)


@pytest.mark.parametrize("world", [2, 3, 8])
@pytest.mark.parametrize("lens,H,n_q", [([0, 5, 64, 129, 700, 3000], 12, 1),
                                        ([4, 130, 2000, 999], 16, 4),
                                        ([513, 77], 8, 2)])
def test_dcp_harness_small(world, lens, H, n_q):
    inp = W.make_inputs("dcp", lens, H=H, n_q=n_q, seed=world * 7 + n_q)
    kv = mla.KVCache.from_inputs(inp, DEV)
    out, lse = dcp.dcp_attention(kv, inp.q.to(DEV), inp.sm_scale, world)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.attention(inp)
    compare(out, lse, ref_out, ref_lse, f"dcp world {world}")


@pytest.mark.parametrize("name,world", [("batched_paged_decode", 8), ("spec_verify", 8),
                                        ("spec_verify", 3)])
def test_dcp_harness_named_workloads(name, world):
    inp = W.WORKLOADS[name]()
    kv = mla.KVCache.from_inputs(inp, DEV)
    out, lse = dcp.dcp_attention(kv, inp.q.to(DEV), inp.sm_scale, world)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.attention(inp)
    compare(out, lse, ref_out, ref_lse, f"dcp {name} world {world}")


@pytest.mark.parametrize("lens,H,n_q", [([2000, 4, 257, 0], 12, 4), ([513, 77], 16, 2),
                                        ([20000] * 2, 12, 3)])
def test_verify_f32_shard_sees_whole_view(lens, H, n_q):
    """visible_shift = n_q - 1: every new position sees every key of the view, as n_q
    one-position queries over it would (the oracle computes it that way); shift 0 is
    mla_verify_f32 bit for bit."""
    import dataclasses
    inp = W.make_inputs("shard", lens, H=H, n_q=n_q, seed=sum(lens) + n_q)
    kv = mla.KVCache.from_inputs(inp, DEV)
    q = inp.q.to(DEV)
    out, lse = mla.mla_verify_f32(kv, q, inp.sm_scale, visible_shift=n_q - 1)
    out0, lse0 = mla.mla_verify_f32(kv, q, inp.sm_scale, visible_shift=0)
    ref0, rl0 = mla.mla_verify_f32(kv, q, inp.sm_scale)
    torch.cuda.synchronize()
    assert torch.equal(out0, ref0) and torch.equal(lse0, rl0)
    one = dataclasses.replace(inp, page_table=inp.page_table.repeat_interleave(n_q, dim=0),
                              seq_lens=inp.seq_lens.repeat_interleave(n_q),
                              q=inp.q.reshape(inp.B * n_q, 1, H, 576))
    ref_out, ref_lse = oracle.attention(one)
    compare(out.reshape(ref_out.shape), lse.reshape(ref_lse.shape), ref_out, ref_lse,
            f"whole-view verify n_q={n_q}")
