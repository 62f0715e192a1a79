"""mla_cache_append (new latent rows into the paged FP8 cache) against the oracle, bit for
bit: every byte of the pool after the call, written rows and untouched ones."""
import math

import numpy as np
import pytest
import torch

import mla_latent_kv_attention_gb300 as mla
import oracle
from mla_latent_kv_attention_gb300 import workloads as W
from tests.parity import compare

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _rows(n, seed, special=True):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, 576, generator=g) * torch.exp(torch.randn(n, 1, generator=g))
    x = x.to(torch.bfloat16)
    if special and n > 0:
        x[0, :6] = torch.tensor([1e30, -1e30, float("inf"), -float("inf"), -0.0, 0.0]).to(torch.bfloat16)
    return x


@pytest.mark.parametrize("n,pages,page_size", [(1, 2, 64), (37, 8, 64), (500, 20, 128),
                                                (8192, 200, 64)])
def test_append_matches_oracle(n, pages, page_size):
    g = torch.Generator().manual_seed(n)
    pool = torch.randint(0, 256, (pages, page_size, 576), dtype=torch.uint8, generator=g)
    x = _rows(n, n + 1)
    rows = pages * page_size
    slots = torch.randperm(rows, generator=g)[:n].to(torch.int64)
    slots[::7] = -1  # padding entries are skipped
    kv_scale = float(x.float().abs().clamp(max=1e4).max()) / 448.0
    ref = oracle.cache_append(pool, x, slots, kv_scale)
    pool_d = pool.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    mla.mla_cache_append(pool_d, x.to(DEV), slots.to(DEV), kv_scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(pool_d.cpu().numpy(), ref)


def test_append_out_of_range_slot_reports_bounds():
    pool = torch.zeros(2, 64, 576, dtype=torch.uint8)
    x = _rows(3, 9, special=False)
    slots = torch.tensor([5, 128, 7], dtype=torch.int64)  # 128 rows in the pool
    pool_d = pool.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    mla.mla_cache_append(pool_d, x.to(DEV), slots.to(DEV), 0.01, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 6
    ref = oracle.cache_append(pool, x[[0, 2]], slots[[0, 2]], 0.01)
    assert np.array_equal(pool_d.cpu().numpy(), ref)


def test_append_then_verify():
    """The speculative-verify loop: write four new positions per sequence into their cache
    slots, then verify them; the attention reads exactly the appended codes."""
    inp = W.make_inputs("append", [900, 4100, 64], H=12, n_q=4, seed=61)
    # new rows drawn like the cached ones (N(0, 1) latent entries)
    x = torch.randn(4 * inp.B, 576, generator=torch.Generator().manual_seed(62)).to(torch.bfloat16)
    slots = []
    for b, L in enumerate(inp.seq_lens.tolist()):
        for pos in range(L - 4, L):
            slots.append(int(inp.page_table[b, pos // 64]) * 64 + pos % 64)
    slots = torch.tensor(slots, dtype=torch.int64)
    new_pool = torch.from_numpy(oracle.cache_append(inp.pool, x, slots, inp.kv_scale))
    kv = mla.KVCache.from_inputs(inp, DEV)
    mla.mla_cache_append(kv.pool, x.to(DEV), slots.to(DEV), inp.kv_scale)
    torch.cuda.synchronize()
    assert torch.equal(kv.pool.cpu(), new_pool)
    out, lse = mla.mla_verify(kv, inp.q.to(DEV), inp.sm_scale)
    torch.cuda.synchronize()
    inp2 = W.MlaInputs("append2", new_pool, inp.page_table, inp.seq_lens, inp.q, inp.kv_scale,
                       inp.sm_scale, 64)
    ref_out, ref_lse = oracle.attention(inp2)
    compare(out, lse, ref_out, ref_lse, "verify after append")


def test_append_reproduces_generator_codes():
    """Rows appended through mla_cache_append hold exactly the codes the input generator
    gives the same values (x * (1 / kv_scale) in binary32, clamped, rounded to nearest
    even): appended rows and generated rows are indistinguishable to the attention
    kernels."""
    g = torch.Generator().manual_seed(71)
    n = 4096
    x = torch.randn(n, 576, generator=g).to(torch.bfloat16)
    kv_scale = float(x.float().abs().max()) / 448.0
    want = W.quantize_e4m3(x.float(), kv_scale)
    pool_d = torch.zeros(n // 64, 64, 576, dtype=torch.uint8, device=DEV)
    slots = torch.randperm(n, generator=g).to(torch.int64)
    mla.mla_cache_append(pool_d, x.to(DEV), slots.to(DEV), kv_scale)
    torch.cuda.synchronize()
    got = pool_d.view(n, 576).cpu()[slots]
    assert torch.equal(got, want)
