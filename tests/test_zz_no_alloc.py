"""mla_decode_static_ws: decode for callers that cannot allocate device memory.

Engines that have reserved almost all device memory for their own pools, and hot loops
that must not call cudaMalloc/cudaFree (which can synchronise the device), cannot hand
the library a workspace. This entry point runs decode on a fixed workspace the library
keeps in device memory. The test calls it through the C ABI twice in a row, on two
different batches so the second call inherits the first call's leftovers in the shared
workspace, and checks each result against mla_decode with a workspace of its own, within
the tolerances every parity test here uses. It also checks that a batch too large for
the fixed workspace is refused before any work is enqueued, that its device-side status
words (a page index outside the pool) are read through mla_read_status_static, and, once,
that its result agrees with the float64 oracle.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import mla_latent_kv_attention_gb300 as mla
import oracle
from mla_latent_kv_attention_gb300 import workloads as W
from tests.parity import compare

pytestmark = pytest.mark.gpu


def _static_decode(inp, kv):
    lib = mla.library()
    q = inp.q[:, 0].contiguous().cuda()
    out = torch.full((inp.B, inp.H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((inp.B, inp.H), float("nan"), dtype=torch.float32, device="cuda")
    c = kv.c_struct()
    status = lib.mla_decode_static_ws(ctypes.byref(c), q.data_ptr(), inp.B, inp.H,
                                      inp.sm_scale, out.data_ptr(), lse.data_ptr(),
                                      torch.cuda.current_stream().cuda_stream)
    assert status == 0, mla.STATUS.get(status, status)
    return out, lse


def test_static_workspace_decode_matches_decode_twice():
    batches = [
        W.make_inputs("nalloc_a", [5000, 1200, 64, 3001], H=12, n_q=1, seed=41),
        W.make_inputs("nalloc_b", [900, 17000], H=16, n_q=1, seed=42),
    ]
    for inp in batches:
        kv = mla.KVCache.from_inputs(inp, "cuda")
        got_out, got_lse = _static_decode(inp, kv)
        ref_out, ref_lse = mla.mla_decode(kv, inp.q[:, 0].contiguous().cuda(), inp.sm_scale)
        torch.cuda.synchronize()
        compare(got_out, got_lse, ref_out.double().cpu().numpy(),
                ref_lse.double().cpu().numpy(), f"static workspace {inp.name}")


def test_static_workspace_covers_any_batch():
    """The decode workspace depends on the heads and the SM count, not on the batch: the
    fixed 16 MiB array serves 16-head decode of any batch, and a call with invalid
    arguments is still rejected before anything is enqueued."""
    lib = mla.library()
    dev = torch.cuda.current_device()
    sizes = [mla.mla_workspace_size(mla.MLA_OP_DECODE, B, 16, 1, dev) for B in (1, 32, 1 << 20)]
    assert sizes[0] > 0 and len(set(sizes)) == 1 and sizes[0] <= (16 << 20)
    fake = 0x100000  # never touched: the call must fail before enqueuing work
    kv = mla.mla_kv_t(fake, 1, 64, fake, 1, fake, 1.0)
    status = lib.mla_decode_static_ws(ctypes.byref(kv), fake, -1, 16, 0.1, fake, fake, None)
    assert status == 1  # MLA_ERR_INVALID_ARG


def test_static_workspace_status_and_oracle():
    """A page index outside the pool is reported by mla_read_status_static (the kernel
    reads no such page); the next call on the same fixed workspace is clean and agrees
    with the oracle."""
    lib = mla.library()
    stream = torch.cuda.current_stream().cuda_stream
    inp = W.make_inputs("nalloc_bad", [200, 700], H=12, n_q=1, seed=43)
    kv = mla.KVCache.from_inputs(inp, "cuda")
    kv.page_table[1, 2] = inp.pool.shape[0] + 5
    _static_decode(inp, kv)
    assert lib.mla_read_status_static(stream) == 6  # MLA_ERR_BOUNDS
    kv.page_table[1, 2] = int(inp.page_table[1, 2])
    out, lse = _static_decode(inp, kv)
    assert lib.mla_read_status_static(stream) == 0
    ref_out, ref_lse = oracle.attention(inp)
    compare(out[:, None], lse[:, None], ref_out, ref_lse, "static workspace vs oracle")
