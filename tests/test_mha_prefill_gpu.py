"""MHA-form causal prefill (latent up-projected per head, then dense causal attention)
against the float64 oracle, through the C ABI. Small cases on every row; the full chunk
(8,192 new positions on a 32,768 prefix, 12 heads) on sampled rows. The default form is held
to the absorbed path's relative L2 and LSE bounds; the bf16 form (mla_prefill_mha_bf16) to
its own, looser ones (tests/parity.py)."""
import numpy as np
import pytest
import torch

import mla_latent_kv_attention_gb300 as mla
import oracle
from mla_latent_kv_attention_gb300 import workloads as W
from tests.parity import (LSE_REL, MHA_BF16_LSE_REL, MHA_BF16_REL_L2, MHA_MAX_ABS_ROW, REL_L2,
                          compare)

pytestmark = pytest.mark.gpu

DEV = "cuda"


def run(m, bf16=False):
    kv = mla.KVCache.from_inputs(m.cache, DEV)
    out, lse = mla.mla_prefill_mha(kv, m.q.to(DEV), m.w_ukv.to(DEV), m.cache.sm_scale, bf16=bf16)
    torch.cuda.synchronize()
    return out, lse


def check(got, gl, ref_out, ref_lse, what, bf16=False):
    return compare(got, gl, ref_out, ref_lse, what,
                   rel_l2=MHA_BF16_REL_L2 if bf16 else REL_L2,
                   lse_rel=MHA_BF16_LSE_REL if bf16 else LSE_REL, max_abs_row=MHA_MAX_ABS_ROW)


# (1280, 1000, 16): 80 pairs of query tiles for 76 clusters, so the four pairs of the last
# round are cut along the key axis and merged from partials
@pytest.mark.parametrize("T,prefix,H", [(128, 0, 1), (200, 300, 2), (384, 1000, 12), (64, 4096, 16),
                                        (1, 77, 8), (300, 0, 3), (129, 127, 12), (1280, 1000, 16)])
def test_mha_prefill_small(T, prefix, H):
    m = W.mha_prefill_inputs(T, prefix, H=H, seed=T + prefix + H)
    out, lse = run(m)
    ref_out, ref_lse = oracle.mha_prefill_rows(m.cache, m.q, m.w_ukv)
    check(out, lse, ref_out, ref_lse, f"mha T={T} prefix={prefix} H={H}")


@pytest.mark.parametrize("T,prefix,H", [(128, 0, 1), (384, 1000, 12), (1280, 1000, 16)])
def test_mha_prefill_bf16_form(T, prefix, H):
    m = W.mha_prefill_inputs(T, prefix, H=H, seed=T + prefix + H)
    out, lse = run(m, bf16=True)
    ref_out, ref_lse = oracle.mha_prefill_rows(m.cache, m.q, m.w_ukv)
    check(out, lse, ref_out, ref_lse, f"mha bf16 T={T} prefix={prefix} H={H}", bf16=True)


def test_mha_prefill_matches_absorbed_kernel_path():
    """The identity the oracle is pinned by, on the GPU: with signed-selection up-projections
    the MHA output is the selected entries of the absorbed kernel's output."""
    rng = np.random.default_rng(4)
    T, H = 96, 4
    m = W.mha_prefill_inputs(T, 500, H=H, seed=4)
    wk = np.zeros((512, H, 128))
    wv = np.zeros((512, H, 128))
    q_abs = np.zeros((T, H, 576))
    sel = []
    qf = m.q.double().numpy()
    for h in range(H):
        rk, rv = rng.permutation(512)[:128], rng.permutation(512)[:128]
        wk[rk, h, np.arange(128)] = 1.0
        wv[rv, h, np.arange(128)] = 1.0
        q_abs[:, h, rk] = qf[:, h, :128]
        q_abs[:, h, 512:] = qf[:, h, 128:]
        sel.append(rv)
    w = torch.from_numpy(np.concatenate([wk, wv], axis=2)).to(torch.bfloat16)
    kv = mla.KVCache.from_inputs(m.cache, DEV)
    out, lse = mla.mla_prefill_mha(kv, m.q.to(DEV), w.to(DEV), m.cache.sm_scale)
    qa = torch.from_numpy(q_abs).to(torch.bfloat16).to(DEV)
    out_a, lse_a = mla.mla_prefill(kv, qa, m.cache.sm_scale)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.mha_prefill_rows(m.cache, m.q, w)
    check(out, lse, ref_out, ref_lse, "mha selection")
    oa = out_a.float().cpu().numpy()
    picked = np.stack([oa[:, h][:, sel[h]] for h in range(H)], 1)
    got = out.float().cpu().numpy()
    assert np.linalg.norm(got - picked) / np.linalg.norm(picked) < REL_L2


def test_mha_prefill_full_chunk_sampled_rows():
    m = W.mha_prefill()
    out, lse = run(m)
    rng = np.random.default_rng(0)
    ts = np.concatenate([[0, 1, 127, 128, 4095, 8190, 8191], rng.integers(0, m.T, 25)])
    rows = np.array([[t, h] for h in (0, 11) for t in ts])
    ref_out, ref_lse = oracle.mha_prefill_rows(m.cache, m.q, m.w_ukv, rows)
    got = out[rows[:, 0], rows[:, 1]]
    gl = lse[rows[:, 0], rows[:, 1]]
    check(got, gl, ref_out, ref_lse, "mha full chunk")


def test_mha_prefill_reports_no_error():
    m = W.mha_prefill_inputs(256, 256, H=2, seed=9)
    kv = mla.KVCache.from_inputs(m.cache, DEV)
    L = int(m.cache.seq_lens[0])
    ws = torch.zeros(mla.library().mla_prefill_mha_workspace_size(L, 2, 0), dtype=torch.uint8,
                     device=DEV)
    mla.mla_prefill_mha(kv, m.q.to(DEV), m.w_ukv.to(DEV), m.cache.sm_scale, ws=ws)
    torch.cuda.synchronize()
    assert mla.mla_read_status(ws) == 0


@pytest.mark.parametrize("page_size", [128, 256])
def test_mha_prefill_larger_pages(page_size):
    m = W.mha_prefill_inputs(300, 700, H=4, seed=page_size, page_size=page_size)
    out, lse = run(m)
    ref_out, ref_lse = oracle.mha_prefill_rows(m.cache, m.q, m.w_ukv)
    check(out, lse, ref_out, ref_lse, f"mha pages of {page_size}")


def test_mha_prefill_reports_a_page_outside_the_pool():
    """A page-table entry past the pool is reported through the status words; the
    dequantisation checks the index before it reads, so nothing outside the pool is touched."""
    m = W.mha_prefill_inputs(64, 200, H=2, seed=5)
    pt = m.cache.page_table.clone()
    pt[0, 1] = m.cache.pool.shape[0] + 3
    kv = mla.KVCache(m.cache.pool.to(DEV), pt.to(DEV), m.cache.seq_lens.to(DEV), m.cache.kv_scale)
    L = int(m.cache.seq_lens[0])
    ws = torch.zeros(mla.library().mla_prefill_mha_workspace_size(L, 2, 0), dtype=torch.uint8,
                     device=DEV)
    mla.mla_prefill_mha(kv, m.q.to(DEV), m.w_ukv.to(DEV), m.cache.sm_scale, ws=ws)
    torch.cuda.synchronize()
    assert mla.mla_read_status(ws) == mla.MLA_ERR_BOUNDS
    # the next correct call on the same workspace reports no error
    kv_ok = mla.KVCache.from_inputs(m.cache, DEV)
    mla.mla_prefill_mha(kv_ok, m.q.to(DEV), m.w_ukv.to(DEV), m.cache.sm_scale, ws=ws)
    torch.cuda.synchronize()
    assert mla.mla_read_status(ws) == 0
