"""The profiling hook (mla_set_trace_buffer): a traced call runs its own instantiation of
the attention kernel, gives bit-identical results to an untraced one, and leaves ordered
per-CTA timestamps and counts of the tiles and units each CTA processed."""
import numpy as np
import pytest
import torch

import mla_latent_kv_attention_gb300 as mla
from mla_latent_kv_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda"
WORDS = 16  # stamps a CTA: entry, wait done, plan done, first scores, last P, last PV,
            # last epilogue, exit, tiles << 32 | units, ...


@pytest.mark.parametrize("n_q", [1, 4])
def test_traced_call_matches_and_stamps_are_ordered(n_q):
    inp = W.make_inputs(f"trace_{n_q}", [5000, 300, 12000, 0, 77], H=12, n_q=n_q, seed=40 + n_q)
    kv = mla.KVCache.from_inputs(inp, DEV)
    q = inp.q.to(DEV)
    ws = mla.workspace(mla.MLA_OP_VERIFY, inp.B, inp.H, n_q, DEV)
    ref_out, ref_lse = mla.mla_verify(kv, q, inp.sm_scale, ws=ws)
    torch.cuda.synchronize()
    n_ctas = torch.cuda.get_device_properties(0).multi_processor_count
    tr = torch.zeros(n_ctas * WORDS, dtype=torch.int64, device=DEV)
    lib = mla.library()
    lib.mla_set_trace_buffer(tr.data_ptr(), tr.numel() * 8)
    try:
        out, lse = mla.mla_verify(kv, q, inp.sm_scale, ws=ws)
        torch.cuda.synchronize()
    finally:
        lib.mla_set_trace_buffer(None, 0)
    assert mla.mla_read_status(ws) == 0
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
    t = tr.view(n_ctas, WORDS).cpu().numpy()
    assert np.all(t[:, 0] > 0) and np.all(t[:, 7] > 0)  # every CTA entered and left
    for a, b in ((0, 1), (1, 2), (2, 7)):
        assert np.all(t[:, a] <= t[:, b]), (a, b)
    worked = (t[:, 8] >> 32) > 0
    assert worked.any()
    # CTAs with tiles: scores read after the plan, the last epilogue before the exit
    assert np.all(t[worked, 2] <= t[worked, 3]) and np.all(t[worked, 6] <= t[worked, 7])
    # every cached position of every sequence is covered by the CTAs' tiles
    tiles = int((t[:, 8] >> 32).sum())
    need = int(sum((int(L) + 127) // 128 for L in inp.seq_lens.tolist()))
    assert tiles >= need
