"""CUDA path against the float64 oracle, through the C ABI, on seeded workloads.

Small cases span several 128-key blocks with ragged tails and every head count and
verify depth; the named workloads run at full size (the oracle on every row where it
finishes in seconds, on sampled rows otherwise). Tolerances are in tests/parity.py.
"""
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


def run_split(inp, kv=None, ws=None):
    kv = kv or mla.KVCache.from_inputs(inp, DEV)
    q = inp.q.to(DEV)
    if inp.n_q == 1:
        out, lse = mla.mla_decode(kv, q[:, 0].contiguous(), inp.sm_scale, ws=ws)
        out, lse = out[:, None], lse[:, None]
    else:
        out, lse = mla.mla_verify(kv, q, inp.sm_scale, ws=ws)
    torch.cuda.synchronize()
    return out, lse


def check_full(inp, what):
    out, lse = run_split(inp)
    ref_out, ref_lse = oracle.attention(inp)
    return compare(out, lse, ref_out, ref_lse, what)


def test_tiny_decode():
    check_full(W.tiny_decode(), "tiny decode")


SMALL = [
    # (lens, H, n_q, contiguous)
    ([1], 12, 1, False),
    ([63, 64, 65], 12, 1, False),
    ([127, 128, 129, 1000], 16, 1, False),
    ([300], 8, 1, True),
    ([5, 700], 1, 1, False),
    ([2000, 3, 257], 12, 4, False),
    ([4, 130], 12, 4, False),
    ([999], 16, 4, False),
    ([513, 77], 8, 2, False),
    ([1500], 12, 3, False),
    ([2], 5, 2, False),
]


@pytest.mark.parametrize("lens,H,n_q,contig", SMALL)
def test_small(lens, H, n_q, contig):
    inp = W.make_inputs("small", lens, H=H, n_q=n_q, contiguous=contig, seed=sum(lens) + H + n_q)
    check_full(inp, f"lens={lens} H={H} n_q={n_q}")


def test_batched_paged_decode():
    check_full(W.batched_paged_decode(), "batched paged decode")


@pytest.mark.parametrize("H", [8, 12, 16])
def test_long_history_decode(H):
    check_full(W.long_history_decode(H), f"long history H={H}")


def _sample_rows(B, n_q, H, extra, seed, must=()):
    g = np.random.default_rng(seed)
    rows = {tuple(r) for r in must}
    while len(rows) < len(must) + extra:
        rows.add((int(g.integers(B)), int(g.integers(n_q)), int(g.integers(H))))
    return np.array(sorted(rows), dtype=np.int32)


@pytest.mark.parametrize("page_size,n_q", [(128, 1), (256, 4), (128, 3)])
def test_larger_pages(page_size, n_q):
    """Pages of 128 and 256 positions: a 128-key tile is one page, or half of one."""
    inp = W.make_inputs("pages", [3000, 129, 777, 4096], H=12, n_q=n_q, page_size=page_size,
                        seed=page_size + n_q)
    check_full(inp, f"page_size={page_size} n_q={n_q}")


def test_causal_prefill_larger_pages():
    inp = W.make_inputs("prefill_pages", [1300], H=12, n_q=300, page_size=256, seed=52)
    out, lse = run_prefill(inp)
    ref_out, ref_lse = oracle.attention(inp)
    compare(out, lse, ref_out, ref_lse, "prefill, 256-position pages")


@pytest.mark.parametrize("n_q", [1, 4])
def test_many_short_sequences(n_q):
    """Hundreds of short sequences: every CTA's block range covers several sequences, so
    units past a CTA's second go through the staged query image, and most sequences are
    whole units written without a merge."""
    g = np.random.default_rng(40 + n_q)
    lens = [int(x) for x in g.integers(1, 400, size=500)]
    lens[7] = 0
    lens[300] = 0
    inp = W.make_inputs("short", lens, H=12, n_q=n_q, seed=43 + n_q)
    check_full(inp, f"500 short sequences, n_q={n_q}")


def test_spec_verify_sampled():
    inp = W.spec_verify()
    out, lse = run_split(inp)
    must = [(b, j, h) for b in (0, inp.B - 1) for j in range(inp.n_q) for h in range(inp.H)]
    rows = _sample_rows(inp.B, inp.n_q, inp.H, 64, 1, must)
    ref_out, ref_lse = oracle.attention_rows(inp, rows)
    idx = (rows[:, 0], rows[:, 1], rows[:, 2])
    compare(out.cpu()[idx], lse.cpu()[idx], ref_out, ref_lse, "spec verify (sampled rows)")


def run_prefill(inp):
    kv = mla.KVCache.from_inputs(inp, DEV)
    q = inp.q[0].to(DEV).contiguous()
    out, lse = mla.mla_prefill(kv, q, inp.sm_scale)
    torch.cuda.synchronize()
    return out[None], lse[None]


@pytest.mark.parametrize("T,prefix,H", [(1, 0, 12), (7, 5, 3), (200, 300, 12), (1024, 4096, 12),
                                        (130, 0, 16)])
def test_causal_prefill_small(T, prefix, H):
    inp = W.causal_prefill(T=T, prefix=prefix, H=H, seed=T + prefix)
    out, lse = run_prefill(inp)
    ref_out, ref_lse = oracle.attention(inp)
    compare(out, lse, ref_out, ref_lse, f"prefill T={T} prefix={prefix}")


@pytest.mark.parametrize("prefix,H", [(0, 12), (2000, 12), (500, 8)])
def test_causal_prefill_split_last_round(prefix, H):
    """Position blocks one and a quarter times the SM count: the blocks of the incomplete
    last round (the first positions) run as two halves along the keys on different CTAs
    and are merged. With no prefix the first blocks see fewer than 128 keys, so their
    second half is empty (a partial with lse = -inf)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    P = 48 // H
    units = sms + sms // 4
    T = units * P - 1  # the last position block (handed out first) is ragged
    inp = W.causal_prefill(T=T, prefix=prefix, H=H, seed=7 + prefix + H)
    out, lse = run_prefill(inp)
    ref_out, ref_lse = oracle.attention(inp)
    compare(out, lse, ref_out, ref_lse, f"prefill T={T} prefix={prefix} H={H} (split last round)")


def test_causal_prefill_full_sampled():
    """8,192 new positions on a 32,768-position prefix, 12 heads: every row is computed on
    the GPU; the oracle checks every head of the first six positions (the first sits on
    the boundary between the prefix and the chunk), the middle two, the last six (they
    see all 40,960 keys) and twelve random positions (rows are independent)."""
    inp = W.causal_prefill()
    out, lse = run_prefill(inp)
    T, H = inp.n_q, inp.H
    g = np.random.default_rng(5)
    pos = [0, 1, 2, 3, 4, 5, T // 2 - 1, T // 2] + list(range(T - 6, T))
    pos += [int(x) for x in g.choice(np.arange(6, T - 6), 12, replace=False)]
    rows = np.array([(0, j, h) for j in pos for h in range(H)], dtype=np.int32)
    assert len(rows) >= 256 and (rows[:, 1] == T - 1).any() and (rows[:, 1] == T // 2).any()
    print(f"causal prefill: {len(rows)} sampled rows over positions {min(pos)}..{max(pos)}")
    ref_out, ref_lse = oracle.attention_rows(inp, rows)
    idx = (rows[:, 0], rows[:, 1], rows[:, 2])
    compare(out.cpu()[idx], lse.cpu()[idx], ref_out, ref_lse, "causal prefill (sampled rows)")


# ---- edge cases and invariants -------------------------------------------------------

def test_empty_and_short_sequences():
    """seq_len 0 and seq_len < n_q: rows with no visible key give out = 0, lse = -inf."""
    inp = W.make_inputs("edge", [0, 2, 150], H=12, n_q=4, seed=21)
    check_full(inp, "empty/short")
    inp1 = W.make_inputs("edge1", [0, 70], H=8, n_q=1, seed=22)
    check_full(inp1, "empty decode")


def test_garbage_past_seq_len_is_ignored():
    """NaN codes in the unused tail of a sequence's last page must not reach the output."""
    inp = W.make_inputs("tail", [100, 191], H=12, n_q=2, seed=23)
    for b, L in enumerate(inp.seq_lens.tolist()):
        last = int(inp.page_table[b, (L - 1) // 64])
        inp.pool[last, L % 64:] = 0x7F  # e4m3 NaN
    check_full(inp, "NaN tail")


def test_bad_page_index_reports_bounds():
    inp = W.make_inputs("bad", [200], H=12, n_q=1, seed=24)
    kv = mla.KVCache.from_inputs(inp, DEV)
    kv.page_table[0, 1] = inp.pool.shape[0] + 5  # outside the pool
    ws = mla.workspace(mla.MLA_OP_DECODE, 1, 12, 1)
    run_split(inp, kv=kv, ws=ws)
    assert mla.mla_read_status(ws) == 6
    kv.page_table[0, 1] = int(inp.page_table[0, 1])
    out, lse = run_split(inp, kv=kv, ws=ws)
    assert mla.mla_read_status(ws) == 0
    ref_out, ref_lse = oracle.attention(inp)
    compare(out, lse, ref_out, ref_lse, "after bad page")


def test_length_beyond_page_table_reports_bounds():
    inp = W.make_inputs("long", [100], H=12, n_q=1, seed=25)
    kv = mla.KVCache.from_inputs(inp, DEV)
    kv.seq_lens[0] = 10 ** 6
    ws = mla.workspace(mla.MLA_OP_DECODE, 1, 12, 1)
    run_split(inp, kv=kv, ws=ws)
    assert mla.mla_read_status(ws) == 6


def test_page_permutation_bit_identical():
    inp = W.make_inputs("perm", [1000, 333], H=12, n_q=1, seed=26)
    out, lse = run_split(inp)
    g = torch.Generator().manual_seed(27)
    perm = torch.randperm(inp.pool.shape[0], generator=g)
    pool2 = torch.empty_like(inp.pool)
    pool2[perm] = inp.pool
    pt2 = inp.page_table.clone()
    m = pt2 >= 0
    pt2[m] = perm[pt2[m].long()].to(torch.int32)
    inp2 = W.MlaInputs("perm2", pool2, pt2, inp.seq_lens, inp.q, inp.kv_scale, inp.sm_scale, 64)
    out2, lse2 = run_split(inp2)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


@pytest.mark.parametrize("pad", ["zero", "repeat"])
def test_head_padding_bit_identical(pad):
    """12 real heads give identical bits whether run as 12 or padded to 16."""
    inp = W.make_inputs("h12", [3000, 517], H=12, n_q=1, seed=28)
    out, lse = run_split(inp)
    q16 = torch.zeros(inp.B, 1, 16, 576, dtype=torch.bfloat16)
    q16[:, :, :12] = inp.q
    if pad == "repeat":
        q16[:, :, 12:] = inp.q[:, :, :4]
    inp16 = W.MlaInputs("h16", inp.pool, inp.page_table, inp.seq_lens, q16, inp.kv_scale,
                        inp.sm_scale, 64)
    out16, lse16 = run_split(inp16)
    assert torch.equal(out16[:, :, :12], out) and torch.equal(lse16[:, :, :12], lse)


def test_verify_one_position_equals_decode():
    inp = W.make_inputs("v1", [777, 64], H=12, n_q=1, seed=29)
    kv = mla.KVCache.from_inputs(inp, DEV)
    q = inp.q.to(DEV)
    o1, l1 = mla.mla_decode(kv, q[:, 0].contiguous(), inp.sm_scale)
    o2, l2 = mla.mla_verify(kv, q, inp.sm_scale)
    assert torch.equal(o1, o2[:, 0]) and torch.equal(l1, l2[:, 0])


def test_verify_rows_match_decode_on_prefix():
    """Verify row j behaves like a decode whose cache ends at prefix + j + 1."""
    prefix = 900
    inp = W.make_inputs("vp", [prefix + 4], H=12, n_q=4, seed=30)
    out, lse = run_split(inp)
    for j in range(4):
        dec = W.MlaInputs("d", inp.pool, inp.page_table,
                          torch.tensor([prefix + j + 1], dtype=torch.int32),
                          inp.q[:, j:j + 1].clone(), inp.kv_scale, inp.sm_scale, 64)
        o, l = run_split(dec)
        ref_o, ref_l = oracle.attention(dec)
        compare(out[:, j:j + 1], lse[:, j:j + 1], ref_o, ref_l, f"verify row {j}")
        compare(o, l, ref_o, ref_l, f"decode prefix {j}")


def test_merge_lse_standalone():
    g = torch.Generator().manual_seed(31)
    S, R = 37, 24
    po = torch.randn(S, R, 512, generator=g)
    pl = torch.randn(S, R, generator=g) * 3
    pl[5, :] = -math.inf
    pl[:, 7] = -math.inf
    out, lse = mla.mla_merge_lse(po.to(DEV), pl.to(DEV))
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.merge_lse(po.double().numpy(), pl.double().numpy())
    compare(out, lse, ref_out, ref_lse, "merge")


def test_merge_lse_many_partials():
    """More partials per row than the merge keeps in registers (256), few rows (narrow
    chunks), rows whose partials are all empty, and a row whose only finite partials come
    after empty ones past the first 256 (an empty piece there must add nothing, not NaN)."""
    g = torch.Generator().manual_seed(33)
    S, R = 300, 4
    po = torch.randn(S, R, 512, generator=g)
    pl = torch.randn(S, R, generator=g) * 4
    pl[::7, 0] = -math.inf
    pl[:, 2] = -math.inf
    pl[:288, 3] = -math.inf
    out, lse = mla.mla_merge_lse(po.to(DEV), pl.to(DEV))
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.merge_lse(po.double().numpy(), pl.double().numpy())
    compare(out, lse, ref_out, ref_lse, "merge, 300 partials")


def test_cuda_graph_replay_matches_eager():
    inp = W.make_inputs("graph", [4000, 2500, 100], H=12, n_q=1, seed=32)
    kv = mla.KVCache.from_inputs(inp, DEV)
    q = inp.q[:, 0].to(DEV).contiguous()
    ws = mla.workspace(mla.MLA_OP_DECODE, inp.B, 12, 1)
    out = torch.empty(inp.B, 12, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(inp.B, 12, dtype=torch.float32, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        mla.mla_decode(kv, q, inp.sm_scale, out=out, lse=lse, ws=ws)
    torch.cuda.synchronize()
    ref = out.clone(), lse.clone()
    out.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        mla.mla_decode(kv, q, inp.sm_scale, out=out, lse=lse, ws=ws)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref[0]) and torch.equal(lse, ref[1])


def test_bounded_wait_reports_timeout_and_context_survives():
    """A wait that nothing satisfies (the test hook switches the key loads off for one call)
    gives up after its limit: the kernel returns, the status words say MLA_ERR_TIMEOUT, and
    the next call on the same workspace is correct and clean."""
    inp = W.make_inputs("stall", [300, 1000], H=12, n_q=1, seed=41)
    kv = mla.KVCache.from_inputs(inp, DEV)
    q = inp.q[:, 0].contiguous().to(DEV)
    ws = mla.workspace(mla.MLA_OP_DECODE, inp.B, inp.H, 1, DEV)
    mla.library().mla_test_stall_next_call()
    mla.mla_decode(kv, q, inp.sm_scale, ws=ws)
    torch.cuda.synchronize()
    assert mla.mla_read_status(ws) == mla.MLA_ERR_TIMEOUT
    out, lse = mla.mla_decode(kv, q, inp.sm_scale, ws=ws)
    torch.cuda.synchronize()
    assert mla.mla_read_status(ws) == 0
    ref_out, ref_lse = oracle.attention(inp)
    compare(out[:, None], lse[:, None], ref_out, ref_lse, "after a timed-out call")
