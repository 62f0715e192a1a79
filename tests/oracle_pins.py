"""Pins that tie the float64 oracle to something other than itself.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with:
  * a library routine (torch's float8_e4m3fn and bfloat16 conversions; float64
    ``scaled_dot_product_attention`` and ``logsumexp`` on CPU),
  * a closed form (constant V, a single visible key, q = 0, duplicated keys),
  * an invariant the pages state (heads attend independently, so padding or
    permuting heads changes nothing for the real ones; partial attention over key
    ranges merged by normalisation statistics equals attention over the whole range;
    a new position sees its prefix and itself only).
The pins are plain functions so that ``test_oracle_mutants.py`` can run all of them
against deliberately broken builds of the oracle and check each break is caught.
"""
from __future__ import annotations

import math

import numpy as np
import torch
import torch.nn.functional as F

from mla_latent_kv_attention_gb300 import workloads as W

D, DV = 576, 512


def _tiny(seed=1, lens=(7, 11), H=3, n_q=2, page_size=4, contiguous=False):
    return W.make_inputs("tiny", list(lens), H=H, n_q=n_q, page_size=page_size,
                         contiguous=contiguous, seed=seed)


def _gather_keys(inp, b):
    """Codes of the cached rows of sequence b in logical order, via the page table."""
    L = int(inp.seq_lens[b])
    ps = inp.page_size
    idx = [int(inp.page_table[b, n // ps]) for n in range(L)]
    return torch.stack([inp.pool[idx[n], n % ps] for n in range(L)]) if L else torch.empty(0, D,
                                                                                           dtype=torch.uint8)


def sdpa_reference(inp):
    """Library reference: decode codes with torch's float8_e4m3fn, then float64 SDPA with
    K = whole row (broadcast over heads), V = first 512 entries, explicit causal mask."""
    B, n_q, H = inp.B, inp.n_q, inp.H
    out = torch.zeros(B, n_q, H, DV, dtype=torch.float64)
    lse = torch.zeros(B, n_q, H, dtype=torch.float64)
    for b in range(B):
        L = int(inp.seq_lens[b])
        k = _gather_keys(inp, b).view(torch.float8_e4m3fn).to(torch.float64) * inp.kv_scale
        v = k[:, :DV]
        q = inp.q[b].to(torch.float64).permute(1, 0, 2)  # [H, n_q, 576]
        mask = torch.zeros(n_q, L, dtype=torch.bool)
        for j in range(n_q):
            mask[j, :max(0, L - n_q + j + 1)] = True
        o = F.scaled_dot_product_attention(q, k.expand(H, L, D), v.expand(H, L, DV),
                                           attn_mask=mask, scale=inp.sm_scale)
        s = (q @ k.T) * inp.sm_scale
        s = s.masked_fill(~mask, float("-inf"))
        out[b] = o.permute(1, 0, 2)
        lse[b] = torch.logsumexp(s, dim=-1).permute(1, 0)
    return out.numpy(), lse.numpy()


def pin_e4m3_all_codes(orc):
    """All 256 codes against torch's float8_e4m3fn, plus the OCP E4M3 anchor values:
    max normal 448 (S.1111.110), min normal 2^-6, max subnormal 0.875*2^-6, min
    subnormal 2^-9, NaN only at S.1111.111."""
    lib_vals = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    for c in range(256):
        mine = orc.e4m3_value(c)
        ref = float(lib_vals[c])
        if math.isnan(ref):
            assert math.isnan(mine), c
        else:
            assert mine == ref, (c, mine, ref)
    assert orc.e4m3_value(0x7E) == 448.0 and orc.e4m3_value(0xFE) == -448.0
    assert orc.e4m3_value(0x08) == 2.0 ** -6
    assert orc.e4m3_value(0x07) == 0.875 * 2.0 ** -6
    assert orc.e4m3_value(0x01) == 2.0 ** -9
    assert math.isnan(orc.e4m3_value(0x7F)) and math.isnan(orc.e4m3_value(0xFF))


def pin_bf16(orc):
    """bfloat16 bit patterns against torch's bfloat16 -> float64 conversion."""
    g = torch.Generator().manual_seed(3)
    bits = torch.randint(0, 1 << 16, (4096,), generator=g, dtype=torch.int32)
    bits = bits[((bits >> 7) & 0xFF) != 0xFF]  # skip inf/nan exponents
    vals = bits.to(torch.int16).view(torch.bfloat16).to(torch.float64)
    for bt, v in zip(bits.tolist(), vals.tolist()):
        assert orc.bf16_value(bt & 0xFFFF) == v, (bt, v)


def pin_brute_force_sdpa(orc):
    """Tiny paged workloads (pages of 4 positions, ragged lengths, several new positions)
    against float64 SDPA; also a contiguous single-sequence decode."""
    for kw in (dict(seed=1), dict(seed=2, lens=(5,), H=2, n_q=1, contiguous=True),
               dict(seed=4, lens=(9, 3, 12), H=3, n_q=3)):
        inp = _tiny(**kw)
        out, lse = orc.attention(inp)
        ref_out, ref_lse = sdpa_reference(inp)
        np.testing.assert_allclose(out, ref_out, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def pin_constant_v(orc):
    """Every row's first 512 codes equal -> output equals that V whatever the scores."""
    inp = _tiny(seed=5, lens=(9,), H=2, n_q=1)
    row = inp.pool[0, 0, :DV].clone()
    inp.pool[:, :, :DV] = row
    out, _ = orc.attention(inp)
    v = row.view(torch.float8_e4m3fn).to(torch.float64).numpy() * inp.kv_scale
    for h in range(inp.H):
        np.testing.assert_allclose(out[0, 0, h], v, rtol=1e-13, atol=0)


def pin_single_key(orc):
    """One visible key -> output is that row's V and lse is its score."""
    inp = _tiny(seed=6, lens=(1,), H=3, n_q=1)
    out, lse = orc.attention(inp)
    codes = inp.pool[int(inp.page_table[0, 0]), 0]
    k = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy() * inp.kv_scale
    for h in range(inp.H):
        q = inp.q[0, 0, h].to(torch.float64).numpy()
        np.testing.assert_allclose(out[0, 0, h], k[:DV], rtol=1e-13, atol=0)
        assert abs(lse[0, 0, h] - inp.sm_scale * float(q @ k)) <= 1e-12 * max(1, abs(lse[0, 0, h]))


def pin_zero_query(orc):
    """q = 0 -> uniform weights: output = mean of the visible V rows, lse = ln(#visible)."""
    inp = _tiny(seed=7, lens=(10,), H=2, n_q=3)
    inp.q.zero_()
    out, lse = orc.attention(inp)
    k = _gather_keys(inp, 0).view(torch.float8_e4m3fn).to(torch.float64).numpy() * inp.kv_scale
    for j in range(3):
        vis = 10 - 3 + j + 1
        for h in range(2):
            np.testing.assert_allclose(out[0, j, h], k[:vis, :DV].mean(axis=0), rtol=1e-12,
                                       atol=1e-15)
            assert abs(lse[0, j, h] - math.log(vis)) < 1e-12


def pin_duplicate_key(orc):
    """Two identical keys instead of one -> lse grows by exactly ln 2, output unchanged."""
    one = W.make_inputs("one", [1], H=2, n_q=1, page_size=4, seed=8)
    two = W.make_inputs("two", [2], H=2, n_q=1, page_size=4, seed=8)
    two.pool[int(two.page_table[0, 0]), 1] = two.pool[int(two.page_table[0, 0]), 0]
    one.pool[int(one.page_table[0, 0]), 0] = two.pool[int(two.page_table[0, 0]), 0]
    one.q.copy_(two.q)
    one.kv_scale = two.kv_scale
    o1, l1 = orc.attention(one)
    o2, l2 = orc.attention(two)
    np.testing.assert_allclose(l2 - l1, math.log(2.0), rtol=0, atol=1e-12)
    np.testing.assert_allclose(o2, o1, rtol=1e-13, atol=0)


def pin_split_merge(orc):
    """Attention over [0, c) and [c, L) merged by their lse equals attention over [0, L),
    for every split point c (including empty ranges)."""
    inp = _tiny(seed=9, lens=(13,), H=2, n_q=1)
    full_out, full_lse = orc.attention(inp)
    for h in range(2):
        for c in range(0, 14):
            o1, l1 = orc.attention_range(inp, 0, 0, h, 0, c)
            o2, l2 = orc.attention_range(inp, 0, 0, h, c, 13)
            mo, ml = orc.merge_lse(np.stack([o1, o2])[:, None, :], np.array([[l1], [l2]]))
            np.testing.assert_allclose(mo[0], full_out[0, 0, h], rtol=1e-12, atol=1e-15)
            assert abs(ml[0] - full_lse[0, 0, h]) < 1e-12
    # a three-way split with one empty middle piece
    o = [orc.attention_range(inp, 0, 0, 1, a, b) for a, b in ((0, 5), (5, 5), (5, 13))]
    mo, ml = orc.merge_lse(np.stack([x[0] for x in o])[:, None, :],
                           np.array([[x[1]] for x in o]))
    np.testing.assert_allclose(mo[0], full_out[0, 0, 1], rtol=1e-12, atol=1e-15)


def pin_merge_weights(orc):
    """Merge against its closed form on random partials: weights exp(lse_s - lse) sum to 1
    and lse equals log(sum exp(lse_s)) computed by torch.logsumexp."""
    rng = np.random.default_rng(10)
    po = rng.standard_normal((5, 7, DV))
    pl = rng.standard_normal((5, 7)) * 4
    pl[2, 3] = -np.inf
    out, lse = orc.merge_lse(po, pl)
    ref_lse = torch.logsumexp(torch.from_numpy(pl), dim=0).numpy()
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-13)
    w = np.exp(pl - ref_lse[None, :])
    np.testing.assert_allclose((w[:, :, None] * po).sum(0), out, rtol=1e-12, atol=1e-14)
    # all-empty row
    out2, lse2 = orc.merge_lse(po[:2, :1], np.full((2, 1), -np.inf))
    assert lse2[0] == -np.inf and np.all(out2 == 0)


def pin_permuted_pages(orc):
    """Moving pages around the pool (and the table with them) changes nothing."""
    inp = _tiny(seed=11, lens=(11, 6), H=2, n_q=2)
    out, lse = orc.attention(inp)
    g = torch.Generator().manual_seed(12)
    perm = torch.randperm(inp.pool.shape[0], generator=g)
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(perm.numel())
    pool2 = torch.empty_like(inp.pool)
    pool2[perm] = inp.pool
    pt2 = inp.page_table.clone()
    m = pt2 >= 0
    pt2[m] = perm[pt2[m].long()].to(torch.int32)
    inp.pool, inp.page_table = pool2, pt2
    out2, lse2 = orc.attention(inp)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def pin_head_padding_and_permutation(orc):
    """12 heads padded to 16 with zero heads or repeated heads leave the 12 real heads
    exactly unchanged; permuting heads permutes outputs exactly."""
    inp = _tiny(seed=13, lens=(9,), H=12, n_q=1)
    out, lse = orc.attention(inp)
    for pad in ("zero", "repeat"):
        q16 = torch.zeros(1, 1, 16, D, dtype=torch.bfloat16)
        q16[:, :, :12] = inp.q
        if pad == "repeat":
            q16[:, :, 12:] = inp.q[:, :, :4]
        inp16 = W.MlaInputs("pad", inp.pool, inp.page_table, inp.seq_lens, q16, inp.kv_scale,
                            inp.sm_scale, inp.page_size)
        o16, l16 = orc.attention(inp16)
        assert np.array_equal(o16[:, :, :12], out) and np.array_equal(l16[:, :, :12], lse)
    perm = torch.randperm(12, generator=torch.Generator().manual_seed(14))
    inpp = W.MlaInputs("perm", inp.pool, inp.page_table, inp.seq_lens, inp.q[:, :, perm],
                       inp.kv_scale, inp.sm_scale, inp.page_size)
    op, lp = orc.attention(inpp)
    assert np.array_equal(op, out[:, :, perm.numpy()]) and np.array_equal(lp, lse[:, :, perm.numpy()])


def pin_causal_prefix(orc):
    """New position j of a chunk equals a one-query decode whose cache ends at that
    position: prefill row i == decode with L = prefix + i + 1."""
    prefix, T = 5, 4
    inp = _tiny(seed=15, lens=(prefix + T,), H=2, n_q=T)
    out, lse = orc.attention(inp)
    for i in range(T):
        dec = W.MlaInputs("dec", inp.pool, inp.page_table,
                          torch.tensor([prefix + i + 1], dtype=torch.int32),
                          inp.q[:, i:i + 1].clone(), inp.kv_scale, inp.sm_scale, inp.page_size)
        o, l = orc.attention(dec)
        np.testing.assert_allclose(o[0, 0], out[0, i], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(l[0, 0], lse[0, i], rtol=1e-13)


def pin_sampled_rows(orc):
    """The row-list entry point returns exactly the rows of the full computation."""
    inp = _tiny(seed=16, lens=(9, 12), H=3, n_q=3)
    out, lse = orc.attention(inp)
    rows = np.array([[1, 2, 0], [0, 0, 2], [1, 0, 1], [0, 2, 2]])
    o, l = orc.attention_rows(inp, rows)
    for i, (b, j, h) in enumerate(rows):
        assert np.array_equal(o[i], out[b, j, h]) and l[i] == lse[b, j, h]


def pin_e4m3_encode(orc):
    """The encoder against the decoder, the OCP rounding rule and torch's float8_e4m3fn
    conversion: every finite code (both signs, zero, subnormals) encodes back to itself;
    the midpoint of two neighbouring codes goes to the one with the even mantissa bit and
    any point off the midpoint to the nearer one; magnitudes past 448 and infinities
    saturate, -0 keeps its sign, NaN gives 0x7F; random binary32 values within +-448 give
    torch's codes (round to nearest even)."""
    for c in list(range(0x7F)) + list(range(0x80, 0xFF)):
        assert orc.e4m3_encode(orc.e4m3_value(c)) == c, c
    for c in range(0x7E):
        lo, hi = orc.e4m3_value(c), orc.e4m3_value(c + 1)
        mid, eps = (lo + hi) / 2, (hi - lo) * 1e-3
        even = c if c % 2 == 0 else c + 1
        assert orc.e4m3_encode(mid) == even, c
        assert orc.e4m3_encode(-mid) == 0x80 | even, c
        assert orc.e4m3_encode(mid - eps) == c and orc.e4m3_encode(mid + eps) == c + 1, c
    for v, code in ((448.0, 0x7E), (464.0, 0x7E), (1e6, 0x7E), (-1e6, 0xFE), (math.inf, 0x7E),
                    (-math.inf, 0xFE), (0.0, 0x00), (-0.0, 0x80), (2.0 ** -10, 0x00),
                    (1.5 * 2.0 ** -10, 0x01)):
        assert orc.e4m3_encode(v) == code, (v, code)
    assert orc.e4m3_encode(math.nan) == 0x7F
    g = torch.Generator().manual_seed(5)
    x = torch.randn(20000, generator=g) * torch.exp(torch.randn(20000, generator=g) * 3)
    x = x.clamp(-448, 448)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).tolist()
    mine = [orc.e4m3_encode(float(v)) for v in x.tolist()]
    assert mine == ref


def pin_cache_append(orc):
    """Appending rows against torch: a written row holds torch's float8_e4m3fn codes of the
    binary32 product x * (1/kv_scale) (saturated at +-448); rows with a negative slot and
    rows nobody writes stay as they were; a slot past the pool is refused."""
    g = torch.Generator().manual_seed(6)
    pool = torch.randint(0, 256, (6, 4, D), dtype=torch.uint8, generator=g)  # 24 rows
    x = (torch.randn(5, D, generator=g) * 3).to(torch.bfloat16)
    x[0, :4] = torch.tensor([1e30, -1e30, float("inf"), -0.0]).to(torch.bfloat16)
    slots = [3, -1, 23, 0, 10]
    scale = 0.0173
    new = orc.cache_append(pool, x, slots, scale).reshape(-1, D)
    old = pool.reshape(-1, D).numpy()
    inv = torch.tensor(1.0, dtype=torch.float32) / torch.tensor(scale, dtype=torch.float32)
    for r in range(old.shape[0]):
        if r not in slots:
            assert (new[r] == old[r]).all(), r
    for i, slot in enumerate(slots):
        if slot < 0:
            continue
        prod = (x[i].float() * inv).clamp(-448, 448)
        ref = prod.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert (new[slot] == ref).all(), i
    try:
        orc.cache_append(pool, x[:1], [24], scale)
    except ValueError:
        pass
    else:
        raise AssertionError("a slot past the pool was accepted")


def pin_top_k_renorm(orc):
    """Top-k renormalisation against closed forms and torch.topk: k = 1 is one-hot at a
    unique maximum; ties at the pivot are all kept; k <= 0 or k >= V is p / sum p; on rows
    without ties the kept set is torch.topk's and the kept entries keep their ratios and
    sum to 1."""
    p = np.array([[0.1, 0.3, 0.3, 0.3], [0.05, 0.5, 0.2, 0.25], [0.2, 0.2, 0.2, 0.4]])
    out = orc.top_k_renorm_prob(p, [2, 1, 9])
    assert np.allclose(out[0], [0, 1 / 3, 1 / 3, 1 / 3], rtol=0, atol=1e-15)
    assert np.array_equal(out[1], [0, 1, 0, 0])
    assert np.allclose(out[2], p[2] / p[2].sum(), rtol=0, atol=1e-15)
    assert np.allclose(orc.top_k_renorm_prob(p, 0), p / p.sum(1, keepdims=True), rtol=0, atol=1e-15)
    g = torch.Generator().manual_seed(8)
    logits = torch.randn(6, 5000, generator=g, dtype=torch.float64) * 3
    probs = torch.softmax(logits, dim=1)
    ks = [1, 2, 17, 500, 4999, 5000]
    out = orc.top_k_renorm_prob(probs.numpy(), ks)
    for r, k in enumerate(ks):
        keep = np.zeros(5000, dtype=bool)
        keep[torch.topk(probs[r], min(k, 5000)).indices.numpy()] = True
        assert np.array_equal(out[r] > 0, keep), (r, k)
        kept = probs[r].numpy()[keep]
        assert np.allclose(out[r][keep], kept / kept.sum(), rtol=1e-12, atol=0)
        assert abs(out[r].sum() - 1.0) < 1e-12


def _selection(rng, H, n_out):
    """Per head: distinct rows of the 512-wide latent and signs, as a [512][H][n_out] matrix
    with one +-1 per column."""
    w = np.zeros((512, H, n_out))
    picks = []
    for h in range(H):
        rows = rng.permutation(512)[:n_out]
        signs = rng.choice([-1.0, 1.0], n_out)
        w[rows, h, np.arange(n_out)] = signs
        picks.append((rows, signs))
    return w, picks


def pin_mha_absorbed_identity(orc):
    """The MHA form and the absorbed form are one computation ("MI355X Kimi K2.5 vLLM AITER
    7x speedup", section "PR #35850 修复了什么": keys and values come from one shared latent):
    with W_UK_h and W_UV_h signed selections, the absorbed query [W_UK_h q_nope ; q_rope] is
    exact in bf16, the absorbed oracle's scores equal the MHA scores, and the MHA output is
    the selected, signed entries of the absorbed output."""
    rng = np.random.default_rng(21)
    T, H = 5, 3
    m = W.mha_prefill_inputs(T, 120, H=H, seed=21)
    wk, pk = _selection(rng, H, 128)
    wv, pv = _selection(rng, H, 128)
    w = torch.from_numpy(np.concatenate([wk, wv], axis=2)).to(torch.bfloat16)
    out, lse = orc.mha_prefill_rows(m.cache, m.q, w)
    qf = m.q.double().numpy()
    q_abs = np.zeros((1, T, H, 576))
    for h in range(H):
        rows, signs = pk[h]
        q_abs[0, :, h, rows] = (qf[:, h, :128] * signs).T
        q_abs[0, :, h, 512:] = qf[:, h, 128:]
    qa = torch.from_numpy(q_abs).to(torch.bfloat16)
    assert np.array_equal(qa.double().numpy(), q_abs)  # exact in bf16
    absorbed = W.MlaInputs("abs", m.cache.pool, m.cache.page_table, m.cache.seq_lens, qa,
                           m.cache.kv_scale, m.cache.sm_scale, m.cache.page_size)
    out_a, lse_a = orc.attention(absorbed)
    for h in range(H):
        rows, signs = pv[h]
        np.testing.assert_allclose(out[:, h], out_a[0, :, h][:, rows] * signs, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(lse, lse_a[0], rtol=1e-12)


def pin_mha_zero_query(orc):
    """q = 0: every visible key weighs the same, so out = the mean of the visible values and
    lse = ln(#visible); position t of T sees L - T + t + 1 keys."""
    m = W.mha_prefill_inputs(4, 37, H=2, seed=22)
    q0 = torch.zeros_like(m.q)
    out, lse = orc.mha_prefill_rows(m.cache, q0, m.w_ukv)
    L, T = 41, 4
    kv = np.zeros((L, 576))
    table = np.array([orc.e4m3_value(c) for c in range(256)]) * m.cache.kv_scale
    pt = m.cache.page_table[0].numpy()
    P = m.cache.page_size
    for n in range(L):
        kv[n] = table[m.cache.pool[pt[n // P], n % P].numpy()]
    Wf = m.w_ukv.double().numpy()
    for t in range(T):
        vis = L - T + t + 1
        for h in range(2):
            v = kv[:vis, :512] @ Wf[:, h, 128:]
            np.testing.assert_allclose(out[t, h], v.mean(axis=0), rtol=1e-10, atol=1e-13)
            assert abs(lse[t, h] - math.log(vis)) < 1e-12


def pin_mha_sdpa(orc):
    """Against torch's float64 scaled_dot_product_attention with an explicit bottom-right
    causal mask, on keys and values built with torch (einsum) from the same codes."""
    m = W.mha_prefill_inputs(6, 90, H=3, seed=23)
    out, lse = orc.mha_prefill_rows(m.cache, m.q, m.w_ukv)
    L, T, H = 96, 6, 3
    codes = torch.stack([m.cache.pool[m.cache.page_table[0, n // 64], n % 64] for n in range(L)])
    vals = codes.view(torch.float8_e4m3fn).to(torch.float64) * m.cache.kv_scale
    Wf = m.w_ukv.double()
    K = torch.cat([torch.einsum("nd,dhk->hnk", vals[:, :512], Wf[:, :, :128]),
                   vals[None, :, 512:].expand(H, L, 64)], dim=2)
    V = torch.einsum("nd,dhk->hnk", vals[:, :512], Wf[:, :, 128:])
    q = m.q.double().permute(1, 0, 2)
    mask = torch.arange(L)[None, :] <= (L - T + torch.arange(T))[:, None]
    ref = F.scaled_dot_product_attention(q, K, V, attn_mask=mask, scale=m.cache.sm_scale)
    np.testing.assert_allclose(out, ref.permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-12)
    rows = np.array([[5, 2], [0, 0], [3, 1]])
    o, l = orc.mha_prefill_rows(m.cache, m.q, m.w_ukv, rows)
    for i, (t, h) in enumerate(rows):  # (BLAS may block a different row count differently)
        np.testing.assert_allclose(o[i], out[t, h], rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(l[i], lse[t, h], rtol=1e-14)


def pin_attention_sink_closed_form(orc):
    """A long row with one dominant key over a flat tail, in closed form: on the even heads
    of the attention-sink input (query zero on dims 0..511, every RoPE dim equal to a), each
    tail key scores exactly 0 and the sink s = sm_scale * 64 * a * 448 * kv_scale, so
    lse = ln(L - 1 + e^s) and out = (sum of the tail's values + e^s v_sink) / (L - 1 + e^s).
    Computed here from the codes with torch's float8 decode, in float64; causal verify rows
    see the same keys up to their own position."""
    L = 5000
    for n_q in (1, 3):
        inp = W.attention_sink(L=L, H=4, n_q=n_q, seed=11, sink_at=1234)
        out, lse = orc.attention(inp)
        codes = _gather_keys(inp, 0)
        vals = codes.view(torch.float8_e4m3fn).double() * inp.kv_scale
        for h in (0, 2):
            a = inp.q[0, 0, h, W.ROPE0].double().item()
            assert torch.all(inp.q[0, :, h, :W.ROPE0] == 0)
            s = inp.sm_scale * 64 * a * 448.0 * inp.kv_scale
            for j in range(n_q):
                vis = L - n_q + j + 1
                tail = vals[:vis, :DV].sum(0) - vals[1234, :DV]
                den = (vis - 1) + math.exp(s)
                want = (tail + math.exp(s) * vals[1234, :DV]) / den
                assert abs(lse[0, j, h] - math.log(den)) < 1e-12 * max(1.0, abs(math.log(den)))
                assert np.allclose(out[0, j, h], want.numpy(), rtol=1e-11, atol=1e-13)


ALL_PINS = [
    pin_e4m3_all_codes, pin_bf16, pin_brute_force_sdpa, pin_constant_v, pin_single_key,
    pin_zero_query, pin_duplicate_key, pin_split_merge, pin_merge_weights, pin_permuted_pages,
    pin_head_padding_and_permutation, pin_causal_prefix, pin_sampled_rows, pin_e4m3_encode,
    pin_cache_append, pin_top_k_renorm, pin_attention_sink_closed_form, pin_mha_absorbed_identity, pin_mha_zero_query,
    pin_mha_sdpa,
]
