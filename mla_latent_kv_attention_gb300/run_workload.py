"""Run one named seeded workload through the C ABI a few times (for profilers).

    python -m mla_latent_kv_attention_gb300.run_workload batched_paged_decode --iters 5
    python -m mla_latent_kv_attention_gb300.run_workload causal_prefill --T 2048 --iters 3
    python -m mla_latent_kv_attention_gb300.run_workload cache_append --iters 5
    python -m mla_latent_kv_attention_gb300.run_workload top_k_renorm --iters 5

Prints the device status word after the last call. Intended as the command line that
ncu wraps: every launch it makes is a library launch on the named inputs.
"""
from __future__ import annotations

import argparse
import sys

import torch

import mla_latent_kv_attention_gb300 as mla
from mla_latent_kv_attention_gb300 import workloads as W


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("workload", choices=sorted(W.WORKLOADS) + ["cache_append", "top_k_renorm",
                                                                 "mha_prefill"])
    ap.add_argument("--iters", type=int, default=5)
    ap.add_argument("--heads", type=int, default=12, help="long_history_decode only")
    ap.add_argument("--T", type=int, default=8192, help="causal_prefill and mha_prefill only")
    ap.add_argument("--bf16", action="store_true", help="mha_prefill only: the all-bf16 form")
    args = ap.parse_args(argv)
    if args.workload == "cache_append":
        return _cache_append(args.iters)
    if args.workload == "mha_prefill":
        return _mha_prefill(args.T, args.iters, args.bf16)
    if args.workload == "top_k_renorm":
        return _top_k_renorm(args.iters)
    if args.workload == "long_history_decode":
        inp = W.long_history_decode(args.heads)
    elif args.workload == "causal_prefill":
        inp = W.causal_prefill(T=args.T)
    else:
        inp = W.WORKLOADS[args.workload]()
    kv = mla.KVCache.from_inputs(inp, "cuda")
    if args.workload == "causal_prefill":
        q = inp.q[0].contiguous().cuda()
        ws = mla.workspace(mla.MLA_OP_PREFILL, 1, inp.H, inp.n_q)
        for _ in range(args.iters):
            mla.mla_prefill(kv, q, inp.sm_scale, ws=ws)
    else:
        q = inp.q.contiguous().cuda()
        ws = mla.workspace(mla.MLA_OP_VERIFY, inp.B, inp.H, inp.n_q)
        for _ in range(args.iters):
            if inp.n_q == 1:
                mla.mla_decode(kv, q[:, 0].contiguous(), inp.sm_scale, ws=ws)
            else:
                mla.mla_verify(kv, q, inp.sm_scale, ws=ws)
    torch.cuda.synchronize()
    status = mla.mla_read_status(ws)
    print(f"{args.workload}: {args.iters} calls, status {mla.STATUS.get(status, status)}")
    return 0 if status == 0 else 1


def _cache_append(iters: int) -> int:
    """8,192 bf16 rows (a prefill chunk) into a 302 MB pool of 64-position pages at random
    slots, a different slot set each call."""
    g = torch.Generator().manual_seed(7)
    pool = torch.zeros(8192, 64, mla.MLA_D, dtype=torch.uint8, device="cuda")
    x = torch.randn(8192, mla.MLA_D, generator=g).to(torch.bfloat16).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for i in range(iters):
        slots = torch.randperm(pool.shape[0] * 64, generator=g)[:8192].cuda()
        mla.mla_cache_append(pool, x, slots, 0.0125, status=status)
    torch.cuda.synchronize()
    st = int(status.item())
    print(f"cache_append: {iters} calls, status {mla.STATUS.get(st, st)}")
    return 0 if st == 0 else 1


def _mha_prefill(T: int, iters: int, bf16: bool = False) -> int:
    """The causal prefill chunk (T new positions on a 32,768 prefix, 12 heads) in the MHA form
    (the default form, or the all-bf16 one)."""
    m = W.mha_prefill(T=T)
    kv = mla.KVCache.from_inputs(m.cache, "cuda")
    q = m.q.cuda()
    w = m.w_ukv.cuda()
    L = int(m.cache.seq_lens[0])
    ws = torch.zeros(mla.library().mla_prefill_mha_workspace_size(L, m.H, 0), dtype=torch.uint8,
                     device="cuda")
    for _ in range(iters):
        mla.mla_prefill_mha(kv, q, w, m.cache.sm_scale, L=L, ws=ws, bf16=bf16)
    torch.cuda.synchronize()
    status = mla.mla_read_status(ws)
    print(f"mha_prefill: {iters} calls, status {mla.STATUS.get(status, status)}")
    return 0 if status == 0 else 1


def _top_k_renorm(iters: int) -> int:
    """32 probability rows over a 129,280-entry vocabulary, k drawn per row in [1, 1024)."""
    g = torch.Generator().manual_seed(1)
    probs = torch.softmax(torch.randn(32, 129280, generator=g) * 3, dim=1).cuda()
    ks = torch.randint(1, 1024, (32,), generator=g, dtype=torch.int32).cuda()
    out = torch.empty_like(probs)
    for _ in range(iters):
        mla.mla_top_k_renorm_prob(probs, ks, out=out)
    torch.cuda.synchronize()
    ok = bool(torch.isfinite(out).all().item())
    print(f"top_k_renorm: {iters} calls, {'finite' if ok else 'NON-FINITE'} output")
    return 0 if ok else 1


if __name__ == "__main__":
    sys.exit(main())
