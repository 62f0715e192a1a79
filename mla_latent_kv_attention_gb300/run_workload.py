"""Run one named seeded workload through the C ABI a few times (for profilers).

    python -m mla_latent_kv_attention_gb300.run_workload batched_paged_decode --iters 5
    python -m mla_latent_kv_attention_gb300.run_workload causal_prefill --T 2048 --iters 3

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
    ap.add_argument("workload", choices=sorted(W.WORKLOADS))
    ap.add_argument("--iters", type=int, default=5)
    ap.add_argument("--heads", type=int, default=12, help="long_history_decode only")
    ap.add_argument("--T", type=int, default=8192, help="causal_prefill only")
    args = ap.parse_args(argv)
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


if __name__ == "__main__":
    sys.exit(main())
