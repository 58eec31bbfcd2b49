"""Run a few verify calls on one preset workload (a target for profilers).

    python -m speculative_decoding_verification_36_gb300.run_case c4 [--batch B] [--calls N]

Builds the library if needed, generates the preset's synthetic inputs on
cuda:0 and makes N calls of the entry point the preset exercises
(spec_verify for c1-c4, or spec_verify_early_exit with --early-exit;
spec_tree_verify_greedy for c5, its early exit with --early-exit;
spec_tree_verify_sampling at tau = 1 on the
c5 tree for c5s; spec_ngram_draft (n 1..4, K = 8) on 256 repetitive
histories of up to 131072 tokens for ngram), then synchronises.
"""
from __future__ import annotations

import argparse
import sys


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("preset", choices=["c1", "c2", "c3", "c4", "c5", "c5s", "ngram"])
    ap.add_argument("--early-exit", action="store_true", help="c1-c5: the early-exit verify")
    ap.add_argument("--batch", type=int, default=0, help="sequences (default: the preset's B)")
    ap.add_argument("--calls", type=int, default=3)
    args = ap.parse_args(argv)

    import torch

    from . import build, spec_get_status, spec_ngram_draft, spec_tree_verify_greedy, spec_tree_verify_sampling
    from . import spec_verify, spec_verify_early_exit
    from . import workloads as wl

    build.build()
    dev = torch.device("cuda", 0)
    if args.preset == "ngram":
        B, L = args.batch or 256, 131072
        h = wl.make_ngram_histories(16, L, seed=1)
        reps = (B + 15) // 16
        tok = h["tokens"].repeat(reps, 1)[:B].contiguous().to(dev)
        ln = h["lengths"].repeat(reps)[:B].contiguous().to(dev)
        for _ in range(args.calls):
            spec_ngram_draft(tok, ln, 1, 4, 8)
        torch.cuda.synchronize()
        flags = spec_get_status()
        print(f"ngram B={B} L<={L}: {args.calls} calls, status flags {flags}")
        return 0 if flags == 0 else 1
    name = "c5" if args.preset == "c5s" else args.preset
    p = wl.preset(name, B=args.batch) if args.batch else wl.preset(name)
    if args.preset == "c5s":
        x = wl.make_tree_sampling(p, 1.0, device=dev, seed=0)
        for i in range(args.calls):
            spec_tree_verify_sampling(x["target"], x["draft"], x["tokens"], x["parents"], 1.0, i)
    elif args.preset == "c5":
        x = wl.make_tree(p, device=dev, seed=0)
        for _ in range(args.calls):
            spec_tree_verify_greedy(x["target"], x["tokens"], x["parents"], early_exit=args.early_exit)
    else:
        x = wl.make_chain(p, device=dev, seed=0)
        verify = spec_verify_early_exit if args.early_exit else spec_verify
        for i in range(args.calls):
            verify(x["target"], x["draft"], x["tokens"], x["temperature"], i)
    torch.cuda.synchronize()
    flags = spec_get_status()
    print(f"{args.preset} B={p.B}: {args.calls} calls, status flags {flags}")
    return 0 if flags == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
