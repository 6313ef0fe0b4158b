"""A small, self-contained run of one workload for profilers (ncu): the full
shapes of a configuration with fewer layers, a few steps, nothing else.

  python -m paged_kv_decode_pages_gb300.profile_case --workload long_context \
      --layers 2 --steps 3

A prefill / mixed-step workload (mixed_qwen3_4b, prefill_qwen3_4b_p128) runs
its append + tensor-core attention per layer instead.
"""
from __future__ import annotations

import argparse


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="long_context")
    ap.add_argument("--layers", type=int, default=2)
    ap.add_argument("--steps", type=int, default=3)
    args = ap.parse_args(argv)

    import torch
    from . import load
    from .step import DecodeStep, PrefillStep
    from .workloads import (CONFIGS, PREFILL_CONFIGS, PrefillTensors, Tensors, make_batch,
                            make_prefill_batch)

    load()
    if args.workload in PREFILL_CONFIGS:
        cfg = PREFILL_CONFIGS[args.workload]
        batch = make_prefill_batch(cfg)
        step = PrefillStep(batch, PrefillTensors(batch, device="cuda", layers=args.layers))
        for _ in range(args.steps):
            step.run()
        torch.cuda.synchronize()
        err = int(step.err.item())
        print("profile_case %s: %d layers x %d steps, err=%d"
              % (cfg.name, args.layers, args.steps, err))
        return 1 if err else 0
    cfg = CONFIGS[args.workload]
    batch = make_batch(cfg)
    tensors = Tensors(batch, device="cuda", layers=args.layers)
    step = DecodeStep(batch, tensors)
    for _ in range(args.steps):
        step.run()
    torch.cuda.synchronize()
    err = int(step.err.item())
    print("profile_case %s: %d layers x %d steps, err=%d" % (cfg.name, args.layers, args.steps, err))
    return 1 if err else 0


if __name__ == "__main__":
    raise SystemExit(main())
