"""Run one stage of the round in isolation (for ncu captures and timing).

python -m history_free_speculative_gb300.profile_stage --stage lm_head --workload qwen3-8b-b32 [--iters N]

Stages: lm_head (tensor-core LM head + merge), seq_head (head products + chain),
backbone (staging + L_D layers), round (draft + verify). The caller's weight
copy is released after the handle is created, so the device holds one copy
of the weights plus the workspace. Prints the CUDA-event time per iteration.
"""
import argparse
import json
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from history_free_speculative_gb300 import binding  # noqa: E402
from history_free_speculative_gb300 import workload as wk  # noqa: E402


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--stage", default="lm_head", choices=["lm_head", "seq_head", "backbone", "round"])
    ap.add_argument("--workload", default="qwen3-8b-b32", choices=sorted(wk.WORKLOADS))
    ap.add_argument("--B", type=int, default=None)
    ap.add_argument("--iters", type=int, default=3)
    args = ap.parse_args()
    dev = "cuda:0"
    wl = wk.WORKLOADS[args.workload]
    cfg = wl.cfg
    B = args.B or wl.B
    T = wl.temperature
    W = wk.make_weights(cfg, wl.weight_seed, device=dev)
    dr = binding.Drafter(cfg, W, B_max=B)
    del W
    torch.cuda.empty_cache()
    hidden, anchor, pos = wk.make_round_inputs(wl, B=B, device=dev)
    out = dr.new_outputs(B, dev)
    g = torch.Generator(device=dev).manual_seed(5)
    hs = torch.randn(B, cfg.K, cfg.D, generator=g, device=dev)
    b = torch.empty(B, cfg.K, cfg.D, device=dev)
    probs = wk.make_target_probs(B, cfg.K, cfg.V, wl.rng_seed, device=dev) if T > 0 else None
    tgt = torch.randint(0, cfg.V, (B, cfg.K + 1), generator=g, device=dev, dtype=torch.int32)

    def run():
        if args.stage == "lm_head":
            dr.lm_head(hs, T, wl.rng_seed, pos, out["cand"], out["qstats"])
        elif args.stage == "seq_head":
            dr.seq_head(hs, b)
        elif args.stage == "backbone":
            dr.backbone(hidden, anchor, b)
        else:
            dr.draft_round(hidden, anchor, T, wl.rng_seed, pos, out["cand"], out["qstats"])
            if T > 0:
                dr.verify_sample(out["cand"], out["qstats"], None, probs, T, wl.rng_seed, pos,
                                 out["accepted"], out["commits"], out["n_commit"], out["next_anchor"])
            else:
                dr.verify(out["cand"], tgt, out["accepted"], out["commits"], out["n_commit"],
                          out["next_anchor"])

    times = []
    for _ in range(args.iters):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        run()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    rc, st = dr.device_status()
    print(json.dumps({"stage": args.stage, "workload": wl.name, "B": B, "ms": [round(t, 4) for t in times],
                      "status": st}))
    dr.close()
    sys.exit(0 if rc == 0 else 1)


if __name__ == "__main__":
    main()
