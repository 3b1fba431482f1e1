"""Runs one named workload's hot path a few times on the current GPU and prints the
per-pass device time of each call.  Meant as the target of a profiler command, e.g.

    ncu --set full --clock-control none -k regex:k_prefill_tc -s 2 -c 1 \\
        python -m relative_bias_hybrid_gb300.run swa --iters 3

Every pass is the whole path (prologue, then prefill or decode + combine) on seeded
synthetic inputs already resident on the device, optionally with the qkvr projections
(their own inputs and outputs) before it and the attention-output conv after it.
``--seqs N`` keeps only the first N sequences of a batched workload (a smaller case of the
same kernel, for captures that must hold less memory).
"""
from __future__ import annotations

import argparse
import dataclasses

import torch

from . import inputs as gen
from .step import AttentionStep, OutputConvStep, QkvrStep


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("workload", choices=["tiny", "swa", "full", "decode", "ragged"])
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--seqs", type=int, default=0, help="keep only the first N sequences")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--splits", type=int, default=0, help="decode splits (0 = the library's heuristic)")
    ap.add_argument("--kv", choices=["bf16", "e4m3"], default="bf16", help="KV-cache element type")
    ap.add_argument("--output-conv", action="store_true",
                    help="also run the attention-output conv (hidden width Hq * 128) after each pass")
    ap.add_argument("--qkvr", action="store_true",
                    help="also run the qkvr projections with the prologue fused in (hidden width "
                         "Hq * 128) before each pass")
    args = ap.parse_args(argv)

    w = gen.workload(args.workload)
    if args.seqs > 0 and args.seqs < w.B:
        w = dataclasses.replace(w, name=f"{w.name}[:{args.seqs}]", q_lens=w.q_lens[:args.seqs],
                                prefix_lens=w.prefix_lens[:args.seqs])
    dev = torch.device("cuda", torch.cuda.current_device())
    x = gen.make_inputs(w, seed=args.seed, device=dev, kv_dtype=args.kv)
    step = AttentionStep(w, x, mode="decode" if args.workload == "decode" else "prefill",
                         num_splits=args.splits)
    oc = OutputConvStep(w, gen.make_output_conv_inputs(w, seed=args.seed, device=dev)) if args.output_conv else None
    qk = (QkvrStep(w, gen.make_qkvr_inputs(w, w.Hq * w.head_dim, seed=args.seed, device=dev, kv_dtype=args.kv))
          if args.qkvr else None)
    stream = torch.cuda.Stream(device=dev)
    print(w.describe(), f"num_splits={step.num_splits}" if step.mode == "decode" else "")
    with torch.cuda.stream(stream):
        for it in range(args.iters):
            e = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
            e[4].record(stream)
            if qk is not None:
                qk.run(stream)
            e[0].record(stream)
            step.run_prologue(stream)
            e[1].record(stream)
            step.run_attention(stream)
            e[2].record(stream)
            if oc is not None:
                oc.run(stream)
            e[3].record(stream)
            stream.synchronize()
            print(f"pass {it}: " + (f"qkvr {e[4].elapsed_time(e[0]):.4f} ms, " if qk is not None else "")
                  + f"prologue {e[0].elapsed_time(e[1]):.4f} ms, "
                  f"attention {e[1].elapsed_time(e[2]):.4f} ms"
                  + (f", output conv {e[2].elapsed_time(e[3]):.4f} ms" if oc is not None else ""))
    status = (step.device_status() | (oc.device_status() if oc is not None else 0)
              | (qk.device_status() if qk is not None else 0))
    print(f"device status {status}")
    if status != 0:
        raise SystemExit(1)


if __name__ == "__main__":
    main()
