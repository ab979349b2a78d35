"""Run and time one stage of the decode layer on a synthetic workload.

    python -m sparse_attention_decode_kpool_gb300.stage_bench --workload 3 \\
        --seq-len 16384 --stage attend --iters 3

Stages: compress, score, select, expand, attend, project, step. ``--rows`` shrinks
the prefill chunk (workload 4), ``--seq-len`` the long-context sequences (workload
3); ``--always-select-tail`` widens the index rows by the trailing partial pool;
``--latent-fp8`` gives attention the FP8 latent cache.
Each iteration is preceded by a write-then-read of 256 MiB so that the stage
starts from a cold L2; the median of the CUDA-event times is printed as one JSON
line. Meant for profiler runs (a fixed, small number of launches of one stage)."""
from __future__ import annotations

import argparse
import dataclasses
import json

import torch

from . import workloads as W
from .pipeline import DsaDecodeLayer

STAGES = ("compress", "score", "select", "expand", "attend", "project", "step")


def make(workload: int, seq_len=None, rows=None):
    kw = {}
    if seq_len is not None:
        if workload != 3:
            raise SystemExit("--seq-len applies to workload 3")
        kw["seq_len"] = seq_len
    if rows is not None:
        if workload != 4:
            raise SystemExit("--rows applies to workload 4")
        kw["rows"] = rows
    return W.WORKLOADS[workload](**kw)


def main(argv=None) -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", type=int, default=3)
    ap.add_argument("--seq-len", type=int, default=None)
    ap.add_argument("--rows", type=int, default=None)
    ap.add_argument("--stage", choices=STAGES, default="step")
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=1)
    ap.add_argument("--always-select-tail", action="store_true")
    ap.add_argument("--latent-fp8", action="store_true")
    args = ap.parse_args(argv)

    wl = make(args.workload, args.seq_len, args.rows)
    if args.always_select_tail:
        wl.geom = dataclasses.replace(wl.geom, always_select_tail=True)
    layer = DsaDecodeLayer(wl, latent_fp8=args.latent_fp8)
    layer.compress()
    layer.step()  # every stage's inputs exist from here on
    torch.cuda.synchronize()
    flush_w = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    flush_r = torch.ones(64 << 20, dtype=torch.float32, device="cuda")
    fn = getattr(layer, args.stage)
    times = []
    for i in range(args.warmup + args.iters):
        flush_w.zero_()
        flush_r.sum()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        b.synchronize()
        if i >= args.warmup:
            times.append(a.elapsed_time(b) * 1e3)
    times.sort()
    st = int(layer.status.item())
    print(json.dumps({"workload": wl.name, "stage": args.stage, "iters": args.iters,
                      "us_median": round(times[len(times) // 2], 2), "status": st}))
    if st:
        raise SystemExit(f"device status {st}")


if __name__ == "__main__":
    main()
