"""Run and time one stage of the decode layer on a synthetic workload.

    python -m sparse_attention_decode_kpool_gb300.stage_bench --workload 3 \\
        --seq-len 16384 --stage attend --iters 3

Stages: compress, score, select, expand, attend, project, step, append, frontend,
quantize. ``--rows`` shrinks the prefill chunk (workload 4), ``--seq-len`` the
long-context sequences (workload 3) or caps the paged lengths (workload 2);
``--always-select-tail`` widens the index rows by the trailing partial pool;
``--latent-fp8`` gives attention the FP8 latent cache. Workload 5 is a contiguous
batch of ``--batch`` sequences of ``--seq-len`` tokens whose geometry ``--geom
key=value`` overrides (e.g. index_heads=64, hidden=96). ``--unfused`` runs expand
and append as separate calls; ``--select-kernel``, ``--mla-kernel`` and
``--project-kernel`` force a kernel through dsa_set_option.
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

STAGES = ("compress", "score", "select", "expand", "attend", "project", "step", "append",
          "frontend", "quantize")


def _custom(seq_len, batch, geom):
    base = dict(W.GLM53)
    for kv in geom:
        k, v = kv.split("=", 1)
        base[k] = type(base.get(k, 0))(v) if k in base else int(v)
    S = seq_len or 16384
    return W.make_workload(f"custom-b{batch}-S{S}", 5, W.Geometry(**base), [S] * batch,
                           invalid_per_seq=S // 100)


def make(workload: int, seq_len=None, rows=None, batch=8, geom=()):
    if workload == 5:
        return _custom(seq_len, batch, geom)
    kw = {}
    if seq_len is not None and workload == 2:
        wl = W.paged_batch()
        lens = [min(int(L), seq_len) for L in wl.seq_lens]
        return W.make_workload(f"paged-decode-b64-L4k-{seq_len}", 2, wl.geom, lens,
                               block_size=64, max_seq_len=(seq_len + 63) // 64 * 64)
    if seq_len is not None:
        if workload != 3:
            raise SystemExit("--seq-len applies to workloads 2, 3 and 5")
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
    ap.add_argument("--batch", type=int, default=8)
    ap.add_argument("--geom", action="append", default=[])
    ap.add_argument("--unfused", action="store_true")
    ap.add_argument("--select-kernel", choices=("merge", "radix"), default=None)
    ap.add_argument("--mla-kernel", choices=("auto", "tcgen05", "mma", "cluster"), default=None)
    ap.add_argument("--project-kernel", choices=("auto", "tcgen05", "mma"), default=None)
    args = ap.parse_args(argv)

    from . import api
    if args.select_kernel:
        api.select_kernel(args.select_kernel).__enter__()
    if args.mla_kernel:
        api.mla_kernel(args.mla_kernel).__enter__()
    if args.project_kernel:
        api.project_kernel(args.project_kernel).__enter__()
    wl = make(args.workload, args.seq_len, args.rows, args.batch, args.geom)
    if args.always_select_tail:
        wl.geom = dataclasses.replace(wl.geom, always_select_tail=True)
    kw = {}
    if args.stage == "append":  # room for every appended token
        import numpy as np
        kw["decode_from"] = np.maximum(wl.seq_lens.astype(np.int64) - 4 * (args.iters + 2), 0)
        kw["fuse_append"] = not args.unfused
    if args.stage == "frontend":
        kw["frontend"] = W.make_frontend(wl.geom, wl.rows, seed=wl.seed + 100)
    layer = DsaDecodeLayer(wl, latent_fp8=args.latent_fp8, fuse_expand=not args.unfused, **kw)
    layer.compress()
    if args.stage == "append":
        layer.stage(0)
    if args.stage == "frontend":
        layer.frontend()
    layer.step()  # every stage's inputs exist from here on
    torch.cuda.synchronize()
    if args.stage == "quantize":
        if layer.ckv_codes is None:
            raise SystemExit("--stage quantize needs --latent-fp8")
        layer.quantize = lambda: api.dsa_quantize_latent(layer.ckv, layer.ckv_codes,
                                                          layer.ckv_scales)
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
