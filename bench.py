"""Benchmark: DSA decode queries/s at 262,144-token context on one GB300 (or N
independent replicas), with the HBM roofline fraction of the dominant stage.

One step = one decode query per sequence for the whole batch: score -> select ->
expand -> sparse latent MLA (split attention, combine, o_absorb projection), as a
CUDA-graph replay of the four C-ABI calls. Inputs are resident in HBM; L2 is
flushed (a 256 MiB write) between timed steps, outside the timed events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload 3] [--no-cpu-baseline] [--no-e2e] [--always-select-tail]
                  [--decode-append] [--latent-fp8] [--frontend [--q-lora-rank Q]]

--impl reference times the CPU oracle (the plain float64 restatement of the
method) on the host, one query row per step, single-threaded.
"""
from __future__ import annotations

import os

# The CPU oracle is timed single-threaded: hold numpy's BLAS to one thread before
# numpy loads.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import ctypes
import dataclasses
import json
import platform
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_attention_decode_kpool_gb300 import workloads as W  # noqa: E402

METRIC = "DSA decode queries/s (select + sparse MLA) at 262K ctx; % of HBM roofline"
PREFILL_METRIC = ("DSA chunked-prefill query rows/s (tensor-core index scores + select + expand "
                  "+ sparse latent attention to olat); % of bf16 tensor peak")
PREFILL_WORKLOAD = 4  # scored on the tensor cores; the o_absorb GEMM is not in its step

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of a stage's
# kernels, from one ncu capture of the current kernels; a stage not listed, or whose
# kernels changed since the capture, reports null. The projection reads all of
# o_absorb whatever the context length, so its capture at 8 rows of a 32,768-token
# context holds for the 262,144-token workload.
MEASURED_TRAFFIC = {
    "project": (268_993_280 + 2_810_368,
                "ncu dram__bytes_read.sum + dram__bytes_write.sum of project_tc_kernel<16, 1, 8> "
                "(8 rows, S=32,768: the o_absorb stream does not depend on S)"),
}
FLUSH_BYTES = 256 << 20


# ---------------------------------------------------------------------------
# distributed plumbing (replicas: no data-path collective)


def dist_init(gpus: int):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return ws, rank, local


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region (NVML read-only queries)


class ClockSampler:
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x2: "applications_clocks_setting", 0x1: "gpu_idle"}

    def __init__(self, device: torch.device, period_s: float = 0.005):
        self.samples, self.reasons, self.max_mhz = [], set(), None
        self.period = period_s
        self._stop = threading.Event()
        self._nvml = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            h = ctypes.c_void_p()
            p = torch.cuda.get_device_properties(device)
            bus = "%08x:%02x:%02x.0" % (getattr(p, "pci_domain_id", 0), p.pci_bus_id,
                                        p.pci_device_id)
            if nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
                raise OSError("no NVML handle for " + bus)
            self._nvml, self._h = nv, h
            self._reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:  # NVML_CLOCK_SM
                self.max_mhz = int(mx.value)
        except (OSError, AttributeError):
            self._nvml = None

    def _run(self):
        nv, h = self._nvml, self._h
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                self.samples.append(int(clk.value))
            if self._reasons_fn(h, ctypes.byref(rs)) == 0:
                for bit, name in self.REASONS.items():
                    if rs.value & bit:
                        self.reasons.add(name)
            time.sleep(self.period)

    def __enter__(self):
        if self._nvml is not None:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *a):
        if self._nvml is not None:
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                    "samples": 0}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons - {"gpu_idle"}), "samples": len(self.samples)}


# ---------------------------------------------------------------------------
# algorithmic bytes (the roofline numerator)


def algorithmic_bytes(wl, layer) -> dict:
    """Per step: pooled keys of candidate pools + pool flags, indexer q and w,
    selected latent rows, absorbed Q, o_absorb once, the output."""
    g = wl.geom
    pv = layer.pool_valid
    ctx = layer.row_ctx.cpu().numpy()  # the live context (it grows under --decode-append)
    # candidate pools of each row = valid pools among those visible to the row
    cand = 0
    if wl.paged:
        cand = int(pv.sum().item())  # decode rows see all their complete pools
    else:
        for r in range(wl.rows):
            b = int(wl.row_seq[r])
            nvis = max(0, (int(ctx[r]) - g.first_key) // g.index_kpool)
            cand += int(pv[b, :nvis].sum().item())
    flags = sum(max(0, (int(ctx[r]) - g.first_key) // g.index_kpool) for r in range(wl.rows))
    keys = cand * g.index_head_dim * 2
    q = wl.rows * g.index_heads * (g.index_head_dim * 2 + 4)
    sel_tokens = int((layer.token_ids >= 0).sum().item())
    # a gathered latent row: bf16, or E4M3 codes plus one f32 scale per 128 channels
    row_bytes = (g.kv_lora_rank + g.kv_lora_rank // 128 * 4 if layer.latent_fp8
                 else g.kv_lora_rank * 2)
    latent = sel_tokens * row_bytes
    qlat = wl.rows * g.heads * g.kv_lora_rank * 2
    oabs = g.hidden * g.heads * g.kv_lora_rank * 2 if layer.o_absorb is not None else 0
    y = wl.rows * g.hidden * 2 if layer.o_absorb is not None else 0
    # the projection's input: the bf16 copy of olat the combine writes for it
    olat = wl.rows * g.heads * g.kv_lora_rank * 2 if layer.o_absorb is not None else 0
    # --decode-append: per sequence the staged rows in and out, the valid byte, and
    # at most one newly whole pool (kpool token rows of keys, gates and flags in,
    # one pooled key and flag out).
    app = 0
    if layer.decode_from is not None:
        ihd, kp = g.index_head_dim, g.index_kpool
        # the latent row goes out as bf16, or (FP8 cache) as codes and scales
        ckv_out = (g.kv_lora_rank + g.kv_lora_rank // 128 * 4 if layer.latent_fp8
                   else g.kv_lora_rank * 2)
        app = wl.batch * ((2 * ihd + g.kv_lora_rank) * 2 + 2 * ihd * 2 + ckv_out + 1
                          + kp * (2 * ihd * 2 + 1) + ihd * 2 + 1)
    # --frontend: every front-end weight once, the hidden state in, and its outputs
    # (qlat, qidx, w, the staged rows) out.
    fe = 0
    if layer.fe is not None:
        wts = (layer.w_x, layer.w_q, layer.q_a_norm, layer.kv_a_norm)
        fe = sum(t.numel() * t.element_size() for t in wts)
        fe += layer.x.numel() * 2 + qlat + q
        fe += wl.rows * (2 * g.index_head_dim + g.kv_lora_rank) * 2
    return {"score": keys + flags + q, "attend": latent + qlat, "project": oabs + olat + y,
            "append": app, "frontend": fe,
            "total": keys + flags + q + latent + qlat + oabs + y + app + fe,
            "selected_tokens": sel_tokens, "candidate_pools": cand}


def compress_bytes(wl, seq_lens) -> int:
    """dsa_compress over the given context lengths: raw keys, gate logits and validity
    of every token in; one pooled key and flag per whole pool out."""
    g = wl.geom
    ihd, kp = g.index_head_dim, g.index_kpool
    toks = int(np.sum(seq_lens))
    pools = int(sum(max(0, (int(L) - g.first_key) // kp) for L in seq_lens))
    return toks * (2 * ihd * 2 + 1) + pools * (ihd * 2 + 1)


def cpu_info() -> dict:
    """The host's CPU model and thread count (for the CPU baseline's label)."""
    model = None
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except OSError:
        pass
    if model is None:
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                if line.strip().lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    return {"cpu_model": model or platform.machine(), "nproc": os.cpu_count()}


def algorithmic_flops(wl, layer) -> dict:
    """Per step of the prefill chunk: the dense index-score contraction over every
    pool of the row stride (2 * rows * heads * p_stride * ihd) and the sparse
    attention over the selected tokens (QK and PV: 4 * heads * 512 per token)."""
    g = wl.geom
    sel_tokens = int((layer.token_ids >= 0).sum().item())
    score = 2.0 * wl.rows * g.index_heads * wl.p_stride * g.index_head_dim
    attend = 4.0 * g.heads * g.kv_lora_rank * sel_tokens
    return {"score": score, "attend": attend, "total": score + attend,
            "selected_tokens": sel_tokens}


# ---------------------------------------------------------------------------
# CPU oracle timing (the cpu_baseline leg and the reference arm)


class OracleRunner:
    """Times the oracle's decode_row on rows of the workload. The oracle's own
    pooled-key cache of a sequence is built once, untimed (it is layer state)."""

    def __init__(self, wl, with_project: bool = True, latent_fp8: bool = False):
        from oracle import dsa_oracle as O

        self.O, self.wl = O, wl
        self.with_project = with_project
        self.latent_fp8 = latent_fp8
        self._pools = {}
        self._A = None

    def _tokens(self, t: torch.Tensor, b: int) -> np.ndarray:
        """Logical rows of sequence b of a cache, gathered on the raw bits and only
        then widened (the whole 262K-token latent cache would be 4 GiB as f32)."""
        wl = self.wl
        bt = None if wl.block_table is None else wl.block_table.numpy()
        raw = t.view(torch.int16).numpy() if t.dtype == torch.bfloat16 else t.numpy()
        rows = self.O.sequence_tokens(raw, b, int(wl.seq_lens[b]), bt, wl.block_size or 0)
        if t.dtype == torch.bfloat16:
            return torch.from_numpy(np.ascontiguousarray(rows)).view(torch.bfloat16).float().numpy()
        return rows

    def _prep(self, r: int):
        O, wl, g = self.O, self.wl, self.wl.geom
        b = int(wl.row_seq[r])
        if b not in self._pools:
            f = lambda t: t.float().numpy().astype(np.float64)
            keys, pv, _ = O.kpool_compress(self._tokens(wl.k_raw, b), self._tokens(wl.gate, b),
                                           self._tokens(wl.valid, b), wl.ape.numpy(), f(wl.ln_w),
                                           f(wl.ln_b), g.eps, g.first_key, g.index_kpool)
            ckv = self._tokens(wl.ckv, b)
            if self.latent_fp8:  # the FP8 cache, encoded and decoded once (layer state)
                ckv = O.dequantize_latent_fp8(*O.quantize_latent_fp8(ckv))
            self._pools[b] = (keys, pv, ckv)
        if self._A is None and wl.o_absorb is not None and self.with_project:
            self._A = wl.o_absorb.float().numpy()
        return b

    def run_row(self, r: int) -> float:
        """Seconds for one query row (score, top-k, expand, attention, o_absorb)."""
        O, wl, g = self.O, self.wl, self.wl.geom
        b = self._prep(r)
        keys, pv, ckv = self._pools[b]
        q = wl.qidx[r].float().numpy()
        w = wl.w[r].numpy()
        ql = wl.qlat[r].float().numpy()
        t0 = time.perf_counter()
        O.decode_row(q, w, keys, pv, int(wl.row_ctx[r]), g.first_key, g.index_kpool,
                     g.index_scale, g.index_topk, wl.p_stride, ql, ckv, g.softmax_scale, self._A,
                     always_select_tail=g.always_select_tail)
        return time.perf_counter() - t0


def cpu_baseline(wl, budget_s: float = 12.0, max_rows: int = 2, latent_fp8: bool = False) -> dict:
    prefill = wl.name.startswith("prefill")
    runner = OracleRunner(wl, with_project=not prefill, latent_fp8=latent_fp8)
    # one thread, held on one core for the timed rows
    old_aff = os.sched_getaffinity(0) if hasattr(os, "sched_getaffinity") else None
    core = min(old_aff) if old_aff else None
    if core is not None:
        os.sched_setaffinity(0, {core})
    try:
        return _cpu_baseline(runner, wl, budget_s, max_rows, prefill, core)
    finally:
        if old_aff:
            os.sched_setaffinity(0, old_aff)


def _cpu_baseline(runner, wl, budget_s, max_rows, prefill, core) -> dict:
    times, rows = [], []
    for r in range(min(max_rows, wl.rows)):
        runner._prep(r)
        rows.append(r)
        times.append(runner.run_row(r))
        if sum(times) > budget_s:
            break
    # Repeat the prepared rows until the time budget is used.
    i = 0
    while sum(times) < budget_s and i < 5000:
        times.append(runner.run_row(rows[i % len(rows)]))
        i += 1
    v = len(times) / sum(times)
    tail = "olat (no o_absorb, as the GPU step)" if prefill else "o_absorb"
    return {"value": v, "unit": "queries/s", "cores": 1, "kind": "oracle",
            "sample": f"{len(times)} query rows (rows {rows}) of {wl.name}: score over all "
                      f"{wl.p_stride} pools, top-k, expand, attention over the selected tokens, "
                      f"{tail}; float64 numpy, one thread; pooled-key cache built untimed",
            "seconds": sum(times), "pinned_core": core, **cpu_info()}


# ---------------------------------------------------------------------------


def make_wl(args):
    wl = (W.long_262k(seq_len=args.seq_len) if (args.seq_len and args.workload == 3)
          else W.WORKLOADS[args.workload]())
    if args.always_select_tail:
        wl.geom = dataclasses.replace(wl.geom, always_select_tail=True)
    return wl


def run_reference(args, ws, rank):
    if rank != 0:
        return
    wl = make_wl(args)
    prefill = args.workload == PREFILL_WORKLOAD
    runner = OracleRunner(wl, with_project=not prefill, latent_fp8=args.latent_fp8)
    rows = [r % wl.rows for r in range(min(2, wl.rows))]
    for r in rows:
        runner._prep(r)
    old_aff = os.sched_getaffinity(0) if hasattr(os, "sched_getaffinity") else None
    core = min(old_aff) if old_aff else None
    if core is not None:
        os.sched_setaffinity(0, {core})  # one thread on one core, as the CPU baseline
    try:
        for i in range(args.warmup):
            runner.run_row(rows[i % len(rows)])
        ts = [runner.run_row(rows[i % len(rows)]) for i in range(args.steps)]
    finally:
        if old_aff:
            os.sched_setaffinity(0, old_aff)
    total = sum(ts)
    v = args.steps / total
    line = {
        "impl": "reference", "metric": PREFILL_METRIC if prefill else METRIC, "value": v,
        "unit": "queries/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(wl, args),
        "cpu_baseline": {"value": v, "unit": "queries/s", "cores": 1, "kind": "oracle",
                         "sample": f"one query row per step (rows {rows}) of {wl.name}",
                         "pinned_core": core, **cpu_info()},
        "e2e": {"value": v, "unit": "queries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(wl, args) -> dict:
    g = wl.geom
    return {"workload": wl.name, "sequences": wl.batch, "seq_len": int(wl.max_seq_len),
            "query_rows": wl.rows, "index_kpool": g.index_kpool, "index_heads": g.index_heads,
            "index_head_dim": g.index_head_dim, "index_topk": g.index_topk, "heads": g.heads,
            "kv_lora_rank": g.kv_lora_rank, "hidden": g.hidden,
            "paged_block": wl.block_size, "seed": wl.seed,
            "always_select_tail": bool(g.always_select_tail),
            "decode_append": bool(getattr(args, "decode_append", False)),
            "latent_cache": "fp8-e4m3" if getattr(args, "latent_fp8", False) else "bf16",
            "frontend": ({"q_lora_rank": args.q_lora_rank}
                         if getattr(args, "frontend", False) else None),
            "o_absorb_l2_prefetch_mib": getattr(args, "l2_prefetch_mib_used", 0.0),
            "l2": "flushed between timed steps (256 MiB write, then a 256 MiB read so the dirty "
                  "lines are written back; both outside the timed events)",
            "parallelism": f"replicas x{args.gpus}" if args.gpus > 1 else "single GPU"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", type=int, default=3)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--seq-len", type=int, default=None,
                    help="shrink the 262K workload's sequences (profiling runs only)")
    ap.add_argument("--decode-append", action="store_true",
                    help="each step first appends one token per sequence (indexer store, "
                         "device-side geometry, compress of the newly whole pool), replayed "
                         "as one graph over the growing context")
    ap.add_argument("--frontend", action="store_true",
                    help="each step starts from the hidden state: the projection front-end "
                         "(q_a/kv_a/indexer projections, a-norms, q_absorb, wq_b) on the "
                         "device, then the step")
    ap.add_argument("--q-lora-rank", type=int, default=1536)
    ap.add_argument("--latent-fp8", action="store_true",
                    help="attention reads an FP8 latent cache (E4M3 codes + power-of-two "
                         "scales per 128 channels) encoded once from the bf16 cache")
    ap.add_argument("--l2-prefetch-mb", type=float, default=None,
                    help="MiB of o_absorb prefetched into L2 on a second graph branch "
                         "while top-k and the gather run (default: the layer's choice, "
                         "64 MiB for the GLM-5.3 o_absorb; 0 turns it off)")
    ap.add_argument("--always-select-tail", action="store_true",
                    help="index rows index_topk + kpool - 1 wide, the trailing partial "
                         "pool's tokens always attended")
    args = ap.parse_args()
    ws, rank, local = dist_init(args.gpus)
    if args.impl == "reference":
        run_reference(args, ws, rank)
        barrier(ws)
        return

    import __graft_entry__ as ge
    from sparse_attention_decode_kpool_gb300.pipeline import DsaDecodeLayer

    if rank == 0 or ws == 1:
        ge.build()
    barrier(ws)
    ge.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    wl = make_wl(args)
    prefill = args.workload == PREFILL_WORKLOAD
    # The prefill chunk's step ends at olat (its o_absorb GEMM is not part of it).
    append = bool(args.decode_append)
    if append and prefill:
        raise SystemExit("--decode-append applies to the decode workloads")
    decode_from = None
    if append:
        # Room for every replay that appends (warm-up, timed, stage and e2e passes).
        room = args.warmup + 5 * args.steps + 32
        decode_from = np.maximum(wl.seq_lens.astype(np.int64) - room, 0)
    fe = None
    if args.frontend:
        if prefill:
            raise SystemExit("--frontend applies to the decode workloads")
        fe = W.make_frontend(wl.geom, wl.rows, q_lora_rank=args.q_lora_rank, seed=wl.seed + 100)
    layer = DsaDecodeLayer(wl, device=str(dev), with_o_absorb=not prefill, keep_olat=prefill,
                           decode_from=decode_from, latent_fp8=args.latent_fp8, frontend=fe,
                           l2_prefetch_bytes=(None if args.l2_prefetch_mb is None
                                              else int(args.l2_prefetch_mb * (1 << 20))))
    args.l2_prefetch_mib_used = layer.l2_prefetch_bytes / (1 << 20)
    if append:
        layer.stage(0)  # the staged rows stay as they are for every replay
    layer.compress()
    torch.cuda.synchronize()

    # compress alone (setup stage, reported on its own)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    flush_w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    class _Flush:
        """Write 256 MiB (evicts L2), then read another 256 MiB so the dirty lines
        are written back before the timed region instead of inside it."""

        def zero_(self):
            flush_w.zero_()
            flush_r.sum()

    flush = _Flush()
    ct = []
    comp_bytes = compress_bytes(wl, layer.seq_lens.cpu().numpy())
    for _ in range(3):
        flush.zero_()
        e0.record()
        layer.compress()
        e1.record()
        torch.cuda.synchronize()
        ct.append(e0.elapsed_time(e1))

    layer.step()
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0, "device status flagged during the first step"

    # The timed graph: the step's library calls only (with --decode-append, the
    # append of one token per sequence first: every replay grows the context).
    if fe is not None:
        graph = layer.capture_layer()
    elif append:
        graph = layer.capture_append()
    else:
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(s):
            layer.step()
        torch.cuda.current_stream(dev).wait_stream(s)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            layer.step()
    # A second graph with timing event nodes at the stage boundaries (external
    # events when the installed torch supports them): per-stage times.
    stage_names = (["frontend"] if fe is not None else []) + (["append"] if append else []) + [
        "score", "select", "expand", "attend"] + ([] if prefill else ["project"])
    ns = len(stage_names)
    try:
        ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(ns + 1)]
        graph_events = True
    except TypeError:
        ev, graph_events = None, False
    sgraph = None
    if graph_events:
        sgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(sgraph):
            ev[0].record()
            for j, k in enumerate(stage_names):
                getattr(layer, k)()
                ev[j + 1].record()

    launches = (layer.launches_per_layer_step() if fe is not None else
                layer.launches_per_append_step() if append else layer.launches_per_step())
    for _ in range(args.warmup):
        flush.zero_()
        graph.replay()
    torch.cuda.synchronize()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(dev) as clocks:
        for i in range(args.steps):
            flush.zero_()
            starts[i].record()
            graph.replay()
            ends[i].record()
        torch.cuda.synchronize()
    barrier(ws)
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    ms = sum(step_ms) / args.steps
    ms = max_over_ranks(ms, ws)
    # Per-stage times (separate pass; event nodes add a little time of their own).
    stage_ms = {k: 0.0 for k in stage_names}
    for i in range(args.steps):
        flush.zero_()
        if graph_events:
            sgraph.replay()
            ev[ns].synchronize()
            for j, k in enumerate(stage_names):
                stage_ms[k] += ev[j].elapsed_time(ev[j + 1])
        else:
            ev2 = [torch.cuda.Event(enable_timing=True) for _ in range(ns + 1)]
            ev2[0].record()
            for j, k in enumerate(stage_names):
                getattr(layer, k)()
                ev2[j + 1].record()
            ev2[ns].synchronize()
            for j, k in enumerate(stage_names):
                stage_ms[k] += ev2[j].elapsed_time(ev2[j + 1])
    stage_ms = {k: v / args.steps for k, v in stage_ms.items()}

    queries = wl.rows * ws
    value = queries / (ms * 1e-3)

    # e2e: per-step query inputs from pinned host memory, result read back.
    e2e = None
    if not args.no_e2e:
        result = layer.olat if prefill else layer.y
        h_y = torch.empty_like(result, device="cpu").pin_memory()
        # The step's inputs: query tensors and the row contexts; with --decode-append
        # the staged token rows instead of the contexts (those follow the lengths on
        # the device).
        # With --frontend the hidden state replaces the query tensors and the staged
        # rows (the front-end makes both on the device).
        if fe is not None:
            ins = [(layer.x, fe.x.pin_memory())]
        else:  # qidx, w, qlat and row_ctx share one buffer: one transfer
            ins = [(layer.step_inputs, layer.host_step_inputs())]
        if append and fe is None:
            ins += [(d, h.pin_memory()) for d, h in zip((layer.k_new, layer.gate_new,
                                                        layer.ckv_new), layer.staged_rows(0))]
        h2d = sum(h.numel() * h.element_size() for _, h in ins)
        d2h = h_y.numel() * h_y.element_size()
        # One graph per step: the pinned-host copies in, the step's library calls,
        # the result out; the host waits for it and reads the clock. The projection
        # stores y straight into pinned host memory (unified addressing), so the
        # result needs no copy node.
        step_fn = (layer.layer_step if fe is not None else
                   layer.append_step if append else layer.step)
        direct_out = not prefill and layer.o_absorb is not None
        # Two graphs with their own pinned inputs and result buffers, so that the host
        # can queue step i+1 before it reads step i's result.
        h_ys = [h_y, torch.empty_like(h_y).pin_memory()]
        h_ins = [[h for _, h in ins], [h.clone().pin_memory() for _, h in ins]]
        io_graphs = []
        y_dev = layer.y
        for b in range(2):
            gr = torch.cuda.CUDAGraph()
            if direct_out:
                layer.y = h_ys[b]
            with torch.cuda.graph(gr):
                for (d, _), h in zip(ins, h_ins[b]):
                    d.copy_(h, non_blocking=True)
                step_fn()
                if not direct_out:
                    h_ys[b].copy_(result, non_blocking=True)
            io_graphs.append(gr)
        layer.y = y_dev
        for _ in range(3):
            io_graphs[0].replay()
            io_graphs[1].replay()
        torch.cuda.synchronize()
        # host views of the results (bf16 or f32 read as raw bits)
        views = [hy.view(torch.int16 if hy.element_size() == 2 else torch.int32).numpy()
                 for hy in h_ys]
        # (1) one step at a time: L2 flushed, the clock started with the GPU idle,
        # stopped when the result is in host memory
        t_e2e = []
        for _ in range(args.steps):
            flush.zero_()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            io_graphs[0].replay()
            torch.cuda.synchronize()
            _ = int(views[0].flat[0])
            t_e2e.append(time.perf_counter() - t0)
        lat_ms = max_over_ranks(1e3 * sum(t_e2e) / len(t_e2e), ws)
        # (2) throughput: steps back to back with two in flight; each step uploads its
        # inputs, and the host waits for and reads each step's result while the next
        # is already queued. No flush: a step streams over three times the L2's size.
        # For the plain decode step the inputs go through a second device buffer on a
        # copy stream, so step i+1's upload overlaps step i.
        # (the front-end's hidden state the same way)
        # (the staged token rows and the front-end's hidden state the same way)
        # With a result that has to be copied out (the prefill chunk's olat) the result
        # is double-buffered too and read back on a third stream.
        overlap = True
        done = [torch.cuda.Event(), torch.cuda.Event()]
        got = [torch.cuda.Event(), torch.cuda.Event()]  # result in host memory
        if overlap:
            # device input sets in the order of `ins`; point(b) makes the layer read set b
            if fe is None:
                names = ["k_new", "gate_new", "ckv_new"] if append else []
                dsets = [[layer.step_inputs] + [getattr(layer, n) for n in names]]

                def point(b: int) -> None:
                    layer.use_step_inputs(dsets[b][0])
                    for n, t in zip(names, dsets[b][1:]):
                        setattr(layer, n, t)
            else:
                dsets = [[layer.x]]

                def point(b: int) -> None:
                    layer.x = dsets[b][0]
            dsets.append([torch.empty_like(t) for t in dsets[0]])
            obufs = None if direct_out else [layer.olat, torch.empty_like(layer.olat)]
            sgraphs = []
            for b in range(2):
                point(b)
                if direct_out:
                    layer.y = h_ys[b]
                else:
                    layer.olat = obufs[b]
                gr = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gr):
                    step_fn()
                sgraphs.append(gr)
            point(0)
            layer.y = y_dev
            if obufs is not None:
                layer.olat = obufs[0]
            cs = torch.cuda.Stream()
            rs = torch.cuda.Stream()
            main = torch.cuda.current_stream()
            up = [torch.cuda.Event(), torch.cuda.Event()]

            def upload(b: int, after_step: bool) -> None:
                with torch.cuda.stream(cs):
                    if after_step:
                        cs.wait_event(done[b])  # the step that last read set b
                    for d, h in zip(dsets[b], h_ins[b]):
                        d.copy_(h, non_blocking=True)
                    up[b].record(cs)

            def launch(i: int) -> None:
                b = i % 2
                main.wait_event(up[b])
                if obufs is not None and i >= 2:
                    main.wait_event(got[b])  # step i-2's result has left obufs[b]
                sgraphs[b].replay()
                done[b].record(main)
                if obufs is None:
                    got[b].record(main)  # the step stored it in pinned memory itself
                else:
                    with torch.cuda.stream(rs):
                        rs.wait_event(done[b])
                        h_ys[b].copy_(obufs[b], non_blocking=True)
                        got[b].record(rs)

            for b in range(2):  # warm both graphs once
                upload(b, False)
                launch(b)
            torch.cuda.synchronize()
        torch.cuda.synchronize()
        barrier(ws)
        t0 = time.perf_counter()
        if overlap:
            upload(0, False)
            launch(0)
            for i in range(args.steps):
                if i + 1 < args.steps:
                    upload((i + 1) % 2, i >= 1)
                    launch(i + 1)
                got[i % 2].synchronize()
                _ = int(views[i % 2].flat[0])
        else:
            io_graphs[0].replay()
            done[0].record()
            for i in range(args.steps):
                if i + 1 < args.steps:
                    io_graphs[(i + 1) % 2].replay()
                    done[(i + 1) % 2].record()
                done[i % 2].synchronize()
                _ = int(views[i % 2].flat[0])
        e2e_ms = max_over_ranks(1e3 * (time.perf_counter() - t0) / args.steps, ws)
        e2e = {"value": queries / (e2e_ms * 1e-3), "unit": "queries/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "in_flight": 2, "latency_ms_per_step": lat_ms,
               "latency_value": queries / (lat_ms * 1e-3),
               "path": "pinned host " + ("x (hidden state)" if fe is not None else
                                         "qidx/w/qlat/row_ctx (one buffer)")
                       + ("/staged token rows" if append and fe is None else "")
                       + " -> device, the step, " + ("olat" if prefill else "y")
                       + (" stored by the projection straight into pinned host memory"
                          if direct_out else " -> host")
                       + ", as one CUDA graph replayed per step, host-timed; value: steps "
                         "back to back, two in flight, every result waited for and read on "
                         "the host (no L2 flush: each step streams over 3x L2)"
                       + ("; inputs double-buffered on the device, each step's upload on a "
                          "copy stream overlapping the step before"
                          + ("" if direct_out else ", olat double-buffered and read back "
                             "on a second copy stream") if overlap else "")
                       + "; latency_*: one step at a time from an idle GPU and a flushed L2"}

    if rank != 0:
        return

    peaks = {}
    pk = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk):
        peaks = json.load(open(pk))
    hbm_peak = peaks.get("hbm_gbs") or 6800.0
    if prefill:
        tf = peaks.get("bf16_tflops")
        peak_src = "measured (bf16 dense burst)" if tf else "fallback"
        tf = tf or 1900.0
        fl = algorithmic_flops(wl, layer)
        dom = max(("score", "attend"), key=lambda k: stage_ms[k])
        achieved = fl[dom] / (stage_ms[dom] * 1e-3) / 1e12
        step_tf = fl["total"] / (ms * 1e-3) / 1e12
        roofline = {"bound": "tensor", "achieved": achieved, "peak": tf, "unit": "TFLOP/s",
                    "frac": achieved / tf, "traffic": None, "peak_source": peak_src,
                    "kernel": {"score": "dsa_score_prefill (tcgen05 contraction, TMEM epilogue)",
                               "attend": "dsa_sparse_mla_decode (split attention)"}[dom],
                    "algorithmic_flops_per_launch": fl[dom], "step_algorithmic_flops": fl["total"],
                    "step_achieved_tflops": step_tf, "step_frac": step_tf / tf,
                    "stage_tflops": {k: fl[k] / (stage_ms[k] * 1e-3) / 1e12
                                     for k in ("score", "attend")}}
    else:
        hbm = peaks.get("hbm_gbs")
        peak_src = "measured" if hbm else "fallback"
        hbm = hbm or 6800.0
        ab = algorithmic_bytes(wl, layer)
        dom = max(("score", "attend", "project") + (("frontend",) if fe is not None else ()),
                  key=lambda k: stage_ms[k])
        dom_bytes = ab[dom]
        achieved = dom_bytes / (stage_ms[dom] * 1e-3) / 1e9
        total_gbs = ab["total"] / (ms * 1e-3) / 1e9
        tr = MEASURED_TRAFFIC.get(dom) if wl.geom.hidden == 4096 and wl.rows == 8 else None
        roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                    "frac": achieved / hbm, "traffic": tr[0] if tr else None,
                    "traffic_source": tr[1] if tr else None, "peak_source": peak_src,
                    "kernel": {"attend": "dsa_sparse_mla_decode (split attention + combine)",
                               "project": "dsa_latent_project (tcgen05 o_absorb GEMM, TMA "
                                          "ring, K shares summed in a thread-block cluster)",
                               "score": "dsa_score",
                               "frontend": "dsa_frontend (x projections, a-norms, q_absorb and "
                                           "wq_b skinny GEMMs)"}[dom],
                    "algorithmic_bytes_per_launch": dom_bytes,
                    "step_algorithmic_bytes": ab["total"], "step_achieved_gbs": total_gbs,
                    "step_frac": total_gbs / hbm}
        # the step without the o_absorb projection: index scores, top-k (+ token ids)
        # and the sparse attention to olat, timed by their stages
        core_b = ab["score"] + ab["attend"]
        core_ms = sum(stage_ms[k] for k in ("score", "select", "expand", "attend"))
        roofline["attention_core"] = {"bytes": core_b, "ms": core_ms,
                                      "achieved_gbs": core_b / (core_ms * 1e-3) / 1e9,
                                      "frac": core_b / (core_ms * 1e-3) / 1e9 / hbm}
    line = {
        "metric": PREFILL_METRIC if prefill else METRIC, "value": value, "unit": "queries/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(wl, args),
        "roofline": roofline,
        "stages_ms": stage_ms,
        "stage_timing": ("separate pass, graph with event nodes" if graph_events
                         else "separate eager pass")
                        + ("; attention and projection timed as two calls (dsa_sparse_mla_decode "
                           "to olat, dsa_latent_project), the step makes them one"
                           if layer.o_absorb is not None and layer.two_call and not prefill else "")
                        + ("; no o_absorb L2 prefetch branch in this pass (the projection "
                           "streams all of o_absorb from HBM)" if layer.l2_prefetch_bytes else ""),
        "compress_ms": min(ct),
        "compress": {"bytes": comp_bytes, "ms": min(ct),
                     "achieved_gbs": comp_bytes / (min(ct) * 1e-3) / 1e9,
                     "frac": comp_bytes / (min(ct) * 1e-3) / 1e9 / hbm_peak,
                     "note": "dsa_compress alone (setup, not in the step): raw keys, gates "
                             "and flags in, pooled keys and flags out; L2 flushed before"},
        "gpu_launches": launches * args.steps,
        "clocks": clocks.summary(),
    }
    if e2e is not None:
        line["e2e"] = e2e
    if not args.no_cpu_baseline and ws == 1:
        line["cpu_baseline"] = cpu_baseline(wl, latent_fp8=args.latent_fp8)
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
