"""One DSA decode layer on one GPU: device-resident caches plus the per-step chain
score -> select -> expand -> sparse latent MLA, all through the C ABI.

``DsaDecodeLayer`` uploads a workload's caches once (the latent KV cache, the raw
indexer keys, o_absorb), builds the pooled-key cache with ``dsa_compress``, and
owns every step buffer, so a step allocates nothing and can be captured in a
CUDA graph.
"""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from . import api
from .workloads import Workload


class DsaDecodeLayer:
    def __init__(self, wl: Workload, device: str = "cuda", keep_olat: bool = False,
                 with_o_absorb: bool = True, use_drawn_kpool: bool = False,
                 score_path: str = "auto", fuse_expand: bool = True, decode_from=None,
                 fuse_append: bool = True, latent_fp8: bool = False, frontend=None,
                 l2_prefetch_bytes: Optional[int] = None):
        g = wl.geom
        self.wl = wl
        self.geom = g
        dev = torch.device(device)
        self.device = dev
        up = lambda t: None if t is None else t.to(dev, non_blocking=False).contiguous()

        self.seq_lens = torch.from_numpy(wl.seq_lens).to(dev)
        self.block_table = up(wl.block_table)
        self.pg = api.paging(self.seq_lens, wl.max_seq_len, self.block_table,
                             wl.block_size or 0, wl.num_blocks)
        self.row_seq = torch.from_numpy(wl.row_seq).to(dev)
        # The per-step query inputs (qidx, w, qlat, row_ctx) are views of one device
        # buffer, so that a host copy of the step's inputs is a single transfer.
        R0, g0 = wl.rows, wl.geom
        self._in_specs = [("qidx", (R0, g0.index_heads, g0.index_head_dim), torch.bfloat16),
                          ("w", (R0, g0.index_heads), torch.float32),
                          ("qlat", (R0, g0.heads, g0.kv_lora_rank), torch.bfloat16),
                          ("row_ctx", (R0,), torch.int32)]
        self.step_inputs = self._carve(dev, pinned=False)
        self.row_ctx.copy_(torch.from_numpy(wl.row_ctx))

        # Resident state.
        self.ckv = up(wl.ckv)
        # FP8 latent cache (E4M3 codes + power-of-two scales per 128 channels), encoded
        # once from the bf16 cache; attention then gathers 528 instead of 1,024 bytes
        # per token.
        self.latent_fp8 = bool(latent_fp8)
        self.ckv_codes = self.ckv_scales = None
        if self.latent_fp8:
            if decode_from is not None and not fuse_append:
                raise ValueError("the FP8 latent cache is appended by dsa_decode_append_fp8 "
                                 "only (fuse_append=True)")
            kvl = g.kv_lora_rank
            self.ckv_codes = torch.empty(self.ckv.shape, dtype=torch.uint8, device=dev)
            self.ckv_scales = torch.empty(self.ckv.shape[:-1] + (kvl // 128,),
                                          dtype=torch.float32, device=dev)
            api.dsa_quantize_latent(self.ckv, self.ckv_codes, self.ckv_scales)
        self.o_absorb = up(wl.o_absorb) if with_o_absorb else None
        # The step prefetches the first l2_prefetch_bytes of o_absorb into L2 on a
        # second stream while top-k and the gather run (they leave HBM mostly idle);
        # None: a quarter of o_absorb, at most 64 MiB (half of L2; the gathered
        # latent rows pass through the rest).
        if l2_prefetch_bytes is None:
            l2_prefetch_bytes = (min(64 << 20, self.o_absorb.numel() * 2 // 4)
                                 if self.o_absorb is not None else 0)
        self.l2_prefetch_bytes = int(l2_prefetch_bytes) if self.o_absorb is not None else 0
        self._side = torch.cuda.Stream(device=dev) if self.l2_prefetch_bytes > 0 else None
        KP, ihd = g.index_kpool, g.index_head_dim
        if wl.paged:
            pshape = (wl.num_blocks, wl.block_size // KP)
        else:
            pshape = (wl.batch, wl.max_seq_len // KP)
        if use_drawn_kpool:
            self.kpool = up(wl.kpool_keys)
            self.pool_valid = up(wl.kpool_valid)
            self.k_raw = self.gate = self.valid = None
        else:
            self.kpool = torch.zeros(pshape + (ihd,), dtype=torch.bfloat16, device=dev)
            self.pool_valid = torch.zeros(pshape, dtype=torch.uint8, device=dev)
            self.k_raw, self.gate, self.valid = up(wl.k_raw), up(wl.gate), up(wl.valid)
        self.ape, self.ln_w, self.ln_b = up(wl.ape), up(wl.ln_w), up(wl.ln_b)

        # Per-step inputs (device copies) and buffers.
        self.qidx.copy_(wl.qidx)
        self.w.copy_(wl.w)
        self.qlat.copy_(wl.qlat)
        R = wl.rows
        self.p_stride = wl.p_stride
        self.sk = api.dsa_select_k(g.index_topk, KP, self.p_stride)
        self.scores = torch.empty((R, self.p_stride), dtype=torch.float32, device=dev)
        self.pool_ids = torch.empty((R, self.sk), dtype=torch.int32, device=dev)
        self.token_ids = torch.empty((R, g.out_width), dtype=torch.int32, device=dev)
        hidden = g.hidden if self.o_absorb is not None else 0
        self.y = torch.empty((R, hidden), dtype=torch.bfloat16, device=dev) if hidden else None
        # olat feeds the projection, so it always exists when o_absorb does.
        self.keep_olat = bool(keep_olat)
        self.olat = (torch.empty((R, g.heads, g.kv_lora_rank), dtype=torch.float32, device=dev)
                     if (keep_olat or self.o_absorb is not None) else None)
        ws = api.dsa_sparse_mla_decode_workspace(R, g.heads, g.out_width, 0, False)
        self.workspace = torch.zeros(max(ws, 1), dtype=torch.uint8, device=dev)
        # The stages attend() and project() are the two-call form (attention to olat,
        # then dsa_latent_project) where the projection kernels support the shape
        # (hidden % 64 == 0); else attend() makes the one call. step() makes the one
        # call (attention and projection, olat as bf16 straight into the projection)
        # whenever o_absorb is present.
        self.two_call = bool(hidden) and hidden % 64 == 0
        pws = api.dsa_latent_project_workspace(R, g.heads, hidden) if self.two_call else 0
        self.proj_workspace = torch.zeros(max(pws, 1), dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        # Scoring: a chunk of >= 64 query rows of one contiguous sequence goes to the
        # tensor-core contraction (dsa_score_prefill); everything else to dsa_score.
        one_seq = R > 0 and bool((wl.row_seq == wl.row_seq[0]).all())
        gemm_ok = (one_seq and not wl.paged and g.index_heads in (32, 64, 128)
                   and ihd in (64, 128))
        if score_path not in ("auto", "decode", "prefill"):
            raise ValueError(f"score_path {score_path!r}")
        if score_path == "prefill" and not gemm_ok:
            raise ValueError("score_path='prefill' needs one contiguous sequence and "
                             "index_heads in {32, 64, 128}")
        self.prefill_seq = int(wl.row_seq[0]) if R > 0 else 0
        self.score_gemm = score_path == "prefill" or (score_path == "auto" and gemm_ok
                                                      and R >= 64)
        self.graph: Optional[torch.cuda.CUDAGraph] = None
        self._fused_ws: Optional[torch.Tensor] = None
        # select() also expands (dsa_select_expand); expand() is then a no-op.
        self.fuse_expand = bool(fuse_expand)
        # Decode-time append: the caches start at decode_from tokens per sequence and
        # append_step() appends one staged token per sequence before the step.
        # append() is one dsa_decode_append launch, or the three calls it joins.
        self.fuse_append = bool(fuse_append)
        self.decode_from: Optional[np.ndarray] = None
        self.append_graph: Optional[torch.cuda.CUDAGraph] = None
        if decode_from is not None:
            self._init_append(decode_from)
        # Projection front-end (dsa_frontend): the step's query inputs and the token's
        # staged rows computed from a hidden state x on the device.
        self.fe = None
        if frontend is not None:
            self._init_frontend(frontend)

    def _init_frontend(self, fe) -> None:
        g, dev, R = self.geom, self.device, self.wl.rows
        up = lambda t: t.to(dev).contiguous()
        self.fe = fe
        self.x = up(fe.x)
        self.w_x = up(fe.packed_x_weights())
        self.q_a_norm, self.kv_a_norm = up(fe.q_a_norm), up(fe.kv_a_norm)
        self.w_q = up(fe.packed_q_weights())
        if self.decode_from is None:  # the staged rows have nowhere to go: scratch
            self.k_new = torch.zeros((R, g.index_head_dim), dtype=torch.bfloat16, device=dev)
            self.gate_new = torch.zeros_like(self.k_new)
            self.ckv_new = torch.zeros((R, g.kv_lora_rank), dtype=torch.bfloat16, device=dev)
        n = api.dsa_frontend_workspace(R, g.hidden, int(self.w_x.shape[0]), fe.q_lora_rank,
                                       g.kv_lora_rank, g.index_head_dim, g.index_heads, g.heads)
        self.fe_workspace = torch.zeros(max(n, 1), dtype=torch.uint8, device=dev)

    def frontend(self, stream=None) -> None:
        """x -> qlat, qidx, w (the step's inputs) and k_new, gate_new, ckv_new (the
        token's rows that append() stores)."""
        api.dsa_frontend(self.x, self.w_x, self.q_a_norm, self.kv_a_norm, self.fe.eps,
                         self.w_q, self.qlat, self.qidx, self.w, self.k_new, self.gate_new,
                         self.ckv_new, self.status, self.fe_workspace, stream=stream)

    def layer_step(self, stream=None) -> None:
        """The whole decode layer: front-end, the token's append (when the layer was
        built with decode_from), then the step."""
        self.frontend(stream)
        if self.decode_from is not None:
            self.append(stream)
        self.step(stream)

    def _carve(self, device, pinned: bool, names: bool = True) -> torch.Tensor:
        """One byte buffer holding the step inputs at 256-byte aligned offsets; on the
        device the layer's qidx, w, qlat and row_ctx become views of it."""
        offs, off = [], 0
        for _, shape, dt in self._in_specs:
            n = int(np.prod(shape)) * torch.empty((), dtype=dt).element_size()
            offs.append((off, n))
            off = (off + n + 255) & ~255
        buf = (torch.empty(off, dtype=torch.uint8).pin_memory() if pinned
               else torch.empty(off, dtype=torch.uint8, device=device))
        self._in_offs = offs
        if names:
            for (name, shape, dt), (o, n) in zip(self._in_specs, offs):
                setattr(self, name, buf[o:o + n].view(dt).view(shape))
        return buf

    def use_step_inputs(self, buf: torch.Tensor) -> None:
        """Point qidx, w, qlat and row_ctx at device buffer buf (the step_inputs
        layout), e.g. a second buffer so that the next step's inputs can be uploaded
        while this step runs. Graphs captured afterwards read from buf."""
        if buf.numel() != self.step_inputs.numel() or buf.device != self.step_inputs.device:
            raise ValueError("buf must match step_inputs in size and device")
        for (name, shape, dt), (o, n) in zip(self._in_specs, self._in_offs):
            setattr(self, name, buf[o:o + n].view(dt).view(shape))

    def host_step_inputs(self) -> torch.Tensor:
        """A pinned host buffer with the device step-input layout, filled with the
        workload's inputs: one copy_ into step_inputs uploads a step's queries."""
        buf = self._carve(None, pinned=True, names=False)
        wl = self.wl
        src = {"qidx": wl.qidx, "w": wl.w, "qlat": wl.qlat,
               "row_ctx": torch.from_numpy(wl.row_ctx)}
        for (name, shape, dt), (o, n) in zip(self._in_specs, self._in_offs):
            buf[o:o + n].view(dt).view(shape).copy_(src[name])
        return buf

    # -- decode-time append -------------------------------------------------
    def _token_rows(self, b: int, t0: int, t1: int) -> np.ndarray:
        """Flat row numbers of tokens [t0, t1) of sequence b in a token cache."""
        wl = self.wl
        t = np.arange(t0, t1, dtype=np.int64)
        if not wl.paged:
            return b * wl.max_seq_len + t
        blk = wl.block_table.numpy()[b, t // wl.block_size].astype(np.int64)
        return blk * wl.block_size + t % wl.block_size

    def _init_append(self, decode_from) -> None:
        wl, g = self.wl, self.geom
        if self.k_raw is None:
            raise ValueError("decode-time append needs the raw indexer caches")
        if wl.rows != wl.batch or not (wl.row_seq == np.arange(wl.batch)).all():
            raise ValueError("decode-time append takes one decode row per sequence")
        L0 = np.broadcast_to(np.asarray(decode_from, dtype=np.int64), (wl.batch,)).copy()
        if (L0 < 0).any() or (L0 > wl.seq_lens).any():
            raise ValueError("decode_from must lie in [0, seq_lens]")
        self.decode_from = L0
        # The caches hold only the first L0[b] tokens; later rows are staged one per
        # step (the workload's own rows, so a step's result can be checked).
        dev = self.device
        for b in range(wl.batch):
            rows = torch.from_numpy(self._token_rows(b, int(L0[b]), int(wl.seq_lens[b]))).to(dev)
            if rows.numel():
                self.k_raw.view(-1, g.index_head_dim)[rows] = 0
                self.gate.view(-1, g.index_head_dim)[rows] = 0
                self.valid.view(-1)[rows] = 0
                self.ckv.view(-1, g.kv_lora_rank)[rows] = 0
        self.seq_lens.copy_(torch.from_numpy(L0.astype(np.int32)))
        B = wl.batch
        self.k_new = torch.zeros((B, g.index_head_dim), dtype=torch.bfloat16, device=dev)
        self.gate_new = torch.zeros_like(self.k_new)
        self.ckv_new = torch.zeros((B, g.kv_lora_rank), dtype=torch.bfloat16, device=dev)
        self.row_ctx.copy_(self.seq_lens)
        if self.latent_fp8:  # the FP8 cache of the cut-back bf16 cache
            api.dsa_quantize_latent(self.ckv, self.ckv_codes, self.ckv_scales)

    def staged_rows(self, i: int):
        """Host rows (k, gate, ckv) [batch, ...] of the token each sequence appends at
        step i: the workload's token at position decode_from[b] + i (zeros past the
        workload's own length)."""
        wl, g = self.wl, self.geom
        out = []
        for name, width in (("k_raw", g.index_head_dim), ("gate", g.index_head_dim),
                            ("ckv", g.kv_lora_rank)):
            src = getattr(wl, name).reshape(-1, width)
            rows = torch.zeros((wl.batch, width), dtype=torch.bfloat16)
            for b in range(wl.batch):
                t = int(self.decode_from[b]) + i
                if t < int(wl.seq_lens[b]):
                    rows[b] = src[int(self._token_rows(b, t, t + 1)[0])]
            out.append(rows)
        return tuple(out)

    def stage(self, i: int) -> None:
        """Copy step i's staged rows into the device buffers append_step() reads."""
        k, gt, c = self.staged_rows(i)
        self.k_new.copy_(k)
        self.gate_new.copy_(gt)
        self.ckv_new.copy_(c)

    def append_step(self, stream=None) -> None:
        """append() then step(): one decode step over the grown context."""
        self.append(stream)
        self.step(stream)

    def append(self, stream=None) -> None:
        """indexer_store -> write_geom -> compress of the newly whole pool."""
        g = self.geom
        if self.latent_fp8:  # the token's latent row goes to the FP8 cache only
            api.dsa_decode_append_fp8(self.k_new, self.gate_new, self.ckv_new, self.ape, self.ln_w,
                                      self.ln_b, g.eps, self.pg, self.seq_lens, g.first_key,
                                      g.index_kpool, self.k_raw, self.gate, self.valid,
                                      self.ckv_codes, self.ckv_scales, self.kpool,
                                      self.pool_valid, row_ctx=self.row_ctx, status=self.status,
                                      stream=stream)
            return
        if self.fuse_append:
            api.dsa_decode_append(self.k_new, self.gate_new, self.ape, self.ln_w, self.ln_b, g.eps,
                                  self.pg, self.seq_lens, g.first_key, g.index_kpool, self.k_raw,
                                  self.gate, self.valid, self.kpool, self.pool_valid,
                                  ckv_new=self.ckv_new, ckv=self.ckv, row_ctx=self.row_ctx,
                                  status=self.status, stream=stream)
            return
        api.dsa_indexer_store(self.k_new, self.gate_new, self.pg, self.seq_lens, self.k_raw,
                              self.gate, self.valid, self.ckv_new, self.ckv, self.status,
                              stream=stream)
        api.dsa_write_geom(self.seq_lens, self.row_seq, self.row_ctx, self.status, stream=stream)
        api.dsa_compress_append(self.k_raw, self.gate, self.valid, self.ape, self.ln_w, self.ln_b,
                                g.eps, self.pg, g.first_key, g.index_kpool, 1, self.kpool,
                                self.pool_valid, status=self.status, stream=stream)

    def capture_append(self) -> torch.cuda.CUDAGraph:
        """Capture append_step() into a CUDA graph. Each replay appends the staged
        rows at the live lengths and runs the step over the grown context. step()
        runs once eagerly first (it changes no cache or length)."""
        if self.decode_from is None:
            raise ValueError("the layer was not built with decode_from")
        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(s):
            self.step()
        torch.cuda.current_stream(self.device).wait_stream(s)
        torch.cuda.synchronize(self.device)
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            self.append_step()
        self.append_graph = gr
        return gr

    def fused_workspace(self) -> torch.Tensor:
        """Workspace for the one-call form dsa_sparse_mla_decode(..., o_absorb, y)."""
        if self._fused_ws is None:
            g, R = self.geom, self.wl.rows
            hidden = g.hidden if self.o_absorb is not None else 0
            n = api.dsa_sparse_mla_decode_workspace(R, g.heads, g.out_width, hidden,
                                                    self.o_absorb is not None)
            self._fused_ws = torch.zeros(max(n, 1), dtype=torch.uint8, device=self.device)
        return self._fused_ws

    # -- stages ------------------------------------------------------------
    def compress(self, stream=None) -> None:
        g = self.geom
        api.dsa_compress(self.k_raw, self.gate, self.valid, self.ape, self.ln_w, self.ln_b, g.eps,
                         self.pg, g.first_key, g.index_kpool, self.kpool, self.pool_valid,
                         status=self.status, stream=stream)

    def score(self, stream=None) -> None:
        g = self.geom
        if self.score_gemm:
            api.dsa_score_prefill(self.qidx, self.w, self.prefill_seq, self.row_ctx, self.kpool,
                                  self.pool_valid, self.pg, g.first_key, g.index_kpool,
                                  g.index_scale, self.scores, status=self.status, stream=stream)
            return
        api.dsa_score(self.qidx, self.w, self.row_seq, self.row_ctx, self.kpool, self.pool_valid,
                      self.pg, g.first_key, g.index_kpool, g.index_scale, self.scores,
                      status=self.status, stream=stream)

    def select(self, stream=None) -> None:
        g = self.geom
        if self.fuse_expand and g.always_select_tail:
            api.dsa_select_expand_tail(self.scores, g.index_topk, g.index_kpool, g.first_key,
                                       self.row_ctx, self.pool_ids, self.token_ids, stream=stream)
            return
        if self.fuse_expand:
            api.dsa_select_expand(self.scores, g.index_topk, g.index_kpool, g.first_key,
                                  self.pool_ids, self.token_ids, stream=stream)
            return
        api.dsa_select(self.scores, g.index_topk, g.index_kpool, self.pool_ids, stream=stream)

    def expand(self, stream=None) -> None:
        g = self.geom
        if self.fuse_expand:
            return
        if g.always_select_tail:
            api.dsa_expand_tail(self.pool_ids, g.first_key, g.index_kpool, g.index_topk,
                                self.row_ctx, self.token_ids, stream=stream)
            return
        api.dsa_expand(self.pool_ids, g.first_key, g.index_kpool, self.token_ids, stream=stream)

    def _mla(self, o_absorb, y, workspace, stream, olat=None) -> None:
        if self.latent_fp8:
            api.dsa_sparse_mla_decode_fp8(self.qlat, self.row_seq, self.ckv_codes, self.ckv_scales,
                                          self.pg, self.token_ids, self.geom.softmax_scale,
                                          o_absorb, y, olat, self.status, workspace,
                                          stream=stream)
        else:
            api.dsa_sparse_mla_decode(self.qlat, self.row_seq, self.ckv, self.pg, self.token_ids,
                                      self.geom.softmax_scale, o_absorb, y, olat,
                                      self.status, workspace, stream=stream)

    def attend(self, stream=None) -> None:
        """Sparse latent attention over the selected tokens -> olat (f32); in the
        one-call form also y."""
        if self.o_absorb is not None and not self.two_call:
            self._mla(self.o_absorb, self.y, self.fused_workspace(), stream, self.olat)
            return
        self._mla(None, None, self.workspace, stream, self.olat)

    def project(self, stream=None) -> None:
        """y = o_absorb . olat (the absorbed output projection)."""
        if self.o_absorb is not None and self.two_call:
            api.dsa_latent_project(self.olat, self.o_absorb, self.y, self.status,
                                   self.proj_workspace, stream=stream)

    def attend_project(self, stream=None) -> None:
        """Sparse latent attention and the o_absorb projection in one call (olat f32
        and y); without o_absorb, the attention alone."""
        if self.o_absorb is not None:
            # the f32 olat is written only when the layer keeps it (the projection reads
            # the bf16 copy the combine writes for it)
            self._mla(self.o_absorb, self.y, self.fused_workspace(), stream,
                      self.olat if self.keep_olat else None)
        else:
            self._mla(None, None, self.workspace, stream, self.olat)

    def step(self, stream=None) -> None:
        """One decode step over the whole batch: score, select (with the token ids),
        attention and projection."""
        self.score(stream)
        if self._side is not None:  # fork: the o_absorb prefetch beside the middle stages
            main = stream if stream is not None else torch.cuda.current_stream(self.device)
            self._side.wait_stream(main)
            api.dsa_prefetch_l2(self.o_absorb, self.l2_prefetch_bytes, stream=self._side)
        self.select(stream)
        self.expand(stream)
        self.attend_project(stream)
        if self._side is not None:  # join (the prefetch is long done by now)
            main.wait_stream(self._side)

    def launches_per_step(self) -> int:
        """Library kernel launches one step() makes."""
        R, g = self.wl.rows, self.geom
        n = 3 if self.fuse_expand else 4  # score, select(+expand), [expand], split attention
        if api.dsa_sparse_mla_decode_workspace(R, g.heads, g.out_width, 0, False) > 0:
            n += 1  # split combine
        if self.o_absorb is not None:
            # tensor-core projection: one launch per 64 query rows; else the stream-K
            # kernel(s) and the partial-sum reduction
            tc = (api.dsa_get_option(api._lib.DSA_OPT_PROJECT_KERNEL)
                  != api._lib.DSA_PROJECT_KERNEL_MMA and g.hidden % 128 == 0
                  and (g.heads * g.kv_lora_rank) % 512 == 0)
            n += (R + 63) // 64 + (0 if tc else 1)
        return n + (1 if self._side is not None else 0)  # the o_absorb L2 prefetch

    def capture_layer(self) -> torch.cuda.CUDAGraph:
        """Capture layer_step() into a CUDA graph. frontend() and step() run once
        eagerly first (neither changes a cache or a length)."""
        if self.fe is None:
            raise ValueError("the layer was not built with a front-end")
        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(s):
            self.frontend()
            self.step()
        torch.cuda.current_stream(self.device).wait_stream(s)
        torch.cuda.synchronize(self.device)
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            self.layer_step()
        self.layer_graph = gr
        return gr

    def launches_per_layer_step(self) -> int:
        """Library kernel launches one layer_step() makes: the front-end's two GEMMs
        with their reductions and the norm kernel, the append, the step."""
        n = 5 + self.launches_per_step()
        return n + (0 if self.decode_from is None else (1 if self.fuse_append else 3))

    def launches_per_append_step(self) -> int:
        """Library kernel launches one append_step() makes."""
        # store, write_geom, compress of the new pool (one launch when fused)
        return self.launches_per_step() + (1 if self.fuse_append else 3)

    # -- graphs ------------------------------------------------------------
    def capture(self) -> torch.cuda.CUDAGraph:
        """Capture step() into a CUDA graph (run step() once eagerly first)."""
        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(s):
            self.step()
        torch.cuda.current_stream(self.device).wait_stream(s)
        torch.cuda.synchronize(self.device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.step()
        self.graph = g
        return g

    def replay(self) -> None:
        assert self.graph is not None
        self.graph.replay()
