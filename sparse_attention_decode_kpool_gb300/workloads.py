"""Seeded synthetic inputs for one DSA decode layer.

This module only draws random numbers and lays them out in memory. It holds none
of the method's arithmetic, so both the CUDA path and the CPU oracle can consume
the same bytes without sharing code.

Every tensor is drawn from its own numpy ``Generator(PCG64)`` stream, keyed by
``(seed, tensor id, sequence)``. A sequence's values therefore do not depend on
which other sequences are generated, and a test can build one sequence of a
262,144-token workload without building the other seven.

Layouts (all row-major):

* contiguous caches: ``k_raw``/``gate`` ``[B, Smax, ihd]``, ``valid`` ``[B, Smax]``,
  ``ckv`` ``[B, Smax, kvl]``;
* paged caches: ``[NB, block_size, ...]`` with ``block_table [B, max_blocks]``
  (int32, -1 past a sequence's last block); the pooled-key cache that the
  compression step writes is then ``[NB, block_size / kpool, ihd]`` and uses the
  same table.

Value recipes follow the workload descriptions of the GLM-5.3 DSA layer
(``metrale_model_arch/glm5next_dsa/mod.rs``, "Shape of the pipeline", and the
tensor shape table of ``tp.rs``, ``DsaTpPlan::new``): bf16 storage rounded to
nearest even, ``ape`` kept in f32, index weights pre-multiplied by
``index_heads^-0.5``.
"""
from __future__ import annotations

import concurrent.futures as cf
import dataclasses
import math
import os
import threading
from typing import Optional, Sequence

import numpy as np
import torch

# Stream ids: one per tensor, fixed forever (changing one changes the workload).
_T_KRAW, _T_LNW, _T_LNB, _T_GATE, _T_APE, _T_VALID = 1, 2, 3, 4, 5, 6
_T_QIDX, _T_W, _T_QLAT, _T_CKV, _T_OABS, _T_LENS, _T_PERM = 7, 8, 9, 10, 11, 12, 13
_T_KPOOL = 14
_T_FX, _T_FQA, _T_FKVA, _T_FWK, _T_FGATE, _T_FWP, _T_FQN, _T_FKVN, _T_FQABS, _T_FWQB = (
    20, 21, 22, 23, 24, 25, 26, 27, 28, 29)


def _rng(seed: int, tensor: int, seq: int = 0, chunk: Optional[int] = None) -> np.random.Generator:
    key = [seed, tensor, seq] if chunk is None else [seed, tensor, seq, chunk]
    return np.random.Generator(np.random.PCG64(key))


_CHUNK = 1 << 22  # elements per independently seeded stream of a large tensor
_POOL = cf.ThreadPoolExecutor(max_workers=max(1, min(32, os.cpu_count() or 1)))
_TLS = threading.local()


def _tls_buffers():
    if getattr(_TLS, "f32", None) is None:
        _TLS.f32 = np.empty(_CHUNK, dtype=np.float32)
        _TLS.bf16 = torch.empty(_CHUNK, dtype=torch.bfloat16)
    return _TLS.f32, _TLS.bf16


def _fill_normal(dst: torch.Tensor, seed: int, tensor: int, seq: int, width: int,
                 mean: float, std: float, row_index: Optional[np.ndarray] = None,
                 nrows: Optional[int] = None) -> None:
    """Fill ``nrows`` rows of ``width`` bf16 values ~ N(mean, std^2) into the 2-D bf16
    tensor ``dst``: rows 0.. in order, or rows ``row_index[i]`` when given. Values are
    drawn in fixed chunks of _CHUNK elements, chunk i from stream (seed, tensor, seq,
    i); numpy releases the GIL, so chunks run in parallel threads and the result does
    not depend on the thread count."""
    assert _CHUNK % width == 0
    if nrows is None:
        nrows = dst.shape[0] if row_index is None else len(row_index)
    n = nrows * width

    def one(i: int) -> None:
        lo, hi = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        f32, b16 = _tls_buffers()
        x = f32[: hi - lo]
        _rng(seed, tensor, seq, i).standard_normal(out=x, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        if mean != 0.0:
            x += np.float32(mean)
        r0, r1 = lo // width, hi // width
        src = torch.from_numpy(x).view(r1 - r0, width)
        if row_index is None:
            dst[r0:r1].copy_(src)  # float32 -> bf16, nearest even
        else:
            tmp = b16[: hi - lo].view(r1 - r0, width)
            tmp.copy_(src)
            dst.index_copy_(0, torch.from_numpy(row_index[r0:r1]), tmp)

    list(_POOL.map(one, range((n + _CHUNK - 1) // _CHUNK)))


def _normal_bf16(seed: int, tensor: int, seq: int, n: int, mean: float, std: float) -> torch.Tensor:
    """n bf16 values ~ N(mean, std^2) (see ``_fill_normal``)."""
    out = torch.empty(n, dtype=torch.bfloat16)
    width = 64 if n % 64 == 0 else 1
    _fill_normal(out.view(-1, width), seed, tensor, seq, width, mean, std)
    return out


def _normal_f32(rng: np.random.Generator, shape, mean: float, std: float) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    if mean != 0.0:
        x += np.float32(mean)
    return x


def _to_bf16(x: np.ndarray) -> torch.Tensor:
    """float32 -> bf16, round to nearest even (torch's conversion)."""
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16)


@dataclasses.dataclass
class Geometry:
    """Per-layer sizes (the fields of ``Glm5NextDsaConfig`` the hot path reads)."""

    index_kpool: int
    index_heads: int
    index_head_dim: int
    index_topk: int
    heads: int
    hidden: int
    kv_lora_rank: int = 512
    first_key: int = 0
    eps: float = 1e-6
    qk_head_dim: int = 256  # GLM-5.3: q_b_proj has 256 rows per head
    always_select_tail: bool = False  # the trailing partial pool's tokens are always attended

    @property
    def index_scale(self) -> float:
        return self.index_head_dim ** -0.5

    @property
    def softmax_scale(self) -> float:
        return self.qk_head_dim ** -0.5

    @property
    def out_width(self) -> int:
        return self.index_topk + (self.index_kpool - 1 if self.always_select_tail else 0)


@dataclasses.dataclass
class Workload:
    """All host tensors of one decode (or chunked-prefill) batch, plus its geometry.

    Token-side tensors are the caches as they sit in memory; ``seq_lens`` says
    how many tokens of each sequence exist; query row ``r`` belongs to sequence
    ``row_seq[r]`` and sees the first ``row_ctx[r]`` tokens of it.
    """

    name: str
    seed: int
    geom: Geometry
    batch: int
    max_seq_len: int
    seq_lens: np.ndarray  # int32 [B]
    rows: int
    row_seq: np.ndarray  # int32 [R]
    row_ctx: np.ndarray  # int32 [R]
    block_size: Optional[int]
    block_table: Optional[torch.Tensor]  # int32 [B, max_blocks]
    num_blocks: int
    k_raw: Optional[torch.Tensor]
    gate: Optional[torch.Tensor]
    valid: Optional[torch.Tensor]
    ape: torch.Tensor
    ln_w: torch.Tensor
    ln_b: torch.Tensor
    qidx: torch.Tensor
    w: torch.Tensor
    qlat: torch.Tensor
    ckv: torch.Tensor
    o_absorb: Optional[torch.Tensor]
    # Optional directly drawn pooled-key cache (stage-isolated tests only).
    kpool_keys: Optional[torch.Tensor] = None
    kpool_valid: Optional[torch.Tensor] = None

    @property
    def paged(self) -> bool:
        return self.block_table is not None

    @property
    def max_blocks(self) -> int:
        return 0 if self.block_table is None else int(self.block_table.shape[1])

    @property
    def pool_capacity(self) -> int:
        """Pooled-key rows reserved per sequence in the contiguous layout."""
        return self.max_seq_len // self.geom.index_kpool

    @property
    def p_stride(self) -> int:
        """Score-row width: the most pools any row can see."""
        g = self.geom
        return max(0, (self.max_seq_len - g.first_key) // g.index_kpool)

    @property
    def select_k(self) -> int:
        g = self.geom
        return min(g.index_topk // g.index_kpool, self.p_stride)


def make_workload(
    name: str,
    seed: int,
    geom: Geometry,
    seq_lens: Sequence[int],
    *,
    block_size: Optional[int] = None,
    max_seq_len: Optional[int] = None,
    invalid_tail: int = 0,
    invalid_per_seq: int = 0,
    rows_ctx: Optional[Sequence[int]] = None,
    prefill_seq: int = 0,
    sequences: Optional[Sequence[int]] = None,
    with_raw: bool = True,
    with_o_absorb: bool = True,
    direct_kpool: bool = False,
    ckv_std: float = 1.0,
) -> Workload:
    """Draw one workload.

    ``invalid_tail``: the last ``n`` tokens of every sequence are marked invalid.
    ``invalid_per_seq``: that many token positions per sequence, drawn uniformly
    without replacement, are marked invalid.
    ``rows_ctx``: chunked prefill on sequence ``prefill_seq``: one query row per
    entry, seeing that many tokens; default is one decode row per sequence seeing
    all of it.
    ``sequences``: draw only these sequences' cache contents (others stay zero);
    values of a drawn sequence are identical to a full draw.
    ``direct_kpool``: also draw a pooled-key cache N(0, 0.5) with 0.2 % of pools
    invalid, for tests that isolate the score stage from compression.
    """
    g = geom
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    B = len(seq_lens)
    smax = int(max_seq_len if max_seq_len is not None else seq_lens.max())
    if rows_ctx is None:
        rows = B
        row_seq = np.arange(B, dtype=np.int32)
        row_ctx = seq_lens.astype(np.int32)
    else:
        rows = len(rows_ctx)
        row_seq = np.full(rows, prefill_seq, dtype=np.int32)
        row_ctx = np.asarray(rows_ctx, dtype=np.int32)
    want = set(range(B)) if sequences is None else set(int(s) for s in sequences)
    ihd, kvl, KP = g.index_head_dim, g.kv_lora_rank, g.index_kpool

    # Physical layout.
    if block_size is None:
        block_table = None
        num_blocks = 0
        n_tok_rows = B * smax

        def token_rows(b: int) -> np.ndarray:
            return b * smax + np.arange(int(seq_lens[b]))
    else:
        assert block_size % KP == 0
        nblk = [math.ceil(int(L) / block_size) for L in seq_lens]
        max_blocks = max(1, math.ceil(smax / block_size))
        num_blocks = int(sum(nblk))
        perm = _rng(seed, _T_PERM).permutation(num_blocks).astype(np.int32)
        bt = np.full((B, max_blocks), -1, dtype=np.int32)
        off = 0
        for b in range(B):
            bt[b, : nblk[b]] = perm[off : off + nblk[b]]
            off += nblk[b]
        block_table = torch.from_numpy(bt)
        n_tok_rows = num_blocks * block_size

        def token_rows(b: int) -> np.ndarray:
            t = np.arange(int(seq_lens[b]))
            return bt[b, t // block_size].astype(np.int64) * block_size + t % block_size

    def tok_shape(*tail):
        if block_size is None:
            return (B, smax) + tail
        return (num_blocks, block_size) + tail

    def fill_tokens(tensor_id: int, width: int, mean: float, std: float) -> torch.Tensor:
        out = torch.zeros((n_tok_rows, width), dtype=torch.bfloat16)
        for b in sorted(want):
            L = int(seq_lens[b])
            if block_size is None:
                _fill_normal(out[b * smax: b * smax + L], seed, tensor_id, b, width, mean, std)
            else:
                _fill_normal(out, seed, tensor_id, b, width, mean, std,
                             row_index=token_rows(b).astype(np.int64))
        return out.view(tok_shape(width))

    k_raw = gate = valid = None
    if with_raw:
        k_raw = fill_tokens(_T_KRAW, ihd, 0.0, 1.0)
        gate = fill_tokens(_T_GATE, ihd, 0.0, 1.0)
        v = np.zeros(n_tok_rows, dtype=np.uint8)
        for b in sorted(want):
            L = int(seq_lens[b])
            vb = np.ones(L, dtype=np.uint8)
            if invalid_tail:
                vb[max(0, L - invalid_tail) :] = 0
            if invalid_per_seq:
                bad = _rng(seed, _T_VALID, b).choice(L, size=min(L, invalid_per_seq),
                                                     replace=False)
                vb[bad] = 0
            v[token_rows(b)] = vb
        valid = torch.from_numpy(v).view(tok_shape())

    ln_w = _to_bf16(_normal_f32(_rng(seed, _T_LNW), (ihd,), 1.0, 0.1))
    ln_b = _to_bf16(_normal_f32(_rng(seed, _T_LNB), (ihd,), 0.0, 0.1))
    ape = torch.from_numpy(_normal_f32(_rng(seed, _T_APE), (KP, ihd), 0.0, 0.1))

    qidx = _normal_bf16(seed, _T_QIDX, 0, rows * g.index_heads * ihd, 0.0, 1.0).view(
        rows, g.index_heads, ihd)
    w_np = _rng(seed, _T_W).random(size=(rows, g.index_heads), dtype=np.float32)
    w_np *= np.float32(g.index_heads ** -0.5)
    w = torch.from_numpy(w_np)
    qlat = _normal_bf16(seed, _T_QLAT, 0, rows * g.heads * kvl, 0.0, 1.0).view(rows, g.heads, kvl)
    ckv = fill_tokens(_T_CKV, kvl, 0.0, ckv_std)
    o_absorb = None
    if with_o_absorb:
        o_absorb = _normal_bf16(seed, _T_OABS, 0, g.hidden * g.heads * kvl, 0.0, 0.02).view(
            g.hidden, g.heads * kvl)

    kpool_keys = kpool_valid = None
    if direct_kpool:
        ppb = None if block_size is None else block_size // KP
        if block_size is None:
            kk = torch.zeros((B, smax // KP, ihd), dtype=torch.bfloat16)
            kv = torch.zeros((B, smax // KP), dtype=torch.uint8)
        else:
            kk = torch.zeros((num_blocks, ppb, ihd), dtype=torch.bfloat16)
            kv = torch.zeros((num_blocks, ppb), dtype=torch.uint8)
        for b in sorted(want):
            P = max(0, (int(seq_lens[b]) - g.first_key) // KP)
            r = _rng(seed, _T_KPOOL, b)
            x = _normal_bf16(seed, _T_KPOOL, b, P * ihd, 0.0, 0.5).view(P, ihd)
            vv = (r.random(P) >= 0.002).astype(np.uint8)
            p = np.arange(P)
            if block_size is None:
                kk[b, :P] = x
                kv[b, :P] = torch.from_numpy(vv)
            else:
                blk = torch.from_numpy(block_table.numpy()[b, p // ppb].astype(np.int64))
                slot = torch.from_numpy(p % ppb)
                kk[blk, slot] = x
                kv[blk, slot] = torch.from_numpy(vv)
        kpool_keys, kpool_valid = kk, kv

    return Workload(
        name=name, seed=seed, geom=g, batch=B, max_seq_len=smax,
        seq_lens=seq_lens.astype(np.int32), rows=rows, row_seq=row_seq, row_ctx=row_ctx,
        block_size=block_size, block_table=block_table, num_blocks=num_blocks,
        k_raw=k_raw, gate=gate, valid=valid, ape=ape, ln_w=ln_w, ln_b=ln_b,
        qidx=qidx, w=w, qlat=qlat, ckv=ckv, o_absorb=o_absorb,
        kpool_keys=kpool_keys, kpool_valid=kpool_valid,
    )


# ---------------------------------------------------------------------------
# Projection front-end inputs (the hidden state and the weights that turn it into
# the step's inputs). Random weights with the checkpoint's shapes, scaled so every
# projection output is O(1); q_absorb is drawn directly (it is a load-time product,
# but only its shape and scale matter here).


@dataclasses.dataclass
class FrontEnd:
    x: torch.Tensor              # [R, hidden] bf16
    q_a_proj: torch.Tensor       # [q_lora, hidden]
    kv_a_proj: torch.Tensor      # [kv_lora, hidden]
    wk: torch.Tensor             # [ihd, hidden]
    compress_gate: torch.Tensor  # [ihd, hidden]
    weights_proj: torch.Tensor   # [index_heads, hidden], already x index_heads^-0.5
    q_a_norm: torch.Tensor       # [q_lora]
    kv_a_norm: torch.Tensor      # [kv_lora]
    q_absorb: torch.Tensor       # [heads * kv_lora, q_lora]
    wq_b: torch.Tensor           # [index_heads * ihd, q_lora]
    eps: float

    @property
    def q_lora_rank(self) -> int:
        return int(self.q_a_proj.shape[0])

    def packed_x_weights(self) -> torch.Tensor:
        """The five x projections as one [n_x, hidden] matrix (row concatenation in
        the order q_a, kv_a, wk, gate, weights_proj, then zero rows to a multiple of
        64): the layout the front-end streams."""
        parts = [self.q_a_proj, self.kv_a_proj, self.wk, self.compress_gate, self.weights_proj]
        n = sum(int(t.shape[0]) for t in parts)
        pad = (-n) % 64
        if pad:
            parts.append(torch.zeros((pad, self.x.shape[1]), dtype=torch.bfloat16))
        return torch.cat(parts, dim=0).contiguous()

    def packed_q_weights(self) -> torch.Tensor:
        """q_absorb with indexer.wq_b below it, [heads*kvl + index_heads*ihd, q_lora]:
        one stream over q_lora's weights."""
        return torch.cat([self.q_absorb, self.wq_b], dim=0).contiguous()


def make_frontend(g: "Geometry", rows: int, q_lora_rank: int = 1536, seed: int = 0,
                  eps: float = 1e-6) -> FrontEnd:
    hidden, kvl, ihd, hi = g.hidden, g.kv_lora_rank, g.index_head_dim, g.index_heads
    mat = lambda t, n, k, std: _normal_bf16(seed, t, 0, n * k, 0.0, std).view(n, k)
    return FrontEnd(
        x=mat(_T_FX, rows, hidden, 1.0),
        q_a_proj=mat(_T_FQA, q_lora_rank, hidden, hidden ** -0.5),
        kv_a_proj=mat(_T_FKVA, kvl, hidden, hidden ** -0.5),
        wk=mat(_T_FWK, ihd, hidden, hidden ** -0.5),
        compress_gate=mat(_T_FGATE, ihd, hidden, hidden ** -0.5),
        weights_proj=mat(_T_FWP, hi, hidden, hidden ** -0.5 * hi ** -0.5),
        q_a_norm=_normal_bf16(seed, _T_FQN, 0, q_lora_rank, 1.0, 0.1),
        kv_a_norm=_normal_bf16(seed, _T_FKVN, 0, kvl, 1.0, 0.1),
        q_absorb=mat(_T_FQABS, g.heads * kvl, q_lora_rank, q_lora_rank ** -0.5),
        wq_b=mat(_T_FWQB, hi * ihd, q_lora_rank, q_lora_rank ** -0.5),
        eps=eps,
    )


# ---------------------------------------------------------------------------
# The five named workloads.

GLM53 = dict(index_kpool=4, index_heads=32, index_head_dim=128, index_topk=2048,
             heads=64, hidden=4096)


def tiny(seed: int = 0, **kw) -> Workload:
    """Tiny single-query decode: S=2048, kpool 4, 4 indexer heads of 64, topk 256,
    4 MLA heads, hidden 1024, last 3 tokens invalid."""
    g = Geometry(index_kpool=4, index_heads=4, index_head_dim=64, index_topk=256,
                 heads=4, hidden=1024)
    return make_workload("tiny-decode-S2048", seed, g, [2048], invalid_tail=3, **kw)


def single_32k(seed: int = 1, **kw) -> Workload:
    """GLM-5.3-like single-sequence decode at S=32,768, all tokens valid."""
    return make_workload("decode-S32768-b1", seed, Geometry(**GLM53), [32768], **kw)


def paged_batch(seed: int = 2, **kw) -> Workload:
    """64 sequences, lengths uniform in [4096, 65536], 64-token blocks in a random
    permutation."""
    lens = _rng(seed, _T_LENS).integers(4096, 65536, size=64, endpoint=True)
    return make_workload("paged-decode-b64-L4k-64k", seed, Geometry(**GLM53), lens,
                         block_size=64, max_seq_len=65536, **kw)


def long_262k(seed: int = 3, seq_len: Optional[int] = None, **kw) -> Workload:
    """8 sequences at S=262,144, 1 % of token positions invalid (2,621 per sequence).
    ``seq_len`` shrinks the sequences (same rows, heads and top-k) for profiling."""
    S = seq_len or 262144
    name = "decode-S262144-b8" if seq_len is None else f"decode-S{S}-b8"
    return make_workload(name, seed, Geometry(**GLM53), [S] * 8,
                         invalid_per_seq=(S * 2621 + 131072) // 262144, **kw)


def prefill_chunk(seed: int = 4, rows: Optional[int] = None, **kw) -> Workload:
    """Chunked prefill: 4,096 query rows; row i sees the first 126,977 + i of
    131,072 tokens. ``rows`` keeps only the last rows of the chunk (same context
    lengths as in the full chunk) for profiling."""
    n = rows or 4096
    name = "prefill-Q4096-S131072" if rows is None else f"prefill-Q{n}-S131072"
    return make_workload(name, seed, Geometry(**GLM53), [131072],
                         rows_ctx=[126977 + i for i in range(4096 - n, 4096)], **kw)


WORKLOADS = {0: tiny, 1: single_32k, 2: paged_batch, 3: long_262k, 4: prefill_chunk}
