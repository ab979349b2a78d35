"""Python binding of libdsa: the C-ABI entry points with the same names, taking
torch CUDA tensors. Argument marshalling only: shape/dtype/device checks, then
``data_ptr()`` and the current stream go to the C call. Every computation runs in
the library's CUDA kernels; there is no fallback.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _lib
from ._lib import DsaPaging, check

__all__ = ["paging", "dsa_compress", "dsa_compress_append", "dsa_indexer_store",
           "dsa_write_geom", "dsa_decode_append", "dsa_decode_append_fp8", "dsa_score", "dsa_score_prefill", "dsa_select", "dsa_expand",
           "dsa_select_expand", "dsa_expand_tail", "dsa_select_expand_tail",
           "dsa_sparse_mla_decode_workspace", "dsa_sparse_mla_decode",
           "dsa_sparse_mla_decode_noalloc", "dsa_sparse_mla_decode_fp8", "dsa_quantize_latent",
           "dsa_frontend_workspace", "dsa_frontend", "dsa_latent_project_workspace",
           "dsa_latent_project", "dsa_select_k",
           "dsa_validate_config", "dsa_prefetch_l2", "dsa_set_option", "dsa_get_option", "mla_kernel",
           "select_kernel", "project_kernel", "DsaPaging"]


def _ptr(t: Optional[torch.Tensor], dtype=None, name: str = "tensor",
         host_ok: bool = False) -> Optional[int]:
    """Device address of t. With host_ok, pinned host memory is accepted too: under
    unified addressing its address is valid in kernels, which then read or write it
    directly (no copy)."""
    if t is None:
        return None
    if not t.is_cuda and not (host_ok and t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor" + (" or pinned host memory" if host_ok else ""))
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def dsa_set_option(option: int, value: int) -> None:
    """Set a process-wide launch option (DSA_OPT_* in include/dsa.h)."""
    check(_lib.load().dsa_set_option(int(option), int(value)))


def dsa_get_option(option: int) -> int:
    """Current value of a launch option (-1 for an unknown option)."""
    return int(_lib.load().dsa_get_option(int(option)))


class mla_kernel:
    """Context manager pinning the sparse-attention kernel: "auto", "tcgen05" (the
    persistent tensor-core split kernel where it supports the shape), "mma" (the
    mma.sync split kernel) or "cluster" (the tensor-core decode kernel that merges a
    row's splits inside a cluster); the previous choice is restored on exit."""

    _VALUES = {"auto": _lib.DSA_MLA_KERNEL_AUTO, "tcgen05": _lib.DSA_MLA_KERNEL_TCGEN05,
               "mma": _lib.DSA_MLA_KERNEL_MMA, "cluster": _lib.DSA_MLA_KERNEL_CLUSTER}

    def __init__(self, which: str):
        if which not in self._VALUES:
            raise ValueError(f"kernel {which!r}: one of {sorted(self._VALUES)}")
        self.value = self._VALUES[which]
        self.prev = None

    def __enter__(self):
        self.prev = dsa_get_option(_lib.DSA_OPT_MLA_KERNEL)
        dsa_set_option(_lib.DSA_OPT_MLA_KERNEL, self.value)
        return self

    def __exit__(self, *exc):
        dsa_set_option(_lib.DSA_OPT_MLA_KERNEL, self.prev)
        return False


class select_kernel:
    """Context manager pinning how clustered rows are selected: "merge" (the
    default) or "radix"; the previous choice is restored on exit."""

    _VALUES = {"merge": _lib.DSA_SELECT_KERNEL_MERGE, "radix": _lib.DSA_SELECT_KERNEL_RADIX}

    def __init__(self, which: str):
        if which not in self._VALUES:
            raise ValueError(f"kernel {which!r}: one of {sorted(self._VALUES)}")
        self.value = self._VALUES[which]
        self.prev = None

    def __enter__(self):
        self.prev = dsa_get_option(_lib.DSA_OPT_SELECT_KERNEL)
        dsa_set_option(_lib.DSA_OPT_SELECT_KERNEL, self.value)
        return self

    def __exit__(self, *exc):
        dsa_set_option(_lib.DSA_OPT_SELECT_KERNEL, self.prev)
        return False


class project_kernel:
    """Context manager pinning the projection kernel: "auto" (the default),
    "tcgen05" or "mma"; the previous choice is restored on exit."""

    _VALUES = {"auto": _lib.DSA_PROJECT_KERNEL_AUTO, "tcgen05": _lib.DSA_PROJECT_KERNEL_TCGEN05,
               "mma": _lib.DSA_PROJECT_KERNEL_MMA}

    def __init__(self, which: str):
        if which not in self._VALUES:
            raise ValueError(f"kernel {which!r}: one of {sorted(self._VALUES)}")
        self.value = self._VALUES[which]
        self.prev = None

    def __enter__(self):
        self.prev = dsa_get_option(_lib.DSA_OPT_PROJECT_KERNEL)
        dsa_set_option(_lib.DSA_OPT_PROJECT_KERNEL, self.value)
        return self

    def __exit__(self, *exc):
        dsa_set_option(_lib.DSA_OPT_PROJECT_KERNEL, self.prev)
        return False


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def paging(seq_lens: torch.Tensor, max_seq_len: int, block_table: Optional[torch.Tensor] = None,
           block_size: int = 0, num_blocks: int = 0) -> DsaPaging:
    """Describe where sequences live (see ``dsa_paging`` in include/dsa.h).

    The tensors must outlive every call that uses the returned descriptor."""
    pg = DsaPaging()
    pg.batch = int(seq_lens.numel())
    pg.max_seq_len = int(max_seq_len)
    pg.seq_lens = _ptr(seq_lens, torch.int32, "seq_lens")
    if block_table is not None:
        pg.block_table = _ptr(block_table, torch.int32, "block_table")
        pg.max_blocks = int(block_table.shape[1])
        pg.block_size = int(block_size)
        pg.num_blocks = int(num_blocks)
    else:
        pg.block_table = None
        pg.max_blocks = 0
        pg.block_size = 0
        pg.num_blocks = 0
    return pg


def dsa_validate_config(index_kpool: int, index_topk: int, kv_lora_rank: int,
                        local_heads: int) -> None:
    check(_lib.load().dsa_validate_config(index_kpool, index_topk, kv_lora_rank, local_heads))


def dsa_select_k(index_topk: int, kpool: int, n_pools: int) -> int:
    return _lib.load().dsa_select_k(index_topk, kpool, n_pools)


def dsa_compress(k_raw, gate, token_valid, ape, ln_w, ln_b, eps: float, pg: DsaPaging,
                 first_key: int, kpool: int, kpool_out, pool_valid, pool_idx=None, status=None,
                 stream=None) -> None:
    ihd = int(k_raw.shape[-1])
    check(_lib.load().dsa_compress(
        _ptr(k_raw, torch.bfloat16, "k_raw"), _ptr(gate, torch.bfloat16, "gate"),
        _ptr(token_valid, torch.uint8, "token_valid"), _ptr(ape, torch.float32, "ape"),
        _ptr(ln_w, torch.bfloat16, "ln_w"), _ptr(ln_b, torch.bfloat16, "ln_b"), float(eps),
        ctypes.byref(pg), int(first_key), int(kpool), ihd,
        _ptr(kpool_out, torch.bfloat16, "kpool_out"), _ptr(pool_valid, torch.uint8, "pool_valid"),
        _ptr(pool_idx, torch.int32, "pool_idx"), _ptr(status, torch.int32, "status"),
        _stream(stream)))


def dsa_compress_append(k_raw, gate, token_valid, ape, ln_w, ln_b, eps: float, pg: DsaPaging,
                        first_key: int, kpool: int, new_tokens: int, kpool_out, pool_valid,
                        pool_idx=None, status=None, stream=None) -> None:
    """dsa_compress for the pools the last ``new_tokens`` tokens of each sequence
    completed (the lengths are read on the device)."""
    ihd = int(k_raw.shape[-1])
    check(_lib.load().dsa_compress_append(
        _ptr(k_raw, torch.bfloat16, "k_raw"), _ptr(gate, torch.bfloat16, "gate"),
        _ptr(token_valid, torch.uint8, "token_valid"), _ptr(ape, torch.float32, "ape"),
        _ptr(ln_w, torch.bfloat16, "ln_w"), _ptr(ln_b, torch.bfloat16, "ln_b"), float(eps),
        ctypes.byref(pg), int(first_key), int(kpool), ihd, int(new_tokens),
        _ptr(kpool_out, torch.bfloat16, "kpool_out"), _ptr(pool_valid, torch.uint8, "pool_valid"),
        _ptr(pool_idx, torch.int32, "pool_idx"), _ptr(status, torch.int32, "status"),
        _stream(stream)))


def dsa_indexer_store(k_new, gate_new, pg: DsaPaging, seq_lens, k_raw, gate, token_valid,
                      ckv_new=None, ckv=None, status=None, stream=None) -> None:
    """Append one staged token per sequence at its current length (read on the
    device) and advance ``seq_lens`` (the tensor ``pg`` was built from)."""
    batch, ihd = (int(x) for x in k_new.shape)
    if tuple(gate_new.shape) != (batch, ihd):
        raise ValueError(f"gate_new must be [{batch}, {ihd}]")
    kvl = int(ckv_new.shape[-1]) if ckv_new is not None else 0
    check(_lib.load().dsa_indexer_store(
        _ptr(k_new, torch.bfloat16, "k_new"), _ptr(gate_new, torch.bfloat16, "gate_new"),
        _ptr(ckv_new, torch.bfloat16, "ckv_new"), ihd, kvl, ctypes.byref(pg),
        _ptr(seq_lens, torch.int32, "seq_lens"), _ptr(k_raw, torch.bfloat16, "k_raw"),
        _ptr(gate, torch.bfloat16, "gate"), _ptr(token_valid, torch.uint8, "token_valid"),
        _ptr(ckv, torch.bfloat16, "ckv"), _ptr(status, torch.int32, "status"), _stream(stream)))


def dsa_write_geom(seq_lens, row_seq, row_ctx, status=None, stream=None) -> None:
    """row_ctx[r] = seq_lens[row_seq[r]] on the device (row_seq None: r)."""
    check(_lib.load().dsa_write_geom(
        _ptr(seq_lens, torch.int32, "seq_lens"), int(seq_lens.numel()),
        _ptr(row_seq, torch.int32, "row_seq"), int(row_ctx.numel()),
        _ptr(row_ctx, torch.int32, "row_ctx"), _ptr(status, torch.int32, "status"),
        _stream(stream)))


def dsa_decode_append(k_new, gate_new, ape, ln_w, ln_b, eps: float, pg: DsaPaging, seq_lens,
                      first_key: int, kpool: int, k_raw, gate, token_valid, kpool_out, pool_valid,
                      ckv_new=None, ckv=None, pool_idx=None, row_ctx=None, status=None,
                      stream=None) -> None:
    """dsa_indexer_store + dsa_write_geom + dsa_compress_append(new_tokens=1) in one
    launch (identical results)."""
    batch, ihd = (int(x) for x in k_new.shape)
    if tuple(gate_new.shape) != (batch, ihd):
        raise ValueError(f"gate_new must be [{batch}, {ihd}]")
    kvl = int(ckv_new.shape[-1]) if ckv_new is not None else 0
    check(_lib.load().dsa_decode_append(
        _ptr(k_new, torch.bfloat16, "k_new"), _ptr(gate_new, torch.bfloat16, "gate_new"),
        _ptr(ckv_new, torch.bfloat16, "ckv_new"), _ptr(ape, torch.float32, "ape"),
        _ptr(ln_w, torch.bfloat16, "ln_w"), _ptr(ln_b, torch.bfloat16, "ln_b"), float(eps),
        ctypes.byref(pg), _ptr(seq_lens, torch.int32, "seq_lens"), int(first_key), int(kpool),
        ihd, kvl, _ptr(k_raw, torch.bfloat16, "k_raw"), _ptr(gate, torch.bfloat16, "gate"),
        _ptr(token_valid, torch.uint8, "token_valid"), _ptr(ckv, torch.bfloat16, "ckv"),
        _ptr(kpool_out, torch.bfloat16, "kpool_out"), _ptr(pool_valid, torch.uint8, "pool_valid"),
        _ptr(pool_idx, torch.int32, "pool_idx"), _ptr(row_ctx, torch.int32, "row_ctx"),
        _ptr(status, torch.int32, "status"), _stream(stream)))


def dsa_decode_append_fp8(k_new, gate_new, ckv_new, ape, ln_w, ln_b, eps: float, pg: DsaPaging,
                          seq_lens, first_key: int, kpool: int, k_raw, gate, token_valid,
                          ckv_codes, ckv_scales, kpool_out, pool_valid, ckv=None, pool_idx=None,
                          row_ctx=None, status=None, stream=None) -> None:
    """dsa_decode_append that also encodes the staged latent row into the FP8 cache
    (same codec and bytes as dsa_quantize_latent); the bf16 cache ``ckv`` is optional."""
    batch, ihd = (int(x) for x in k_new.shape)
    if tuple(gate_new.shape) != (batch, ihd):
        raise ValueError(f"gate_new must be [{batch}, {ihd}]")
    kvl = int(ckv_new.shape[-1])
    if int(ckv_codes.shape[-1]) != kvl or int(ckv_scales.shape[-1]) != kvl // 128:
        raise ValueError(f"ckv_codes must be [.., {kvl}] and ckv_scales [.., {kvl // 128}]")
    check(_lib.load().dsa_decode_append_fp8(
        _ptr(k_new, torch.bfloat16, "k_new"), _ptr(gate_new, torch.bfloat16, "gate_new"),
        _ptr(ckv_new, torch.bfloat16, "ckv_new"), _ptr(ape, torch.float32, "ape"),
        _ptr(ln_w, torch.bfloat16, "ln_w"), _ptr(ln_b, torch.bfloat16, "ln_b"), float(eps),
        ctypes.byref(pg), _ptr(seq_lens, torch.int32, "seq_lens"), int(first_key), int(kpool),
        ihd, kvl, _ptr(k_raw, torch.bfloat16, "k_raw"), _ptr(gate, torch.bfloat16, "gate"),
        _ptr(token_valid, torch.uint8, "token_valid"), _ptr(ckv, torch.bfloat16, "ckv"),
        _ptr(ckv_codes, torch.uint8, "ckv_codes"), _ptr(ckv_scales, torch.float32, "ckv_scales"),
        _ptr(kpool_out, torch.bfloat16, "kpool_out"), _ptr(pool_valid, torch.uint8, "pool_valid"),
        _ptr(pool_idx, torch.int32, "pool_idx"), _ptr(row_ctx, torch.int32, "row_ctx"),
        _ptr(status, torch.int32, "status"), _stream(stream)))


def dsa_score(qidx, w, row_seq, row_ctx, kpool, pool_valid, pg: DsaPaging, first_key: int,
              kpool_size: int, scale: float, scores, status=None, stream=None) -> None:
    rows, heads, ihd = (int(x) for x in qidx.shape)
    if tuple(w.shape) != (rows, heads):
        raise ValueError(f"w must be [{rows}, {heads}]")
    if scores.dim() != 2 or scores.shape[0] != rows:
        raise ValueError("scores must be [rows, p_stride]")
    check(_lib.load().dsa_score(
        _ptr(qidx, torch.bfloat16, "qidx"), _ptr(w, torch.float32, "w"), rows, heads, ihd,
        _ptr(row_seq, torch.int32, "row_seq"), _ptr(row_ctx, torch.int32, "row_ctx"),
        _ptr(kpool, torch.bfloat16, "kpool"), _ptr(pool_valid, torch.uint8, "pool_valid"),
        ctypes.byref(pg), int(first_key), int(kpool_size), float(scale),
        _ptr(scores, torch.float32, "scores"), int(scores.shape[1]),
        _ptr(status, torch.int32, "status"), _stream(stream)))


def dsa_score_prefill(qidx, w, seq: int, row_ctx, kpool, pool_valid, pg: DsaPaging,
                      first_key: int, kpool_size: int, scale: float, scores, status=None,
                      stream=None) -> None:
    """Index scores of a chunk of query rows of sequence ``seq`` on the tensor cores
    (contiguous pooled-key cache; index_heads in {32, 64, 128})."""
    rows, heads, ihd = (int(x) for x in qidx.shape)
    if tuple(w.shape) != (rows, heads):
        raise ValueError(f"w must be [{rows}, {heads}]")
    if scores.dim() != 2 or scores.shape[0] != rows:
        raise ValueError("scores must be [rows, p_stride]")
    check(_lib.load().dsa_score_prefill(
        _ptr(qidx, torch.bfloat16, "qidx"), _ptr(w, torch.float32, "w"), rows, heads, ihd,
        int(seq), _ptr(row_ctx, torch.int32, "row_ctx"),
        _ptr(kpool, torch.bfloat16, "kpool"), _ptr(pool_valid, torch.uint8, "pool_valid"),
        ctypes.byref(pg), int(first_key), int(kpool_size), float(scale),
        _ptr(scores, torch.float32, "scores"), int(scores.shape[1]),
        _ptr(status, torch.int32, "status"), _stream(stream)))


def dsa_select(scores, index_topk: int, kpool: int, pool_ids, stream=None) -> None:
    rows, p_stride = (int(x) for x in scores.shape)
    sk = dsa_select_k(index_topk, kpool, p_stride)
    if tuple(pool_ids.shape) != (rows, max(sk, 0)):
        raise ValueError(f"pool_ids must be [{rows}, {sk}]")
    check(_lib.load().dsa_select(
        _ptr(scores, torch.float32, "scores"), rows, p_stride, int(index_topk), int(kpool),
        _ptr(pool_ids, torch.int32, "pool_ids"), _stream(stream)))


def dsa_select_expand(scores, index_topk: int, kpool: int, first_key: int, pool_ids, token_ids,
                      stream=None) -> None:
    """dsa_select and dsa_expand in one launch (identical results)."""
    rows, p_stride = (int(x) for x in scores.shape)
    sk = dsa_select_k(index_topk, kpool, p_stride)
    if tuple(pool_ids.shape) != (rows, max(sk, 0)):
        raise ValueError(f"pool_ids must be [{rows}, {sk}]")
    if token_ids.dim() != 2 or token_ids.shape[0] != rows:
        raise ValueError("token_ids must be [rows, out_width]")
    check(_lib.load().dsa_select_expand(
        _ptr(scores, torch.float32, "scores"), rows, p_stride, int(index_topk), int(kpool),
        int(first_key), int(token_ids.shape[1]), _ptr(pool_ids, torch.int32, "pool_ids"),
        _ptr(token_ids, torch.int32, "token_ids"), _stream(stream)))


def dsa_expand(pool_ids, first_key: int, kpool: int, token_ids, stream=None) -> None:
    rows, sk = (int(x) for x in pool_ids.shape)
    if token_ids.dim() != 2 or token_ids.shape[0] != rows:
        raise ValueError("token_ids must be [rows, out_width]")
    check(_lib.load().dsa_expand(
        _ptr(pool_ids, torch.int32, "pool_ids"), rows, sk, int(first_key), int(kpool),
        int(token_ids.shape[1]), _ptr(token_ids, torch.int32, "token_ids"), _stream(stream)))


def dsa_expand_tail(pool_ids, first_key: int, kpool: int, index_topk: int, row_ctx, token_ids,
                    stream=None) -> None:
    """dsa_expand with always_select_tail: the trailing partial pool's tokens of
    each row (row_ctx [rows] i32) follow the pools from position index_topk on."""
    rows, sk = (int(x) for x in pool_ids.shape)
    if token_ids.dim() != 2 or token_ids.shape[0] != rows:
        raise ValueError("token_ids must be [rows, out_width]")
    if tuple(row_ctx.shape) != (rows,):
        raise ValueError(f"row_ctx must be [{rows}]")
    check(_lib.load().dsa_expand_tail(
        _ptr(pool_ids, torch.int32, "pool_ids"), rows, sk, int(first_key), int(kpool),
        int(index_topk), _ptr(row_ctx, torch.int32, "row_ctx"), int(token_ids.shape[1]),
        _ptr(token_ids, torch.int32, "token_ids"), _stream(stream)))


def dsa_select_expand_tail(scores, index_topk: int, kpool: int, first_key: int, row_ctx,
                           pool_ids, token_ids, stream=None) -> None:
    """dsa_select and dsa_expand_tail in one launch (identical results)."""
    rows, p_stride = (int(x) for x in scores.shape)
    sk = dsa_select_k(index_topk, kpool, p_stride)
    if tuple(pool_ids.shape) != (rows, max(sk, 0)):
        raise ValueError(f"pool_ids must be [{rows}, {sk}]")
    if token_ids.dim() != 2 or token_ids.shape[0] != rows:
        raise ValueError("token_ids must be [rows, out_width]")
    if tuple(row_ctx.shape) != (rows,):
        raise ValueError(f"row_ctx must be [{rows}]")
    check(_lib.load().dsa_select_expand_tail(
        _ptr(scores, torch.float32, "scores"), rows, p_stride, int(index_topk), int(kpool),
        int(first_key), _ptr(row_ctx, torch.int32, "row_ctx"), int(token_ids.shape[1]),
        _ptr(pool_ids, torch.int32, "pool_ids"), _ptr(token_ids, torch.int32, "token_ids"),
        _stream(stream)))


def dsa_sparse_mla_decode_workspace(rows: int, heads: int, out_width: int, hidden: int,
                                    with_o_absorb: bool, kv_lora_rank: int = 512) -> int:
    n = ctypes.c_size_t(0)
    check(_lib.load().dsa_sparse_mla_decode_workspace(
        int(rows), int(heads), int(kv_lora_rank), int(out_width), int(hidden),
        1 if with_o_absorb else 0, ctypes.byref(n)))
    return int(n.value)


def dsa_sparse_mla_decode(qlat, row_seq, ckv, pg: DsaPaging, token_ids, softmax_scale: float,
                          o_absorb=None, y=None, olat=None, status=None, workspace=None,
                          stream=None) -> None:
    rows, heads, kvl = (int(x) for x in qlat.shape)
    ow = int(token_ids.shape[1])
    hidden = int(o_absorb.shape[0]) if o_absorb is not None else 0
    if o_absorb is not None and tuple(o_absorb.shape) != (hidden, heads * kvl):
        raise ValueError(f"o_absorb must be [hidden, {heads * kvl}]")
    if y is not None and tuple(y.shape) != (rows, hidden):
        raise ValueError(f"y must be [{rows}, {hidden}]")
    if olat is not None and tuple(olat.shape) != (rows, heads, kvl):
        raise ValueError(f"olat must be [{rows}, {heads}, {kvl}]")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    check(_lib.load().dsa_sparse_mla_decode(
        _ptr(qlat, torch.bfloat16, "qlat"), rows, heads, kvl,
        _ptr(row_seq, torch.int32, "row_seq"), _ptr(ckv, torch.bfloat16, "ckv"),
        ctypes.byref(pg), _ptr(token_ids, torch.int32, "token_ids"), ow, float(softmax_scale),
        _ptr(o_absorb, torch.bfloat16, "o_absorb"), hidden,
        _ptr(y, torch.bfloat16, "y", host_ok=True),
        _ptr(olat, torch.float32, "olat"), _ptr(status, torch.int32, "status"),
        _ptr(workspace, None, "workspace"), ws_bytes, _stream(stream)))


def dsa_sparse_mla_decode_fp8(qlat, row_seq, ckv_codes, ckv_scales, pg: DsaPaging, token_ids,
                              softmax_scale: float, o_absorb=None, y=None, olat=None,
                              status=None, workspace=None, stream=None) -> None:
    """dsa_sparse_mla_decode over an FP8 latent cache (E4M3 codes + per-128-channel
    power-of-two scales, see dsa_quantize_latent)."""
    rows, heads, kvl = (int(x) for x in qlat.shape)
    ow = int(token_ids.shape[1])
    hidden = int(o_absorb.shape[0]) if o_absorb is not None else 0
    if o_absorb is not None and tuple(o_absorb.shape) != (hidden, heads * kvl):
        raise ValueError(f"o_absorb must be [hidden, {heads * kvl}]")
    if y is not None and tuple(y.shape) != (rows, hidden):
        raise ValueError(f"y must be [{rows}, {hidden}]")
    if olat is not None and tuple(olat.shape) != (rows, heads, kvl):
        raise ValueError(f"olat must be [{rows}, {heads}, {kvl}]")
    if ckv_codes.shape[-1] != kvl or ckv_scales.shape[-1] != kvl // 128:
        raise ValueError("ckv_codes must be [..., kvl] and ckv_scales [..., kvl/128]")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    check(_lib.load().dsa_sparse_mla_decode_fp8(
        _ptr(qlat, torch.bfloat16, "qlat"), rows, heads, kvl,
        _ptr(row_seq, torch.int32, "row_seq"), _ptr(ckv_codes, torch.uint8, "ckv_codes"),
        _ptr(ckv_scales, torch.float32, "ckv_scales"), ctypes.byref(pg),
        _ptr(token_ids, torch.int32, "token_ids"), ow, float(softmax_scale),
        _ptr(o_absorb, torch.bfloat16, "o_absorb"), hidden, _ptr(y, torch.bfloat16, "y", host_ok=True),
        _ptr(olat, torch.float32, "olat"), _ptr(status, torch.int32, "status"),
        _ptr(workspace, None, "workspace"), ws_bytes, _stream(stream)))


def dsa_quantize_latent(x, codes, scales, stream=None) -> None:
    """FP8 latent cache from bf16 rows: codes [..., kvl] u8, scales [..., kvl/128] f32."""
    kvl = int(x.shape[-1])
    rows = x.numel() // kvl
    if codes.numel() != x.numel() or scales.numel() != rows * (kvl // 128):
        raise ValueError("codes must match x and scales hold kvl/128 per row")
    check(_lib.load().dsa_quantize_latent(
        _ptr(x, torch.bfloat16, "x"), rows, kvl, _ptr(codes, torch.uint8, "codes"),
        _ptr(scales, torch.float32, "scales"), _stream(stream)))


def dsa_frontend_workspace(rows: int, hidden: int, n_x: int, q_lora_rank: int, kv_lora_rank: int,
                           ihd: int, index_heads: int, heads: int) -> int:
    n = ctypes.c_size_t(0)
    check(_lib.load().dsa_frontend_workspace(int(rows), int(hidden), int(n_x), int(q_lora_rank),
                                             int(kv_lora_rank), int(ihd), int(index_heads),
                                             int(heads), ctypes.byref(n)))
    return int(n.value)


def dsa_frontend(x, w_x, q_a_norm, kv_a_norm, eps: float, w_q, qlat, qidx, w, k_new, gate_new,
                 ckv_new, status=None, workspace=None, stream=None) -> None:
    """The step's inputs from the hidden state (see dsa_frontend in include/dsa.h):
    w_x packs the five x projections, w_q packs q_absorb over indexer.wq_b."""
    rows, hidden = (int(v) for v in x.shape)
    n_x = int(w_x.shape[0])
    ql, kvl = int(q_a_norm.numel()), int(kv_a_norm.numel())
    _, heads, kvl2 = (int(v) for v in qlat.shape)
    _, hi, ihd = (int(v) for v in qidx.shape)
    if kvl2 != kvl or tuple(w_x.shape) != (n_x, hidden):
        raise ValueError("qlat's width must be kv_lora_rank and w_x [n_x, hidden]")
    if tuple(w_q.shape) != (heads * kvl + hi * ihd, ql):
        raise ValueError("w_q must be [heads*kvl + index_heads*ihd, q_lora]")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    check(_lib.load().dsa_frontend(
        _ptr(x, torch.bfloat16, "x"), rows, hidden, _ptr(w_x, torch.bfloat16, "w_x"), n_x, ql, kvl,
        ihd, hi, _ptr(q_a_norm, torch.bfloat16, "q_a_norm"),
        _ptr(kv_a_norm, torch.bfloat16, "kv_a_norm"), float(eps),
        _ptr(w_q, torch.bfloat16, "w_q"), heads,
        _ptr(qlat, torch.bfloat16, "qlat"), _ptr(qidx, torch.bfloat16, "qidx"),
        _ptr(w, torch.float32, "w"), _ptr(k_new, torch.bfloat16, "k_new"),
        _ptr(gate_new, torch.bfloat16, "gate_new"), _ptr(ckv_new, torch.bfloat16, "ckv_new"),
        _ptr(status, torch.int32, "status"), _ptr(workspace, None, "workspace"), ws_bytes,
        _stream(stream)))


def dsa_latent_project_workspace(rows: int, heads: int, hidden: int,
                                 kv_lora_rank: int = 512) -> int:
    n = ctypes.c_size_t(0)
    check(_lib.load().dsa_latent_project_workspace(int(rows), int(heads), int(kv_lora_rank),
                                                   int(hidden), ctypes.byref(n)))
    return int(n.value)


def dsa_prefetch_l2(t: torch.Tensor, nbytes: Optional[int] = None, stream=None) -> None:
    """Bring the first nbytes of device tensor t (all of it by default) into L2: a hint
    issued beside latency-bound work, e.g. on a second stream."""
    total = t.numel() * t.element_size()
    n = total if nbytes is None else min(int(nbytes), total)
    check(_lib.load().dsa_prefetch_l2(_ptr(t, None, "t"), n, _stream(stream)))


def dsa_latent_project(olat, o_absorb, y, status=None, workspace=None, stream=None) -> None:
    """y = bf16(o_absorb @ bf16(olat)) per row; olat [rows, heads, 512] f32."""
    rows, heads, kvl = (int(x) for x in olat.shape)
    hidden = int(o_absorb.shape[0])
    if tuple(o_absorb.shape) != (hidden, heads * kvl) or tuple(y.shape) != (rows, hidden):
        raise ValueError("o_absorb must be [hidden, heads*kvl] and y [rows, hidden]")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    check(_lib.load().dsa_latent_project(
        _ptr(olat, torch.float32, "olat"), rows, heads, kvl, _ptr(o_absorb, torch.bfloat16, "o_absorb"),
        hidden, _ptr(y, torch.bfloat16, "y", host_ok=True), _ptr(status, torch.int32, "status"),
        _ptr(workspace, None, "workspace"), ws_bytes, _stream(stream)))


def dsa_sparse_mla_decode_noalloc(qlat, row_seq, ckv, pg: DsaPaging, token_ids,
                                  softmax_scale: float, o_absorb=None, y=None, olat=None,
                                  status=None, stream=None) -> None:
    """dsa_sparse_mla_decode without a workspace: the library's fixed scratch array
    is used instead (for hosts that cannot allocate device memory; see
    include/dsa.h). Calls whose GPU work overlaps in time must be serialised."""
    rows, heads, kvl = (int(x) for x in qlat.shape)
    ow = int(token_ids.shape[1])
    hidden = int(o_absorb.shape[0]) if o_absorb is not None else 0
    check(_lib.load().dsa_sparse_mla_decode_noalloc(
        _ptr(qlat, torch.bfloat16, "qlat"), rows, heads, kvl,
        _ptr(row_seq, torch.int32, "row_seq"), _ptr(ckv, torch.bfloat16, "ckv"),
        ctypes.byref(pg), _ptr(token_ids, torch.int32, "token_ids"), ow, float(softmax_scale),
        _ptr(o_absorb, torch.bfloat16, "o_absorb"), hidden, _ptr(y, torch.bfloat16, "y", host_ok=True),
        _ptr(olat, torch.float32, "olat"), _ptr(status, torch.int32, "status"),
        _stream(stream)))
