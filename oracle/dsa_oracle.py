"""CPU oracle for one DSA decode layer (k-pooled indexer + sparse latent MLA).

TEST INFRASTRUCTURE. Only the tests, the package smoke check and the benchmark's
CPU-baseline leg may import or run this module. The product path never does: it
runs CUDA kernels or fails.

Plain float64 numpy, single-threaded where the BLAS is held to one thread,
written for a reader to check against the pages by eye. Library primitives
(a matrix product, a sort) serve as steps; there is no blocking, fusion or
reordering beyond what the definitions state. bf16 rounding (nearest even) is
applied only where the layer stores bf16: the normalised indexer keys, the pooled
keys, and the output ``y``.

Sources (page title, section):

* ``metrale_model_arch/glm5next_dsa/mod.rs``, module doc, "Shape of the pipeline"
  and "Checkpoint and kernel facts the code depends on"; ``Glm5NextDsaConfig``
  methods ``select_k`` and ``out_width``.
* ``metrale_model_arch/glm5next_dsa/tp.rs``, module doc, "Why the indexer is
  replicated" (the index-score formula).
* ``metrale_model_arch/glm5next_dsa/build.rs``, module doc "The transforms, each
  done once at load", ``absorb_q`` and ``absorb_o``.

Every function here is pinned by a CPU test against values or identities fixed
independently of it (tests/test_oracle_pins.py, tests/golden/); none is "parity
unpinned".
"""
from __future__ import annotations

import math
from typing import Optional

import numpy as np

F64 = np.float64


# ---------------------------------------------------------------------------
# bf16 storage rounding


def bf16_round(x) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value, ties to even.

    bfloat16 has 8 significant bits and float32's exponent range (normal numbers
    down to 2^-126, subnormal spacing 2^-133, largest finite 65280 * 2^112).
    The host uploads of the layer round this way (``build.rs``, ``up_bf16``:
    ``half::bf16::from_f32``).
    """
    x = np.asarray(x, dtype=F64)
    _, e = np.frexp(x)  # x = m * 2**e, 0.5 <= |m| < 1 (e = 0 for 0, inf, nan)
    # quantum = 2**(exponent of the leading bit - 7); subnormals share 2**-133.
    q = np.ldexp(1.0, np.maximum(e - 1, -126) - 7)
    r = np.rint(x / q) * q  # rint: round half to even; x/q is exact
    big = np.ldexp(F64(255.0), 120)  # largest finite bf16 = 255 * 2^120
    r = np.where(np.abs(r) > big, np.copysign(np.inf, r), r)
    return np.where(np.isfinite(x), r, x)


# ---------------------------------------------------------------------------
# (a1) k_norm + kpool_compress


def layernorm_bias(x, gamma, beta, eps: float) -> np.ndarray:
    """``indexer.k_norm``: a LayerNorm with a bias over the last axis.

    ``(x - mean) / sqrt(var + eps) * gamma + beta`` with the biased variance.
    mod.rs, "Checkpoint and kernel facts": k_norm is a LayerNorm with a bias (an
    RMSNorm would drop the mean and the bias). Returns float64, before the bf16
    store.
    """
    x = np.asarray(x, dtype=F64)
    d = x - x.mean(axis=-1, keepdims=True)
    var = (d * d).mean(axis=-1, keepdims=True)
    return d / np.sqrt(var + F64(eps)) * np.asarray(gamma, F64) + np.asarray(beta, F64)


def kpool_compress(k_tok, gate_tok, valid_tok, ape, gamma, beta, eps: float,
                   first_key: int, kpool: int):
    """Pool one sequence's indexer keys (``dsa_kpool_compress`` after ``k_norm``).

    Inputs are token-major for ONE sequence in logical order: ``k_tok`` and
    ``gate_tok`` ``[S, ihd]``, ``valid_tok [S]``, ``ape [kpool, ihd]``.

    mod.rs "Shape of the pipeline": ``k, gate, valid, ape -> kpool_compress ->
    pool keys/indices/valid``. mod.rs "Checkpoint and kernel facts": the pool
    softmax runs over the pool-slot axis, per channel; pooling starts at
    ``first_key``; a pool counts only if every one of its slots is valid, so a
    trailing partial pool is not a pool.

    Pool ``p`` holds tokens ``t_s = first_key + p*kpool + s``, ``s < kpool``:
    ``kn = bf16(LN(k))``; logit ``l_s[c] = gate[t_s, c] + ape[s, c]``;
    ``kpool[p, c] = bf16(sum_s softmax_s(l[:, c])_s * kn[t_s, c])``.
    Invalid pools are written as zeros (only their flag is read downstream).

    Returns ``(keys [P, ihd] float64 of bf16 values, pool_valid [P] uint8,
    pool_idx [P, kpool] int64)``.
    """
    k_tok = np.asarray(k_tok, dtype=F64)
    gate_tok = np.asarray(gate_tok, dtype=F64)
    valid_tok = np.asarray(valid_tok)
    S, ihd = k_tok.shape
    P = max(0, (S - first_key) // kpool)
    keys = np.zeros((P, ihd), dtype=F64)
    pool_valid = np.zeros(P, dtype=np.uint8)
    pool_idx = first_key + np.arange(P)[:, None] * kpool + np.arange(kpool)[None, :]
    if P == 0:
        return keys, pool_valid, pool_idx.astype(np.int64)
    toks = pool_idx  # [P, kpool]
    kn = bf16_round(layernorm_bias(k_tok[toks], gamma, beta, eps))  # [P, kpool, ihd]
    logits = gate_tok[toks] + np.asarray(ape, dtype=F64)[None, :, :]  # [P, kpool, ihd]
    m = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - m)
    alpha = e / e.sum(axis=1, keepdims=True)  # softmax over the slot axis
    pooled = bf16_round((alpha * kn).sum(axis=1))
    ok = np.all(valid_tok[toks] != 0, axis=1)
    keys[ok] = pooled[ok]
    pool_valid[ok] = 1
    return keys, pool_valid, pool_idx.astype(np.int64)


# ---------------------------------------------------------------------------
# (a2) index_scores


def index_scores(qidx_row, w_row, keys, pool_valid, ctx_len: int, first_key: int,
                 kpool: int, scale: float, p_stride: Optional[int] = None) -> np.ndarray:
    """Scores of one query row over one sequence's pools (``dsa_index_scores``).

    tp.rs, "Why the indexer is replicated": the score of a pool is a sum over the
    indexer heads of each head's weight times the rectified, scaled dot product,
    one score per (query row, pool). build.rs, transform 2: ``w`` already carries
    the ``index_heads^-0.5`` factor, so the score does not apply it again.

    ``score[p] = sum_h w[h] * relu(scale * <qidx[h], keys[p]>)`` when pool p is a
    candidate: flagged valid, and visible to this row (its last slot
    ``first_key + (p+1)*kpool - 1`` is before ``ctx_len``). Every other entry of
    the ``p_stride``-wide row is ``-inf``.
    """
    q = np.asarray(qidx_row, dtype=F64)  # [Hi, ihd]
    w = np.asarray(w_row, dtype=F64)  # [Hi]
    keys = np.asarray(keys, dtype=F64)  # [P, ihd]
    P = keys.shape[0]
    if p_stride is None:
        p_stride = P
    out = np.full(p_stride, -np.inf, dtype=F64)
    n_vis = max(0, (ctx_len - first_key) // kpool)
    n = min(P, n_vis, p_stride)
    if n == 0:
        return out
    dots = keys[:n] @ q.T  # [n, Hi]
    s = (np.maximum(F64(scale) * dots, 0.0) * w[None, :]).sum(axis=1)
    cand = np.asarray(pool_valid[:n]) != 0
    out[:n] = np.where(cand, s, -np.inf)
    return out


# ---------------------------------------------------------------------------
# (a3) topk_pools, (a4) expand_selection


def select_k(index_topk: int, kpool: int, n_pools: int) -> int:
    """Pools selected per query, capped by how many pools exist
    (mod.rs, ``Glm5NextDsaConfig::select_k``)."""
    return min(index_topk // kpool, n_pools)


def topk_pools(scores_row, sk: int) -> np.ndarray:
    """``dsa_topk_pools`` for one row: ``[P]`` scores -> ``[sk]`` pool ids.

    mod.rs "Shape of the pipeline": ``topk_pools -> [Q, select_k] pool ids``.
    Reading taken where the pages are silent: the chosen pools are the first
    ``k' = min(sk, #finite)`` in the order (score descending, pool id ascending),
    with -0.0 equal to +0.0; non-candidates (-inf) are never chosen; the chosen
    ids are emitted in ascending order and the row is padded with -1.
    """
    s = np.asarray(scores_row, dtype=F64)
    if np.isnan(s).any():
        raise ValueError("topk_pools: NaN score")
    ids = np.arange(s.shape[0])
    fin = np.isfinite(s)
    kk = min(sk, int(fin.sum()))
    order = np.lexsort((ids[fin], -s[fin]))  # primary: -score; secondary: id
    chosen = np.sort(ids[fin][order[:kk]])
    out = np.full(sk, -1, dtype=np.int64)
    out[:kk] = chosen
    return out


def out_width(index_topk: int, kpool: int, always_select_tail: bool = False) -> int:
    """Width of the emitted index row (mod.rs, ``Glm5NextDsaConfig::out_width``)."""
    return index_topk + (kpool - 1 if always_select_tail else 0)


def expand_selection(pool_ids_row, first_key: int, kpool: int, width: int) -> np.ndarray:
    """``dsa_expand_selection`` for one row: pool ids -> token ids.

    mod.rs "Checkpoint and kernel facts": the expansion first fills the entire
    index row with -1 and only then stores token ids, so no slot keeps a stale
    value.
    Pool id ``p`` at position ``j`` becomes tokens ``first_key + p*kpool + s`` at
    positions ``j*kpool + s``.
    """
    row = np.full(width, -1, dtype=np.int64)
    for j, p in enumerate(np.asarray(pool_ids_row)):
        if p < 0:
            continue
        for s in range(kpool):
            row[j * kpool + s] = first_key + int(p) * kpool + s
    return row


def tail_tokens(ctx_len: int, first_key: int, kpool: int) -> np.ndarray:
    """Tokens of the trailing partial pool a query row sees: ``[first_key + P*kpool,
    ctx_len)`` with ``P = max(0, (ctx_len - first_key) // kpool)`` whole pools.

    mod.rs "Checkpoint and kernel facts": pooling starts at ``first_key`` and a
    trailing partial pool is not a pool, so these tokens are never a top-k
    candidate. There are at most ``kpool - 1`` of them; none when ``ctx_len`` is
    at most ``first_key`` or ends on a pool boundary.
    """
    if ctx_len <= first_key:
        return np.zeros(0, dtype=np.int64)
    P = (ctx_len - first_key) // kpool
    return np.arange(first_key + P * kpool, ctx_len, dtype=np.int64)


def expand_selection_tail(pool_ids_row, first_key: int, kpool: int, index_topk: int,
                          ctx_len: int, width: Optional[int] = None) -> np.ndarray:
    """``dsa_expand_selection`` with ``always_select_tail`` set, for one row.

    ``Glm5NextDsaConfig::out_width`` widens the row by ``index_kpool - 1`` slots
    when ``always_select_tail`` is set; the pages say no more. Reading taken: the
    selected pools expand as without the flag into positions ``[0, index_topk)``,
    and the extra slots, from position ``index_topk`` on, hold ``tail_tokens`` in
    ascending order, then -1. The tail is taken by position alone (token validity
    gates pool candidacy, and the tail is not a pool).
    """
    w = out_width(index_topk, kpool, True) if width is None else width
    row = expand_selection(pool_ids_row, first_key, kpool, w)
    tail = tail_tokens(ctx_len, first_key, kpool)
    row[index_topk: index_topk + tail.size] = tail
    return row


# ---------------------------------------------------------------------------
# (a5) NoPE MLA restricted to the selected tokens, in latent space


def sparse_mla_decode_row(qlat_row, ckv_seq, token_ids_row, softmax_scale: float,
                          o_absorb=None):
    """Attention of one query row over its selected tokens, then ``o_absorb``.

    mod.rs "Shape of the pipeline": NoPE MLA restricted to the expanded tokens
    (-1 = invalid). build.rs transforms 1 and 3: Q is absorbed through
    ``kv_b_proj``'s K half, so scores are taken against the latent row itself,
    and ``o_proj`` is absorbed through the V half, so the latent row is also the
    value and the output projection maps ``[heads, kv_lora_rank]`` back to
    hidden. NoPE: no rope section (mod.rs, ``is_nope``).

    ``logit[h, t] = softmax_scale * <qlat[h], ckv[t]>`` over ``t`` in the row's
    token ids ``>= 0``; ``olat[h] = sum_t softmax(logit[h])_t * ckv[t]``;
    ``y[i] = sum_{h,c} o_absorb[i, h*kvl + c] * olat[h, c]``. An empty selection
    gives ``olat = 0``.

    Returns ``(olat [H, kvl], y_exact [hidden] or None, y_bf16 or None)``.
    """
    q = np.asarray(qlat_row, dtype=F64)  # [H, kvl]
    ids = np.asarray(token_ids_row)
    ids = ids[ids >= 0]
    H, kvl = q.shape
    if ids.size == 0:
        olat = np.zeros((H, kvl), dtype=F64)
    else:
        kv = np.asarray(ckv_seq[ids], dtype=F64)  # [T, kvl]
        logits = F64(softmax_scale) * (q @ kv.T)  # [H, T]
        m = logits.max(axis=1, keepdims=True)
        p = np.exp(logits - m)
        p /= p.sum(axis=1, keepdims=True)
        olat = p @ kv
    if o_absorb is None:
        return olat, None, None
    y, yb = latent_project(olat, o_absorb)
    return olat, y, yb


def latent_project(olat, o_absorb):
    """The absorbed output projection (build.rs, transform 3 and ``absorb_o``):
    ``y[i] = sum_{h,c} o_absorb[i, h*kvl + c] * olat[h, c]``; y is stored bf16.
    Returns ``(y_exact, y_bf16)``."""
    A = np.asarray(o_absorb, dtype=F64)  # [hidden, H*kvl]
    y = A @ np.asarray(olat, dtype=F64).reshape(-1)
    return y, bf16_round(y)


# ---------------------------------------------------------------------------
# Load-time absorptions (build.rs) and the two unabsorbed/dense references the
# equivalence checks compare against.


def absorb_q(q_b, kv_b, heads: int, nope: int, vd: int, kvl: int, ql: int) -> np.ndarray:
    """Load-time Q absorption (build.rs module doc, transform 1; ``absorb_q``).

    Head h owns ``nope`` rows of ``q_b`` (Q_h, ``[nope, ql]``) and a block of
    ``nope + vd`` rows of ``kv_b`` whose first ``nope`` rows form its K half (K_h,
    ``[nope, kvl]``). The absorbed block of head h is K_h^T Q_h (``[kvl, ql]``), so
    that ``<q, K_h c> = <K_h^T q, c>`` for a latent row c; the blocks are stacked
    over heads. ``q_b [heads*nope, ql]`` (NoPE: ``qk_head_dim == nope``),
    ``kv_b [heads*(nope+vd), kvl]``. Returns ``[heads*kvl, ql]``.
    """
    q_b = np.asarray(q_b, dtype=F64).reshape(heads, nope, ql)
    kv_b = np.asarray(kv_b, dtype=F64).reshape(heads, nope + vd, kvl)
    out = np.zeros((heads, kvl, ql), dtype=F64)
    for h in range(heads):
        k_half = kv_b[h, :nope, :]  # [nope, kvl]: rows r < nope of head h's block
        out[h] = k_half.T @ q_b[h]  # [kvl, ql]: sum over r
    return out.reshape(heads * kvl, ql)


def absorb_o(o_proj, kv_b, heads: int, nope: int, vd: int, kvl: int, hidden: int) -> np.ndarray:
    """Load-time output absorption (build.rs module doc, transform 3; ``absorb_o``).

    The V half of head h's ``kv_b`` block (its last ``vd`` rows, V_h ``[vd, kvl]``)
    maps a latent vector to that head's value; ``o_proj``'s columns of head h (O_h,
    ``[hidden, vd]``) map the value to the hidden state. The absorbed columns of
    head h are O_h V_h (``[hidden, kvl]``), placed side by side over heads.
    ``o_proj [hidden, heads*vd]``. Returns ``[hidden, heads*kvl]``.
    """
    o = np.asarray(o_proj, dtype=F64).reshape(hidden, heads, vd)
    kv_b = np.asarray(kv_b, dtype=F64).reshape(heads, nope + vd, kvl)
    out = np.zeros((hidden, heads, kvl), dtype=F64)
    for h in range(heads):
        v_half = kv_b[h, nope:, :]  # [vd, kvl]
        out[:, h, :] = o[:, h, :] @ v_half
    return out.reshape(hidden, heads * kvl)


def mla_unabsorbed(q_lora, q_b, kv_b, o_proj, ckv_sel, heads: int, nope: int, vd: int,
                   kvl: int, softmax_scale: float) -> np.ndarray:
    """Standard (unabsorbed) NoPE MLA for one query over the given latent rows:
    decompress the latent through ``kv_b_proj`` into per-head keys and values,
    attend per head with ``qk_head_dim^-0.5`` scaling, project with ``o_proj``.
    The reference that ``absorb_q``/``absorb_o`` must reproduce (build.rs module
    doc: Q moves into the latent space; ``o_proj`` takes ``[heads, v_head_dim]``).
    """
    q_lora = np.asarray(q_lora, dtype=F64)
    ql = q_lora.shape[0]
    q = (np.asarray(q_b, dtype=F64) @ q_lora).reshape(heads, nope)
    kv_b = np.asarray(kv_b, dtype=F64).reshape(heads, nope + vd, kvl)
    c = np.asarray(ckv_sel, dtype=F64)  # [T, kvl]
    outs = []
    for h in range(heads):
        k = c @ kv_b[h, :nope, :].T  # [T, nope]
        v = c @ kv_b[h, nope:, :].T  # [T, vd]
        logit = F64(softmax_scale) * (k @ q[h])
        p = np.exp(logit - logit.max())
        p /= p.sum()
        outs.append(p @ v)
    return np.asarray(o_proj, dtype=F64) @ np.concatenate(outs)


def dense_masked_attention(qlat_row, ckv_seq, mask, softmax_scale: float) -> np.ndarray:
    """Dense latent attention over ALL tokens of the sequence, with masked tokens'
    logits set to -inf: the role of the pages' oracle kernels
    (``dsa_topk_to_mask`` -> ``dsa_mla_masked_attn``, mod.rs
    ``Glm5NextDsaKernels``)."""
    q = np.asarray(qlat_row, dtype=F64)
    kv = np.asarray(ckv_seq, dtype=F64)
    logits = F64(softmax_scale) * (q @ kv.T)  # [H, S]
    logits = np.where(np.asarray(mask, dtype=bool)[None, :], logits, -np.inf)
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    p /= p.sum(axis=1, keepdims=True)
    return p @ kv


# ---------------------------------------------------------------------------
# FP8 latent cache (mod.rs, ``MASKED_ATTN_MAX_KEYS`` doc: the serve's decode
# kernel is ``glm5next_dsa_mla_decode_fp8``). The pages name the kernel and
# nothing of its format; the format below is this layer's stated choice:
# OCP FP8 E4M3 codes (1 sign, 4 exponent bits with bias 7, 3 mantissa bits,
# largest finite 448, no infinities) with one power-of-two scale per token and
# 128-channel group.

E4M3_MAX = 448.0
FP8_GROUP = 128


def e4m3_round(v) -> np.ndarray:
    """Round float64 values to the nearest E4M3 value, ties to even; magnitudes
    above 448 saturate to 448 (no infinities in the format)."""
    v = np.asarray(v, dtype=F64)
    a = np.abs(v)
    _, E2 = np.frexp(np.where(a > 0, a, 1.0))  # a = f * 2^E2, f in [0.5, 1)
    # Spacing of E4M3 values at a's binade: 2^(e - 3) for normals (e >= -6),
    # 2^-9 throughout the subnormal range.
    e = np.maximum(E2 - 1, -6)
    q = np.ldexp(1.0, e - 3)
    r = np.round(a / q) * q  # numpy rounds halves to even; a / q is exact
    r = np.minimum(r, E4M3_MAX)
    return np.where(a > 0, np.copysign(r, v), v * 0.0)


def e4m3_encode(v) -> np.ndarray:
    """Byte codes of values that are already E4M3 values (``e4m3_round`` output)."""
    v = np.asarray(v, dtype=F64)
    a = np.abs(v)
    sign = np.where(np.signbit(v), 0x80, 0)
    _, E2 = np.frexp(np.where(a > 0, a, 1.0))
    e = E2 - 1
    normal = a >= 2.0 ** -6
    exp_field = np.where(normal, e + 7, 0)
    mant = np.where(normal, (a / np.ldexp(1.0, e) - 1.0) * 8, a / 2.0 ** -9)
    code = (exp_field << 3) | np.rint(mant).astype(np.int64)
    return (sign | np.where(a > 0, code, 0)).astype(np.uint8)


def e4m3_decode(codes) -> np.ndarray:
    """Values of E4M3 byte codes (0x7F and 0xFF, the NaNs, decode to NaN)."""
    c = np.asarray(codes, dtype=np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    ef = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(ef == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.ldexp(1.0, ef - 7))
    val = np.where((c & 0x7F) == 0x7F, np.nan, val)
    return s * val


def fp8_scale_exponent(amax) -> np.ndarray:
    """k of a group's scale 2^k: the smallest integer with amax <= 448 * 2^k, not
    below -126 (so 2^k and 2^-k are normal float32 numbers); 0 for an all-zero
    group."""
    a = np.asarray(amax, dtype=F64)
    f, E2 = np.frexp(np.where(a > 0, a, 1.0))  # a = (2f) * 2^(E2-1), 2f in [1, 2)
    # a <= 448 * 2^k  <=>  (2f) * 2^(E2-1-k) <= 1.75 * 2^8
    k = np.where(2 * f <= 1.75, E2 - 1 - 8, E2 - 1 - 7)
    k = np.maximum(k, -126)
    return np.where(a > 0, k, 0).astype(np.int64)


def quantize_latent_fp8(rows):
    """Latent rows ``[T, kvl]`` -> ``(codes uint8 [T, kvl], scales float64
    [T, kvl/128])``: per 128-channel group, scale ``2^k`` (``fp8_scale_exponent``
    of the group's largest magnitude) and codes ``E4M3(x / 2^k)``."""
    x = np.asarray(rows, dtype=F64)
    T, kvl = x.shape
    g = x.reshape(T, kvl // FP8_GROUP, FP8_GROUP)
    k = fp8_scale_exponent(np.abs(g).max(axis=2))  # [T, G]
    q = e4m3_round(np.ldexp(g, -k[:, :, None]))
    return e4m3_encode(q).reshape(T, kvl), np.ldexp(1.0, k)


def dequantize_latent_fp8(codes, scales) -> np.ndarray:
    """``x[t, c] = E4M3(codes[t, c]) * scales[t, c // 128]`` (float64)."""
    c = np.asarray(codes)
    T, kvl = c.shape
    v = e4m3_decode(c).reshape(T, kvl // FP8_GROUP, FP8_GROUP)
    return (v * np.asarray(scales, dtype=F64)[:, :, None]).reshape(T, kvl)


# ---------------------------------------------------------------------------
# Decode-time append and the geometry derived from the live length (mod.rs,
# ``Glm5NextDsaKernels`` fields ``indexer_store`` and ``write_geom``;
# ``Glm5NextDsaConfig::max_context``)


def max_dsa_context(max_context: int, kpool: int) -> int:
    """Tokens a sequence's indexer cache holds: ``max_context`` rounded down to
    whole pools (mod.rs, ``max_context`` field doc). Reading: a multiple of
    ``kpool``."""
    return (max_context // kpool) * kpool


def indexer_store(k_seq, gate_seq, valid_seq, seq_len: int, k_row, gate_row, capacity: int,
                  ckv_seq=None, ckv_row=None) -> int:
    """``indexer_store`` for one sequence: the staged indexer row goes to position
    ``seq_len`` of the sequence's caches, which is marked valid, and the length
    grows by one (mod.rs, Glm5NextDsaKernels: the position comes from the device,
    and the slot is flagged valid). The caches are the sequence's logical token-major
    arrays, updated in place. A full cache (``seq_len >= capacity``) is left
    unchanged. ``ckv_seq``/``ckv_row``: the layer's latent row for the same token,
    stored alongside (no counterpart on the pages; the latent cache append).
    Returns the new length."""
    if seq_len >= capacity:
        return seq_len
    k_seq[seq_len] = k_row
    gate_seq[seq_len] = gate_row
    valid_seq[seq_len] = 1
    if ckv_seq is not None:
        ckv_seq[seq_len] = ckv_row
    return seq_len + 1


def pools_completed(prev_len: int, new_len: int, first_key: int, kpool: int) -> range:
    """Pools that are whole at ``new_len`` tokens but were not at ``prev_len``:
    pool p is whole once ``first_key + (p+1)*kpool <= length`` (mod.rs, "Checkpoint
    and kernel facts": pooling starts at first_key; a trailing partial pool is not
    a pool)."""
    def whole(n):
        return max(0, (n - first_key) // kpool) if n > first_key else 0
    return range(whole(prev_len), whole(new_len))


def compress_append(k_tok, gate_tok, valid_tok, ape, gamma, beta, eps: float, first_key: int,
                    kpool: int, prev_len: int, new_len: int, keys_out, pool_valid_out):
    """Compress only the pools that the tokens ``[prev_len, new_len)`` completed,
    into the sequence's pooled cache (``keys_out [Pcap, ihd]``, ``pool_valid_out
    [Pcap]``, updated in place); other pools are not touched. Each such pool is
    ``kpool_compress`` of the first ``new_len`` tokens."""
    rng = pools_completed(prev_len, new_len, first_key, kpool)
    if len(rng) == 0:
        return rng
    keys, pv, _ = kpool_compress(np.asarray(k_tok)[:new_len], np.asarray(gate_tok)[:new_len],
                                 np.asarray(valid_tok)[:new_len], ape, gamma, beta, eps,
                                 first_key, kpool)
    keys_out[rng.start:rng.stop] = keys[rng.start:rng.stop]
    pool_valid_out[rng.start:rng.stop] = pv[rng.start:rng.stop]
    return rng


def write_geom(seq_lens, row_seq=None) -> np.ndarray:
    """``write_geom``: the selector's per-row geometry recomputed on the device
    from the current lengths (mod.rs, Glm5NextDsaKernels: this is what keeps one
    captured graph valid while the sequences grow).
    Reading: a decode row sees its whole sequence, so its context length is the
    sequence's current length; the visible pools and the tail follow from it."""
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    if row_seq is None:
        return seq_lens.copy()
    return seq_lens[np.asarray(row_seq, dtype=np.int64)]


# ---------------------------------------------------------------------------
# Projection front-end: the layer's inputs from the hidden state (build.rs, the
# tensor table of ``DsaTpPlan::new`` and ``build_dsa_weights``). The pages give the
# weights and their shapes; the order of the computation is the plain reading of
# those shapes: q_a_proj, q_a_layernorm, then q_absorb (-> qlat) and indexer.wq_b
# (-> qidx) on the normalised q_lora; kv_a_proj_with_mqa and kv_a_layernorm (-> the
# token's latent row); indexer.wk (-> raw indexer key), the compress gate (-> gate
# logits) and weights_proj (already scaled by index_heads^-0.5 at load, -> w) on
# the hidden state. The two a-norms carry a weight and no bias (the pages single out
# k_norm as the one norm with a bias): RMSNorm.


def rms_norm(x, gamma, eps: float) -> np.ndarray:
    """``x / sqrt(mean(x^2) + eps) * gamma`` over the last axis (float64)."""
    x = np.asarray(x, dtype=F64)
    ms = (x * x).mean(axis=-1, keepdims=True)
    return x / np.sqrt(ms + F64(eps)) * np.asarray(gamma, dtype=F64)


def frontend_row(x_row, q_a_proj, q_a_norm, kv_a_proj, kv_a_norm, wk, compress_gate,
                 weights_proj, q_absorb, wq_b, eps: float, heads: int, index_heads: int) -> dict:
    """One decode row's front-end. Storage points (bf16 unless noted): q_lora (the
    normalised q_a), qlat ``[heads, kvl]``, qidx ``[index_heads, ihd]``, the latent
    row ``ckv``, ``k_raw``, ``gate``; ``w`` stays float (f32 on the device)."""
    x = np.asarray(x_row, dtype=F64)
    mm = lambda W, v: np.asarray(W, dtype=F64) @ v
    q_lora = bf16_round(rms_norm(mm(q_a_proj, x), q_a_norm, eps))
    ckv = bf16_round(rms_norm(mm(kv_a_proj, x), kv_a_norm, eps))
    qlat = bf16_round(mm(q_absorb, q_lora))
    qidx = bf16_round(mm(wq_b, q_lora))
    return dict(q_lora=q_lora, ckv=ckv, qlat=qlat.reshape(heads, -1),
                qidx=qidx.reshape(index_heads, -1), k_raw=bf16_round(mm(wk, x)),
                gate=bf16_round(mm(compress_gate, x)), w=mm(weights_proj, x))


# ---------------------------------------------------------------------------
# Cache addressing (the oracle's own, independent of the kernels')


def sequence_tokens(cache, b: int, n_tokens: int, block_table=None, block_size: int = 0):
    """Logical ``[n_tokens, ...]`` view of sequence ``b`` of a token cache:
    contiguous ``[B, Smax, ...]`` or paged ``[NB, block_size, ...]`` through
    ``block_table [B, max_blocks]``."""
    cache = np.asarray(cache)
    if block_table is None:
        return cache[b, :n_tokens]
    t = np.arange(n_tokens)
    blk = np.asarray(block_table)[b, t // block_size]
    return cache[blk, t % block_size]


def sequence_pools(pcache, b: int, n_pools: int, block_table=None, pools_per_block: int = 0):
    """Logical ``[n_pools, ...]`` view of sequence ``b`` of a pooled-key cache:
    contiguous ``[B, Pcap, ...]`` or paged ``[NB, pools_per_block, ...]`` through
    the same block table."""
    pcache = np.asarray(pcache)
    if block_table is None:
        return pcache[b, :n_pools]
    p = np.arange(n_pools)
    blk = np.asarray(block_table)[b, p // pools_per_block]
    return pcache[blk, p % pools_per_block]


# ---------------------------------------------------------------------------
# One query row end to end (a2..a5) on a pooled cache


def decode_row(qidx_row, w_row, keys, pool_valid, ctx_len: int, first_key: int, kpool: int,
               index_scale: float, index_topk: int, p_stride: int, qlat_row, ckv_seq,
               softmax_scale: float, o_absorb=None, always_select_tail: bool = False):
    """score -> top-k -> expand -> sparse latent MLA (-> o_absorb) for one row."""
    s = index_scores(qidx_row, w_row, keys, pool_valid, ctx_len, first_key, kpool,
                     index_scale, p_stride)
    sk = select_k(index_topk, kpool, p_stride)
    ids = topk_pools(s, sk)
    if always_select_tail:
        tok = expand_selection_tail(ids, first_key, kpool, index_topk, ctx_len)
    else:
        tok = expand_selection(ids, first_key, kpool, out_width(index_topk, kpool))
    olat, y, yb = sparse_mla_decode_row(qlat_row, ckv_seq, tok, softmax_scale, o_absorb)
    return dict(scores=s, pool_ids=ids, token_ids=tok, olat=olat, y=y, y_bf16=yb)
