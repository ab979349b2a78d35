"""Test helpers: run the oracle on a workload's sequences/rows and compare with the
GPU path under the acceptance rules (kpool within bf16 ulps, scores within 1e-3
relative, selections bit-exact outside near-ties, attention within 2e-2)."""
from __future__ import annotations

import numpy as np
import torch

from oracle import dsa_oracle as O

SCORE_RTOL = 1e-3
SCORE_ATOL = 1e-5
ATTN_TOL = 2e-2
TIE_BAND = 1e-3


def f(t: torch.Tensor) -> np.ndarray:
    """Host float64 copy of a CPU tensor (bf16 exact)."""
    return t.float().numpy().astype(np.float64)


class OracleSeq:
    """Oracle views of one workload (tokens and pools per sequence), cached."""

    def __init__(self, wl, use_drawn_kpool: bool = False):
        self.wl = wl
        self.drawn = use_drawn_kpool
        self._pools = {}
        self._ckv = {}

    def tokens(self, name: str, b: int) -> np.ndarray:
        """Sequence b's rows of a token cache, gathered on the raw bits (oracle
        addressing) and only then widened to float."""
        wl = self.wl
        t = getattr(wl, name)
        bf = t.dtype == torch.bfloat16
        raw = t.view(torch.int16).numpy() if bf else t.numpy()
        rows = O.sequence_tokens(raw, b, int(wl.seq_lens[b]),
                                 None if wl.block_table is None else wl.block_table.numpy(),
                                 wl.block_size or 0)
        if bf:
            return torch.from_numpy(np.ascontiguousarray(rows)).view(torch.bfloat16).float().numpy()
        return rows

    def ckv(self, b: int) -> np.ndarray:
        if b not in self._ckv:
            self._ckv[b] = self.tokens("ckv", b).astype(np.float64)
        return self._ckv[b]

    def pools(self, b: int):
        """(keys [P, ihd], pool_valid [P]) of sequence b."""
        if b in self._pools:
            return self._pools[b]
        wl, g = self.wl, self.wl.geom
        L = int(wl.seq_lens[b])
        P = max(0, (L - g.first_key) // g.index_kpool)
        if self.drawn:
            bt = None if wl.block_table is None else wl.block_table.numpy()
            ppb = (wl.block_size or 0) // g.index_kpool
            keys = O.sequence_pools(wl.kpool_keys.float().numpy(), b, P, bt, ppb).astype(np.float64)
            pv = O.sequence_pools(wl.kpool_valid.numpy(), b, P, bt, ppb)
            out = (keys, pv, None)
        else:
            out = O.kpool_compress(self.tokens("k_raw", b), self.tokens("gate", b),
                                   self.tokens("valid", b), wl.ape.numpy(), f(wl.ln_w),
                                   f(wl.ln_b), g.eps, g.first_key, g.index_kpool)
        self._pools[b] = out
        return out

    def kn_ulp(self, b: int) -> np.ndarray:
        """[P, ihd]: the largest bf16 ulp among a pool's normalised slot keys. The
        layer stores kn = bf16(LN(k)) before pooling; where the exact LN value sits
        next to a rounding midpoint, f32 and f64 arithmetic may round kn to opposite
        neighbours, which moves the pooled key by softmax weight x ulp(kn)."""
        wl, g = self.wl, self.wl.geom
        k = self.tokens("k_raw", b)
        L = k.shape[0]
        P = max(0, (L - g.first_key) // g.index_kpool)
        toks = g.first_key + np.arange(P)[:, None] * g.index_kpool + np.arange(g.index_kpool)
        kn = O.bf16_round(O.layernorm_bias(k[toks], f(wl.ln_w), f(wl.ln_b), g.eps))
        return bf16_ulp(kn).max(axis=1)

    def scores(self, r: int, p_stride: int) -> np.ndarray:
        wl, g = self.wl, self.wl.geom
        b = int(wl.row_seq[r])
        keys, pv, _ = self.pools(b)
        return O.index_scores(f(wl.qidx[r]), wl.w[r].numpy().astype(np.float64), keys, pv,
                              int(wl.row_ctx[r]), g.first_key, g.index_kpool, g.index_scale,
                              p_stride)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(ax)) - 7)


def check_kpool(gpu: np.ndarray, ref: np.ndarray, kn_ulp: np.ndarray, what: str = "kpool") -> float:
    """bf16 pooled keys. Every element within 2 ulp(ref) + kn_ulp (one slot key
    rounded the other way, see OracleSeq.kn_ulp); at most 0.1 % of elements not
    identical and at most 0.01 % beyond 2 ulp(ref). Returns the mismatch fraction."""
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    if gpu.size == 0:
        return 0.0
    diff = np.abs(gpu - ref)
    two = 2 * bf16_ulp(ref)
    bad = diff > two + kn_ulp
    assert not bad.any(), f"{what}: {bad.sum()} elements beyond bound, e.g. {gpu[bad][:4]} vs {ref[bad][:4]}"
    frac = float((diff != 0).mean())
    assert frac <= 1e-3, f"{what}: {frac:.2e} of elements differ"
    beyond = float((diff > two).mean())
    assert beyond <= 1e-4, f"{what}: {beyond:.2e} of elements beyond 2 ulp"
    return frac


def check_scores(gpu: np.ndarray, ref: np.ndarray, what: str = "scores", extra=None) -> None:
    """|gpu - ref| <= 1e-3 |ref| + 1e-5 on finite entries; identical -inf pattern.
    ``extra`` (per entry) widens the bound by the effect of a known difference in
    the stage's inputs (end-to-end runs, see score_input_bound)."""
    gi, ri = np.isinf(gpu), np.isinf(ref)
    np.testing.assert_array_equal(gi, ri, err_msg=f"{what}: -inf pattern differs")
    if ri.any():
        assert (gpu[gi] < 0).all()
    fin = ~ri
    err = np.abs(gpu[fin] - ref[fin])
    lim = SCORE_RTOL * np.abs(ref[fin]) + SCORE_ATOL
    if extra is not None:
        lim = lim + extra[fin]
    assert (err <= lim).all(), f"{what}: max excess {(err - lim).max():.3e}"


def score_input_bound(qidx_row, w_row, dkeys, scale, p_stride) -> np.ndarray:
    """Largest change of each pool's score when its pooled key moves by dkeys:
    relu is 1-Lipschitz, so |ds_p| <= sum_h |w_h| * scale * |<q_h, dk_p>|."""
    out = np.zeros(p_stride)
    n = min(p_stride, dkeys.shape[0])
    if n:
        out[:n] = (np.abs(dkeys[:n] @ np.asarray(qidx_row, np.float64).T) * abs(scale)
                   * np.abs(np.asarray(w_row, np.float64))[None, :]).sum(axis=1)
    return out


def exact_topk(row: np.ndarray, sk: int) -> np.ndarray:
    return O.topk_pools(row, sk)


def check_selection(gpu_ids: np.ndarray, ref_scores: np.ndarray, sk: int) -> str:
    """The end-to-end selection rule: bit-exact where the oracle's cutoff gap exceeds
    1e-3*|score|; otherwise the GPU set may differ only inside that band. Returns
    'gap' or 'band'."""
    s = ref_scores
    ids = np.arange(s.size)
    fin = np.isfinite(s)
    nfin = int(fin.sum())
    kk = min(sk, nfin)
    ref = O.topk_pools(s, sk)
    np.testing.assert_array_equal(gpu_ids[kk:], -1)
    got = gpu_ids[:kk]
    assert (np.diff(got) > 0).all(), "selection not ascending"
    if kk == 0:
        return "gap"
    order = np.lexsort((ids[fin], -s[fin]))
    sf = s[fin][order]
    c = sf[kk - 1]
    c2 = sf[kk] if kk < nfin else -np.inf
    band = TIE_BAND * abs(c)
    if c - c2 > band:
        np.testing.assert_array_equal(got, ref[:kk])
        return "gap"
    gs = set(got.tolist())
    above = set(ids[fin & (s > c + band)].tolist())
    below = set(ids[fin & (s < c - band)].tolist())
    assert above <= gs, "a pool above the tie band was not selected"
    assert not (gs & below), "a pool below the tie band was selected"
    assert len(gs) == kk
    return "band"


def check_attention(gpu: np.ndarray, ref: np.ndarray, what: str = "y") -> float:
    """Per row: max|gpu - ref| / max|ref| <= 2e-2 (rows where ref is all zero must be 0)."""
    worst = 0.0
    for i in range(ref.shape[0]):
        m = np.abs(ref[i]).max()
        e = np.abs(gpu[i] - ref[i]).max()
        if m == 0:
            assert e == 0, f"{what} row {i}: expected zeros"
            continue
        worst = max(worst, e / m)
        assert e / m <= ATTN_TOL, f"{what} row {i}: rel err {e / m:.3e}"
    return worst


class Guarded:
    """A device tensor with sentinel-filled guard bands before and after it."""

    def __init__(self, shape, dtype, fill, device="cuda", pad_bytes=4096):
        n = int(np.prod(shape))
        esz = torch.empty((), dtype=dtype).element_size()
        self.pad = max(1, pad_bytes // esz)
        # keep the view 16-byte aligned
        align = max(1, 16 // esz)
        self.pad = (self.pad + align - 1) // align * align
        self.full = torch.full((n + 2 * self.pad,), fill, dtype=dtype, device=device)
        self.fill = fill
        self.t = self.full[self.pad: self.pad + n].view(shape)

    def check(self):
        lo = self.full[: self.pad]
        hi = self.full[-self.pad:]
        ok = bool((lo == self.fill).all()) and bool((hi == self.fill).all())
        assert ok, "guard band overwritten"
