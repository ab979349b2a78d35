"""dsa_score_prefill (tensor-core index scores of a chunk of query rows of one
sequence) against the oracle's index_scores, element by element, through the C ABI.

Cases span several 128-pool tiles with a ragged tail, several 256-column query
tiles with a ragged last tile, more work units than CTAs (each CTA reloads its query
tile), a sequence other than the first in the cache, p_stride past the sequence's
pools, causal per-row context, a negative scale, and every supported head count and
head dimension."""
import zlib

import numpy as np
import pytest
import torch

from sparse_attention_decode_kpool_gb300 import api, workloads as W
from sparse_attention_decode_kpool_gb300.pipeline import DsaDecodeLayer
from tests import _harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    torch.cuda.init()


def _geom(**kw):
    base = dict(index_kpool=4, index_heads=32, index_head_dim=128, index_topk=256, heads=8,
                hidden=256)
    base.update(kw)
    return W.Geometry(**base)


def _ctx(rng, n, L, extra=()):
    """n causal context lengths in [1, L], with the given values first."""
    v = list(extra) + [int(x) for x in rng.integers(1, L + 1, size=max(0, n - len(extra)))]
    return v[:n]


PREFILL_CASES = [
    # (name, geometry kwargs, seq_lens, prefill_seq, rows, p_stride extra, scale sign, check rows)
    ("h32-d128-ragged", dict(), [3000], 0, 37, 0, 1, None),
    ("h64-d64", dict(index_heads=64, index_head_dim=64), [2100], 0, 21, 0, 1, None),
    ("h128-d128", dict(index_heads=128), [1500], 0, 5, 0, 1, None),
    ("h32-d64-kp8-fk3", dict(index_head_dim=64, index_kpool=8, index_topk=64, first_key=3),
     [2600], 0, 19, 0, 1, None),
    ("h32-seq1-of-3", dict(), [700, 3000, 900], 1, 24, 0, 1, None),
    ("h32-pstride-past-P", dict(), [1000], 0, 9, 300, 1, None),
    ("h32-neg-scale", dict(), [1200], 0, 11, 0, -1, None),
    ("h32-one-row-tiny", dict(), [10], 0, 1, 0, 1, None),
    # 88 query tiles x 2 pool chunks = 176 units: more units than CTAs.
    ("h32-multi-unit", dict(), [20000], 0, 700, 0, 1, 48),
]


@pytest.mark.parametrize("case", PREFILL_CASES, ids=[c[0] for c in PREFILL_CASES])
def test_score_prefill_parity(case):
    name, gkw, lens, pseq, rows, extra, sign, ncheck = case
    g = _geom(**gkw)
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    L = lens[pseq]
    ctx = _ctx(rng, rows, L, extra=[L, 1, g.first_key + g.index_kpool, L - 1])
    wl = W.make_workload(name, 300, g, lens, rows_ctx=ctx, prefill_seq=pseq, with_raw=False,
                         with_o_absorb=False, direct_kpool=True)
    layer = DsaDecodeLayer(wl, with_o_absorb=False, use_drawn_kpool=True)
    p_stride = wl.p_stride + extra
    scale = sign * g.index_scale
    sc = H.Guarded((rows, p_stride), torch.float32, 12345.0)
    api.dsa_score_prefill(layer.qidx, layer.w, pseq, layer.row_ctx, layer.kpool,
                          layer.pool_valid, layer.pg, g.first_key, g.index_kpool, scale, sc.t,
                          status=layer.status)
    torch.cuda.synchronize()
    sc.check()
    assert int(layer.status.item()) == 0
    got = sc.t.cpu().numpy().astype(np.float64)
    oq = H.OracleSeq(wl, use_drawn_kpool=True)
    check = range(rows)
    if ncheck is not None:  # first, last, the ragged tile and a seeded sample
        pick = {0, 1, rows - 1, rows - 2, 8 * ((rows - 1) // 8)}
        pick |= set(int(x) for x in rng.choice(rows, size=ncheck, replace=False))
        check = sorted(pick)
    for r in check:
        ref = oq.scores(r, p_stride) if sign > 0 else _neg_scores(oq, wl, r, p_stride)
        H.check_scores(got[r], ref, f"{name} row {r}")
    # Every entry was written (no sentinel left) and -inf past the sequence's pools.
    assert not (got == 12345.0).any()
    P = max(0, (L - g.first_key) // g.index_kpool)
    assert np.isneginf(got[:, P:]).all()


def _neg_scores(oq, wl, r, p_stride):
    from oracle import dsa_oracle as O
    g = wl.geom
    keys, pv, _ = oq.pools(int(wl.row_seq[r]))
    return O.index_scores(H.f(wl.qidx[r]), wl.w[r].numpy().astype(np.float64), keys, pv,
                          int(wl.row_ctx[r]), g.first_key, g.index_kpool, -g.index_scale,
                          p_stride)


def test_score_prefill_matches_decode_kernel():
    """Both scorers of the library on the same rows: identical -inf pattern and
    values within the f32 reordering of the same sums."""
    g = _geom()
    rng = np.random.default_rng(7)
    ctx = _ctx(rng, 70, 5000, extra=[5000])
    wl = W.make_workload("pf-vs-decode", 301, g, [5000], rows_ctx=ctx, with_raw=False,
                         with_o_absorb=False, direct_kpool=True)
    a = DsaDecodeLayer(wl, with_o_absorb=False, use_drawn_kpool=True, score_path="prefill")
    b = DsaDecodeLayer(wl, with_o_absorb=False, use_drawn_kpool=True, score_path="decode")
    assert a.score_gemm and not b.score_gemm
    a.score()
    b.score()
    torch.cuda.synchronize()
    x, y = a.scores.cpu().numpy(), b.scores.cpu().numpy()
    np.testing.assert_array_equal(np.isinf(x), np.isinf(y))
    fin = np.isfinite(y)
    assert np.all(np.abs(x[fin] - y[fin]) <= 1e-5 * np.abs(y[fin]) + 1e-6)
