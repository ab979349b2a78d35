"""Stage-by-stage parity of the CUDA path against the CPU oracle, through the C ABI.

Each stage is fed the oracle's (or the generator's) previous-stage output, so one
stage's rounding never reaches the next stage's check."""
import numpy as np
import pytest
import torch

from oracle import dsa_oracle as O
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


# ---------------------------------------------------------------------------
# dsa_compress


COMPRESS_CASES = [
    # (name, geometry kwargs, seq_lens, block_size, first_key, invalid_per_seq)
    ("tiny", None, None, None, 0, 0),
    ("ihd128-kp4-ragged", dict(), [1000, 37, 513], None, 0, 9),
    ("ihd128-kp1", dict(index_kpool=1, index_topk=64), [301, 64], None, 0, 3),
    ("ihd64-kp2-fk5", dict(index_head_dim=64, index_kpool=2, index_topk=64), [333, 90], None, 5, 4),
    ("ihd128-kp3", dict(index_kpool=3, index_topk=48), [400, 11], None, 1, 5),
    ("ihd128-kp8", dict(index_kpool=8, index_topk=64), [777, 64], None, 0, 6),
    ("ihd64-kp16", dict(index_head_dim=64, index_kpool=16, index_topk=64), [999, 15], None, 0, 6),
    ("paged-kp4", dict(), [1000, 300, 64, 5], 64, 0, 7),
    ("paged-kp4-fk8", dict(), [900, 130], 64, 8, 2),
]


@pytest.mark.parametrize("case", COMPRESS_CASES, ids=[c[0] for c in COMPRESS_CASES])
def test_compress_parity(case):
    name, gkw, lens, bs, fk, inval = case
    if gkw is None:
        wl = W.tiny()
    else:
        g = _geom(first_key=fk, **gkw)
        wl = W.make_workload(name, 100, g, lens, block_size=bs, invalid_per_seq=inval,
                             with_o_absorb=False)
    layer = DsaDecodeLayer(wl, with_o_absorb=False)
    g = wl.geom
    KP, ihd = g.index_kpool, g.index_head_dim
    layer.kpool.fill_(7.0)  # sentinel: rows not written must keep it
    layer.pool_valid.fill_(9)
    pidx = torch.full(layer.pool_valid.shape + (KP,), -7, dtype=torch.int32, device="cuda")
    api.dsa_compress(layer.k_raw, layer.gate, layer.valid, layer.ape, layer.ln_w, layer.ln_b,
                     g.eps, layer.pg, g.first_key, KP, layer.kpool, layer.pool_valid, pidx,
                     layer.status)
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    oq = H.OracleSeq(wl)
    kp = layer.kpool.float().cpu().numpy()
    pv = layer.pool_valid.cpu().numpy()
    pi = pidx.cpu().numpy()
    bt = None if wl.block_table is None else wl.block_table.numpy()
    ppb = (wl.block_size or 0) // KP
    touched = np.zeros(pv.shape, dtype=bool)
    for b in range(wl.batch):
        keys, rpv, ridx = oq.pools(b)
        P = keys.shape[0]
        gk = O.sequence_pools(kp, b, P, bt, ppb)
        gv = O.sequence_pools(pv, b, P, bt, ppb)
        gi = O.sequence_pools(pi, b, P, bt, ppb)
        np.testing.assert_array_equal(gv, rpv)
        np.testing.assert_array_equal(gi, ridx)
        H.check_kpool(gk, keys, oq.kn_ulp(b), f"{name} seq {b}")
        if bt is None:
            touched[b, :P] = True
        else:
            p = np.arange(P)
            touched[bt[b, p // ppb], p % ppb] = True
    assert (pv[~touched] == 9).all() and (kp[~touched] == 7.0).all(), "rows past P written"


# ---------------------------------------------------------------------------
# dsa_score (fed the drawn pooled-key cache)


SCORE_CASES = [
    ("h32-d128", dict(), [3000, 517, 64], None, None, 0),
    ("h4-d64", dict(index_heads=4, index_head_dim=64), [2048], None, None, 0),
    ("h20-d128", dict(index_heads=20), [1234, 99], None, None, 0),
    ("h32-paged", dict(), [4000, 1000, 65], 64, None, 0),
    # paged rows of very unequal length (the CTAs split the visible stages only; the
    # rest of each row is filled with -inf): an empty and a 3-token sequence among them
    ("h32-paged-ragged", dict(), [9000, 64, 3, 20000, 0, 777, 4096, 12345], 64, None, 0),
    ("h32-paged-ctx", dict(), [6000], 64, [1, 3, 4, 5, 5999, 6000, 2000, 17], 0),
    ("h8-paged-b16", dict(index_heads=8), [700, 5000, 1, 2048], 16, None, 0),
    ("h32-prefill-ctx", dict(), [2000], None, [1, 3, 4, 5, 1999, 2000, 1500, 17], 0),
    ("h32-fk3", dict(first_key=3), [701, 40], None, None, 0),
    ("h8-kp8", dict(index_heads=8, index_kpool=8, index_topk=64), [1601, 3], None, None, 0),
]


@pytest.mark.parametrize("case", SCORE_CASES, ids=[c[0] for c in SCORE_CASES])
def test_score_parity(case):
    name, gkw, lens, bs, rows_ctx, _ = case
    g = _geom(**gkw)
    wl = W.make_workload(name, 200, g, lens, block_size=bs, rows_ctx=rows_ctx,
                         with_raw=False, with_o_absorb=False, direct_kpool=True)
    layer = DsaDecodeLayer(wl, with_o_absorb=False, use_drawn_kpool=True)
    sc = H.Guarded(layer.scores.shape, torch.float32, 12345.0)
    api.dsa_score(layer.qidx, layer.w, layer.row_seq, layer.row_ctx, layer.kpool,
                  layer.pool_valid, layer.pg, g.first_key, g.index_kpool, g.index_scale, sc.t,
                  status=layer.status)
    torch.cuda.synchronize()
    sc.check()
    assert int(layer.status.item()) == 0
    got = sc.t.cpu().numpy().astype(np.float64)
    oq = H.OracleSeq(wl, use_drawn_kpool=True)
    for r in range(wl.rows):
        H.check_scores(got[r], oq.scores(r, wl.p_stride), f"{name} row {r}")


# ---------------------------------------------------------------------------
# dsa_select (fed oracle-side f32 score rows) and dsa_expand


def _tie_rows(rng, rows, P, kind):
    if kind == "ties":
        vals = np.array([-np.inf, -1.0, -0.0, 0.0, 0.5, 1.0, 2.0], dtype=np.float32)
        return vals[rng.integers(0, len(vals), (rows, P))]
    if kind == "normal":
        x = rng.standard_normal((rows, P)).astype(np.float32)
        x[rng.random((rows, P)) < 0.05] = -np.inf
        return x
    if kind == "sparse":
        x = np.full((rows, P), -np.inf, dtype=np.float32)
        m = rng.random((rows, P)) < 0.01
        x[m] = rng.random(m.sum()).astype(np.float32)
        return x
    if kind == "allinf":
        return np.full((rows, P), -np.inf, dtype=np.float32)
    if kind == "positive":
        return (rng.random((rows, P)) * 3).astype(np.float32)
    if kind == "ramp":
        # scores rise with the pool id (fall on odd rows): a row's top-k sits in the
        # last (first) slice of a clustered row, whose trimmed candidates cannot hold it
        x = np.tile(np.arange(P, dtype=np.float32) / max(P, 1), (rows, 1))
        x[1::2] = x[1::2, ::-1]
        return np.ascontiguousarray(x)
    if kind == "crowd":
        # noise with one raised window of P/16 pools per row, some of it tied
        x = rng.standard_normal((rows, P)).astype(np.float32)
        for r in range(rows):
            w = max(1, P // 16)
            a = int(rng.integers(0, max(1, P - w)))
            x[r, a:a + w] += 4.0
            x[r, a:a + w:3] = 5.0
        return x
    raise ValueError(kind)


SELECT_CASES = [
    (1, 1, 4, 4, "normal"), (3, 5, 8, 4, "ties"), (2, 512, 256, 4, "ties"), (4, 511, 256, 4, "normal"),
    (1, 8192, 2048, 4, "positive"), (8, 65536, 2048, 4, "positive"), (2, 65536, 2048, 4, "ties"),
    (3, 100003, 2048, 4, "normal"), (2, 3000, 2048, 4, "sparse"), (2, 700, 256, 4, "allinf"),
    (5, 16384, 2048, 4, "positive"), (64, 16384, 2048, 4, "normal"), (300, 2048, 512, 4, "ties"),
    (1, 327680, 2048, 4, "positive"), (2, 40000, 64, 1, "ties"),
    # select_k not a multiple of 4 on clustered rows (padded merge slots)
    (3, 60000, 2044, 4, "ties"), (2, 50000, 1026, 1, "normal"),
    # top keys crowded into one slice (the merge's second exchange, with full slice lists)
    (8, 65536, 2048, 4, "ramp"), (4, 65536, 2048, 4, "crowd"), (3, 100003, 2044, 4, "crowd"),
    (2, 16384, 2048, 4, "ramp"),
]


@pytest.fixture(params=["merge", "radix"])
def select_form(request):
    """Both ways clustered rows are selected, each forced through
    DSA_OPT_SELECT_KERNEL (single-CTA rows take the same kernel either way)."""
    with api.select_kernel(request.param):
        yield request.param


@pytest.mark.parametrize("case", SELECT_CASES, ids=[f"{c[0]}x{c[1]}-k{c[2]}/{c[3]}-{c[4]}" for c in SELECT_CASES])
def test_select_parity(case, select_form):
    rows, P, topk, kp, kind = case
    rng = np.random.default_rng(rows * 7919 + P)
    s = _tie_rows(rng, rows, P, kind)
    sk = O.select_k(topk, kp, P)
    scores = torch.from_numpy(s).cuda()
    out = H.Guarded((rows, sk), torch.int32, -77)
    api.dsa_select(scores, topk, kp, out.t)
    torch.cuda.synchronize()
    out.check()
    got = out.t.cpu().numpy()
    for r in range(rows):
        np.testing.assert_array_equal(got[r], O.topk_pools(s[r].astype(np.float64), sk),
                                      err_msg=f"row {r}")


SELECT_EXPAND_CASES = [
    # rows, P, topk, kpool, kind, first_key, out_width extra
    (1, 1, 4, 4, "normal", 0, 0), (3, 5, 8, 4, "ties", 3, 5), (4, 511, 256, 4, "normal", 0, 0),
    (8, 65536, 2048, 4, "positive", 0, 0), (2, 3000, 2048, 4, "sparse", 1, 17),
    (2, 700, 256, 4, "allinf", 0, 0), (64, 16384, 2048, 4, "normal", 0, 0),
    (300, 2048, 512, 4, "ties", 0, 0), (2, 40000, 64, 1, "ties", 2, 3),
    (3, 2000, 128, 16, "normal", 16, 0), (2, 0, 256, 4, "allinf", 0, 9),
    (2, 70001, 2042, 2, "positive", 1, 3),
    (8, 65536, 2048, 4, "ramp", 0, 0), (4, 65536, 2048, 4, "crowd", 2, 5),
]


@pytest.mark.parametrize("case", SELECT_EXPAND_CASES,
                         ids=[f"{c[0]}x{c[1]}-k{c[2]}/{c[3]}-{c[4]}-fk{c[5]}" for c in SELECT_EXPAND_CASES])
def test_select_expand_parity(case, select_form):
    """The fused call equals dsa_select then dsa_expand bit for bit, and the oracle's
    top-k and expansion."""
    rows, P, topk, kp, kind, fk, extra = case
    rng = np.random.default_rng(rows * 31 + P + kp)
    s = _tie_rows(rng, rows, P, kind) if P else np.zeros((rows, 0), np.float32)
    sk = O.select_k(topk, kp, P)
    width = sk * kp + extra
    scores = torch.from_numpy(s).cuda()
    ids = H.Guarded((rows, sk), torch.int32, -77)
    tok = H.Guarded((rows, width), torch.int32, -88)
    api.dsa_select_expand(scores, topk, kp, fk, ids.t, tok.t)
    torch.cuda.synchronize()
    ids.check()
    tok.check()
    got_ids, got_tok = ids.t.cpu().numpy(), tok.t.cpu().numpy()
    if sk:
        ref_ids = torch.empty((rows, sk), dtype=torch.int32, device="cuda")
        api.dsa_select(scores, topk, kp, ref_ids)
        ref_tok = torch.empty((rows, width), dtype=torch.int32, device="cuda")
        api.dsa_expand(ref_ids, fk, kp, ref_tok)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(got_ids, ref_ids.cpu().numpy())
        np.testing.assert_array_equal(got_tok, ref_tok.cpu().numpy())
    for r in range(rows):
        o_ids = O.topk_pools(s[r].astype(np.float64), sk)
        np.testing.assert_array_equal(got_ids[r], o_ids, err_msg=f"row {r}")
        np.testing.assert_array_equal(got_tok[r], O.expand_selection(o_ids, fk, kp, width),
                                      err_msg=f"row {r}")


def test_expand_parity():
    rng = np.random.default_rng(3)
    for kp, fk, sk, width, rows in [(4, 0, 64, 256, 5), (4, 3, 512, 2048, 3), (1, 0, 7, 9, 2),
                                    (16, 16, 4, 70, 4), (3, 1, 10, 31, 6)]:
        ids = np.full((rows, sk), -1, dtype=np.int32)
        for r in range(rows):
            k = int(rng.integers(0, sk + 1))
            ids[r, :k] = np.sort(rng.choice(10 * sk + 10, k, replace=False))
        out = H.Guarded((rows, width), torch.int32, -99)
        api.dsa_expand(torch.from_numpy(ids).cuda(), fk, kp, out.t)
        torch.cuda.synchronize()
        out.check()
        got = out.t.cpu().numpy()
        for r in range(rows):
            np.testing.assert_array_equal(got[r], O.expand_selection(ids[r], fk, kp, width))


def _tail_ctx(rng, rows, P, kp, fk):
    """Context lengths for the tail tests: every remainder mod kpool, rows at and
    below first_key, and lengths past the last pool the scores cover."""
    base = fk + P * kp
    choices = [base + (r % kp) for r in range(rows)]
    for r in range(rows):
        pick = r % 5
        if pick == 1:
            choices[r] = int(rng.integers(0, fk + 1))
        elif pick == 3:
            choices[r] = int(rng.integers(fk, fk + 3 * kp + 5))
        elif pick == 4:
            choices[r] = base + int(rng.integers(0, 4 * kp))
    return np.asarray(choices, dtype=np.int32)


@pytest.mark.parametrize("case", SELECT_EXPAND_CASES,
                         ids=[f"{c[0]}x{c[1]}-k{c[2]}/{c[3]}-{c[4]}-fk{c[5]}" for c in SELECT_EXPAND_CASES])
def test_select_expand_tail_parity(case, select_form):
    """always_select_tail: the fused call equals dsa_select then dsa_expand_tail bit
    for bit, and the oracle's top-k and tail expansion."""
    rows, P, topk, kp, kind, fk, extra = case
    rng = np.random.default_rng(rows * 37 + P + kp)
    s = _tie_rows(rng, rows, P, kind) if P else np.zeros((rows, 0), np.float32)
    sk = O.select_k(topk, kp, P)
    width = O.out_width(topk, kp, True) + extra
    ctx = _tail_ctx(rng, rows, P, kp, fk)
    scores = torch.from_numpy(s).cuda()
    row_ctx = torch.from_numpy(ctx).cuda()
    ids = H.Guarded((rows, sk), torch.int32, -77)
    tok = H.Guarded((rows, width), torch.int32, -88)
    api.dsa_select_expand_tail(scores, topk, kp, fk, row_ctx, ids.t, tok.t)
    torch.cuda.synchronize()
    ids.check()
    tok.check()
    got_ids, got_tok = ids.t.cpu().numpy(), tok.t.cpu().numpy()
    ref_ids = torch.full((rows, sk), -1, dtype=torch.int32, device="cuda")
    if sk:
        api.dsa_select(scores, topk, kp, ref_ids)
    ref_tok = torch.empty((rows, width), dtype=torch.int32, device="cuda")
    api.dsa_expand_tail(ref_ids, fk, kp, topk, row_ctx, ref_tok)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(got_ids, ref_ids.cpu().numpy())
    np.testing.assert_array_equal(got_tok, ref_tok.cpu().numpy())
    for r in range(rows):
        o_ids = O.topk_pools(s[r].astype(np.float64), sk)
        np.testing.assert_array_equal(got_ids[r], o_ids, err_msg=f"row {r}")
        want = O.expand_selection_tail(o_ids, fk, kp, topk, int(ctx[r]), width)
        np.testing.assert_array_equal(got_tok[r], want, err_msg=f"row {r} ctx {ctx[r]}")


def test_expand_tail_parity():
    rng = np.random.default_rng(4)
    for kp, fk, topk, extra, rows in [(4, 0, 256, 0, 7), (4, 3, 2048, 0, 5), (1, 0, 7, 2, 3),
                                      (16, 16, 64, 5, 9), (3, 1, 30, 1, 8)]:
        sk = topk // kp
        ids = np.full((rows, sk), -1, dtype=np.int32)
        for r in range(rows):
            k = int(rng.integers(0, sk + 1))
            ids[r, :k] = np.sort(rng.choice(10 * sk + 10, k, replace=False))
        width = O.out_width(topk, kp, True) + extra
        ctx = _tail_ctx(rng, rows, 10 * sk + 10, kp, fk)
        out = H.Guarded((rows, width), torch.int32, -99)
        api.dsa_expand_tail(torch.from_numpy(ids).cuda(), fk, kp, topk,
                            torch.from_numpy(ctx).cuda(), out.t)
        torch.cuda.synchronize()
        out.check()
        got = out.t.cpu().numpy()
        for r in range(rows):
            np.testing.assert_array_equal(
                got[r], O.expand_selection_tail(ids[r], fk, kp, topk, int(ctx[r]), width),
                err_msg=f"kp {kp} row {r} ctx {ctx[r]}")


# ---------------------------------------------------------------------------
# dsa_sparse_mla_decode (fed oracle-side token ids)


MLA_CASES = [
    # name, heads, hidden, lens, block_size, out_width, o_absorb
    ("h4-tiny", 4, 1024, [2048], None, 256, True),
    ("h64-b1", 64, 512, [5000], None, 2048, True),
    ("h64-b3-paged", 64, 256, [3000, 700, 4097], 64, 512, True),
    ("h20-ragged", 20, 128, [999, 400], None, 300, True),
    ("h16-olat-only", 16, 0, [1500, 1500], None, 700, False),
    ("h96-two-groups", 96, 64, [800], None, 200, True),
    ("h64-b70-rows", 64, 64, [300] * 70, None, 64, True),
    ("h64-r40-two-chunks", 64, 128, [3000] * 40, None, 1024, False),
    ("h8-hidden96-fallback", 8, 96, [600, 333], None, 128, True),
]


def _token_rows(rng, wl, ow, empty_row=True):
    ids = np.full((wl.rows, ow), -1, dtype=np.int32)
    for r in range(wl.rows):
        L = int(wl.seq_lens[int(wl.row_seq[r])])
        if empty_row and r == 1:
            continue
        k = int(rng.integers(1, min(ow, L) + 1))
        pos = np.sort(rng.choice(ow, k, replace=False))
        ids[r, pos] = rng.choice(L, k, replace=False)
    return ids


@pytest.fixture(params=["mma", "tcgen05", "cluster"])
def mla_kernel(request):
    """Every attention kernel, each forced through DSA_OPT_MLA_KERNEL: the mma.sync
    split kernel, the persistent tcgen05 split kernel and the tcgen05 cluster decode
    kernel (the last two: 64 heads only; other head counts keep the mma.sync kernel).
    By default the library picks by batch size."""
    with api.mla_kernel(request.param):
        yield request.param


@pytest.mark.parametrize("case", MLA_CASES, ids=[c[0] for c in MLA_CASES])
def test_mla_parity(case, mla_kernel):
    name, heads, hidden, lens, bs, ow, with_o = case
    if mla_kernel in ("tcgen05", "cluster") and heads != 64:
        pytest.skip("the tcgen05 kernels serve 64 heads")
    g = _geom(heads=heads, hidden=max(hidden, 32), index_topk=ow)
    wl = W.make_workload(name, 300, g, lens, block_size=bs, with_raw=False,
                         with_o_absorb=with_o)
    layer = DsaDecodeLayer(wl, with_o_absorb=with_o, keep_olat=True, use_drawn_kpool=False)
    rng = np.random.default_rng(heads + ow)
    ids = _token_rows(rng, wl, ow)
    tok = torch.from_numpy(ids).cuda()
    olat = H.Guarded((wl.rows, heads, 512), torch.float32, 555.0)
    y = H.Guarded((wl.rows, g.hidden), torch.bfloat16, 3.0) if with_o else None
    api.dsa_sparse_mla_decode(layer.qlat, layer.row_seq, layer.ckv, layer.pg, tok,
                              g.softmax_scale, layer.o_absorb, None if y is None else y.t,
                              olat.t, layer.status, layer.fused_workspace())
    torch.cuda.synchronize()
    olat.check()
    if y is not None:
        y.check()
    assert int(layer.status.item()) == 0
    oq = H.OracleSeq(wl)
    A = H.f(wl.o_absorb) if with_o else None
    ro, ry = [], []
    for r in range(wl.rows):
        o_, y_, _ = O.sparse_mla_decode_row(H.f(wl.qlat[r]), oq.ckv(int(wl.row_seq[r])), ids[r],
                                            g.softmax_scale, A)
        ro.append(o_.reshape(-1))
        if with_o:
            ry.append(y_)
    H.check_attention(olat.t.cpu().numpy().reshape(wl.rows, -1), np.array(ro), f"{name} olat")
    if with_o:
        H.check_attention(y.t.float().cpu().numpy(), np.array(ry), f"{name} y")


def test_mla_rescaled_running_max(mla_kernel):
    """Latent rows whose norm grows with the token position: each 128-token chunk's
    score maximum exceeds the last by far more than 2^8 (log2 units), so the
    attention kernel's running maximum, output and sums are rescaled (64 heads)."""
    g = _geom(heads=64, hidden=64, index_topk=2048)
    wl = W.make_workload("rescale", 302, g, [4096, 2600], with_raw=False, with_o_absorb=False)
    ck = wl.ckv.float()
    flat = ck.view(-1, 512)
    n = flat.shape[0]
    # token row k of the cache gets factor 1 + 6 * (k mod 4096) / 4096
    fac = 1.0 + 6.0 * (torch.arange(n, dtype=torch.float32) % 4096) / 4096.0
    wl.ckv = (flat * fac[:, None]).to(torch.bfloat16).view(wl.ckv.shape)
    layer = DsaDecodeLayer(wl, with_o_absorb=False, keep_olat=True)
    rng = np.random.default_rng(11)
    ids = _token_rows(rng, wl, 2048, empty_row=False)
    for r in range(wl.rows):  # ascending token ids: later chunks hold the larger rows
        v = np.sort(ids[r][ids[r] >= 0])
        ids[r] = -1
        ids[r, : v.size] = v
    tok = torch.from_numpy(ids).cuda()
    olat = H.Guarded((wl.rows, 64, 512), torch.float32, 555.0)
    api.dsa_sparse_mla_decode(layer.qlat, layer.row_seq, layer.ckv, layer.pg, tok,
                              g.softmax_scale, None, None, olat.t, layer.status, layer.workspace)
    torch.cuda.synchronize()
    olat.check()
    assert int(layer.status.item()) == 0
    oq = H.OracleSeq(wl)
    ro = [O.sparse_mla_decode_row(H.f(wl.qlat[r]), oq.ckv(int(wl.row_seq[r])), ids[r],
                                  g.softmax_scale, None)[0].reshape(-1) for r in range(wl.rows)]
    H.check_attention(olat.t.cpu().numpy().reshape(wl.rows, -1), np.array(ro), "rescale olat")


PERSISTENT_CASES = [
    # name, query rows, sequence lengths, the rows' sequence, block_size, out_width,
    # rescale. More (row, split) units than SMs: the tcgen05 kernel's persistent CTAs
    # walk several units each, many 128-token chunks per unit, a ragged last chunk,
    # and rows with no tokens at all.
    ("r400-ow1000-paged", 400, [3100, 6000], 1, 64, 1000, False),
    ("r320-ow2048-rescale", 320, [4096, 2600], 0, None, 2048, True),
]


@pytest.mark.parametrize("case", PERSISTENT_CASES, ids=[c[0] for c in PERSISTENT_CASES])
def test_mla_persistent_many_units(case, mla_kernel):
    name, rows, lens, seq, bs, ow, rescale = case
    g = _geom(heads=64, hidden=64, index_topk=ow)
    wl = W.make_workload(name, 303, g, lens, block_size=bs, with_raw=False, with_o_absorb=False,
                         rows_ctx=[lens[seq]] * rows, prefill_seq=seq)
    if rescale:
        # token row k gets factor 1 + 6 * (k mod 4096) / 4096: later chunks of a row
        # with ascending ids score far above the earlier ones (running-max rescales)
        flat = wl.ckv.float().view(-1, 512)
        fac = 1.0 + 6.0 * (torch.arange(flat.shape[0], dtype=torch.float32) % 4096) / 4096.0
        wl.ckv = (flat * fac[:, None]).to(torch.bfloat16).view(wl.ckv.shape)
    layer = DsaDecodeLayer(wl, with_o_absorb=False, keep_olat=True)
    rng = np.random.default_rng(ow + len(lens))
    ids = _token_rows(rng, wl, ow)
    ids[7] = -1  # another row with no tokens
    if rescale:
        for r in range(wl.rows):
            v = np.sort(ids[r][ids[r] >= 0])
            ids[r] = -1
            ids[r, : v.size] = v
    tok = torch.from_numpy(ids).cuda()
    olat = H.Guarded((wl.rows, 64, 512), torch.float32, 555.0)
    api.dsa_sparse_mla_decode(layer.qlat, layer.row_seq, layer.ckv, layer.pg, tok,
                              g.softmax_scale, None, None, olat.t, layer.status, layer.workspace)
    torch.cuda.synchronize()
    olat.check()
    assert int(layer.status.item()) == 0
    oq = H.OracleSeq(wl)
    ro = [O.sparse_mla_decode_row(H.f(wl.qlat[r]), oq.ckv(int(wl.row_seq[r])), ids[r],
                                  g.softmax_scale, None)[0].reshape(-1) for r in range(wl.rows)]
    H.check_attention(olat.t.cpu().numpy().reshape(wl.rows, -1), np.array(ro), f"{name} olat")


def test_mla_empty_token_lists(mla_kernel):
    """out_width 0: no unit has a chunk; olat and y are exactly zero (R16)."""
    g = _geom(heads=64, hidden=64, index_topk=64)
    wl = W.make_workload("empty", 304, g, [3000, 700], with_raw=False)
    layer = DsaDecodeLayer(wl, keep_olat=True)
    tok = torch.empty((wl.rows, 0), dtype=torch.int32, device="cuda")
    olat = H.Guarded((wl.rows, 64, 512), torch.float32, 555.0)
    y = H.Guarded((wl.rows, g.hidden), torch.bfloat16, 3.0)
    ws = torch.zeros(max(1, api.dsa_sparse_mla_decode_workspace(wl.rows, 64, 0, g.hidden, True)),
                     dtype=torch.uint8, device="cuda")
    api.dsa_sparse_mla_decode(layer.qlat, layer.row_seq, layer.ckv, layer.pg, tok,
                              g.softmax_scale, layer.o_absorb, y.t, olat.t, layer.status, ws)
    torch.cuda.synchronize()
    olat.check()
    y.check()
    assert int(layer.status.item()) == 0
    assert not olat.t.any() and not y.t.float().any()


def test_mla_bad_ids_set_status_and_are_skipped():
    g = _geom(heads=8, hidden=64, index_topk=128)
    wl = W.make_workload("bad", 301, g, [500, 200], block_size=64, with_raw=False)
    layer = DsaDecodeLayer(wl, keep_olat=True)
    rng = np.random.default_rng(5)
    ids = _token_rows(rng, wl, 128, empty_row=False)
    bad = ids.copy()
    bad[0, 3] = 500        # == seq_len: out of range
    bad[1, 5] = -5         # < -1
    bad[1, 6] = 10 ** 6    # far out of range
    clean = bad.copy()
    clean[0, 3] = clean[1, 5] = clean[1, 6] = -1
    layer.status.zero_()
    api.dsa_sparse_mla_decode(layer.qlat, layer.row_seq, layer.ckv, layer.pg,
                              torch.from_numpy(bad).cuda(), g.softmax_scale, layer.o_absorb,
                              layer.y, layer.olat, layer.status, layer.fused_workspace())
    torch.cuda.synchronize()
    assert int(layer.status.item()) & api._lib.DSA_STATUS_BAD_TOKEN
    got = layer.olat.cpu().numpy().reshape(wl.rows, -1)
    assert np.isfinite(got).all()
    oq = H.OracleSeq(wl)
    ref = [O.sparse_mla_decode_row(H.f(wl.qlat[r]), oq.ckv(r), clean[r], g.softmax_scale)[0]
           .reshape(-1) for r in range(wl.rows)]
    H.check_attention(got, np.array(ref), "olat with bad ids")


def test_bad_block_table_entry_sets_status():
    g = _geom(heads=8, hidden=64, index_topk=128)
    wl = W.make_workload("badblk", 302, g, [300, 300], block_size=64, with_raw=False,
                         direct_kpool=True)
    layer = DsaDecodeLayer(wl, keep_olat=True, use_drawn_kpool=True)
    bt = layer.block_table.clone()
    bt[1, 2] = wl.num_blocks + 5  # corrupt one entry of sequence 1
    pg = api.paging(layer.seq_lens, wl.max_seq_len, bt, 64, wl.num_blocks)
    layer.status.zero_()
    api.dsa_score(layer.qidx, layer.w, layer.row_seq, layer.row_ctx, layer.kpool,
                  layer.pool_valid, pg, 0, 4, g.index_scale, layer.scores, status=layer.status)
    ids = torch.full((2, 128), -1, dtype=torch.int32)
    ids[1, :10] = torch.arange(128, 138)  # tokens in block 2 of sequence 1
    api.dsa_sparse_mla_decode(layer.qlat, layer.row_seq, layer.ckv, pg, ids.cuda(),
                              g.softmax_scale, layer.o_absorb, layer.y, layer.olat, layer.status,
                              layer.fused_workspace())
    torch.cuda.synchronize()
    assert int(layer.status.item()) & api._lib.DSA_STATUS_BAD_BLOCK
    s = layer.scores.cpu().numpy()
    assert np.isneginf(s[1, 32:48]).all()  # pools of the bad block are not candidates
    assert (layer.olat[1].abs().sum().item() == 0.0)  # all of row 1's tokens skipped


PROJECT_CASES = [(8, 64, 4096), (1, 64, 4096), (3, 4, 1024), (70, 16, 256), (20, 8, 128),
                 (64, 64, 4096), (128, 8, 512), (16, 64, 1024), (33, 8, 384),
                 # tall A with a short K (1,536): fewer K shares per tile (2, then 1)
                 (8, 3, 12800), (8, 3, 36864), (40, 3, 19456),
                 # short and wide: 128 CTAs share each 64-row block (the many-CTA reduce)
                 (8, 64, 128)]


@pytest.fixture(params=["tcgen05", "mma"])
def proj_kernel(request):
    """Both projection kernels, forced through DSA_OPT_PROJECT_KERNEL (shapes the
    tensor-core form does not take, hidden not a multiple of 128, run the mma.sync
    form either way)."""
    with api.project_kernel(request.param):
        yield request.param


@pytest.mark.parametrize("rows,heads,hidden", PROJECT_CASES)
def test_latent_project_parity(rows, heads, hidden, proj_kernel):
    rng = np.random.default_rng(rows * 100 + heads)
    olat = torch.from_numpy(rng.standard_normal((rows, heads, 512)).astype(np.float32))
    A = torch.from_numpy((rng.standard_normal((hidden, heads * 512)) * 0.02).astype(np.float32)
                         ).to(torch.bfloat16)
    ws = torch.zeros(max(1, api.dsa_latent_project_workspace(rows, heads, hidden)),
                     dtype=torch.uint8, device="cuda")
    y = H.Guarded((rows, hidden), torch.bfloat16, 5.0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.dsa_latent_project(olat.cuda(), A.cuda(), y.t, status, ws)
    torch.cuda.synchronize()
    y.check()
    assert int(status.item()) == 0
    ref = np.array([O.latent_project(olat[r].numpy().astype(np.float64), H.f(A))[0]
                    for r in range(rows)])
    H.check_attention(y.t.float().cpu().numpy(), ref, "y")


@pytest.mark.parametrize("rows,heads,hidden", [(8, 8, 1024), (40, 16, 512), (3, 64, 4096)])
def test_projection_wait_timeout_flags_status(rows, heads, hidden):
    """A bounded pipeline wait that runs out: DSA_OPT_INJECT_STALL stops the next
    tensor-core projection's copies before their last stage, so its MMA warp waits on
    a stage that nothing fills. After about a second that launch ORs
    DSA_STATUS_TIMEOUT into its status word and returns (no fault, no hang); the
    option is taken by that launch, and the next launch on the same context is
    bit-identical to one before it."""
    rng = np.random.default_rng(rows * 3 + hidden)
    olat = torch.from_numpy(rng.standard_normal((rows, heads, 512)).astype(np.float32)).cuda()
    A = torch.from_numpy((rng.standard_normal((hidden, heads * 512)) * 0.02).astype(np.float32)
                         ).to(torch.bfloat16).cuda()
    ws = torch.zeros(max(1, api.dsa_latent_project_workspace(rows, heads, hidden)),
                     dtype=torch.uint8, device="cuda")
    with api.project_kernel("tcgen05"):
        st0 = torch.zeros(1, dtype=torch.int32, device="cuda")
        y0 = torch.zeros((rows, hidden), dtype=torch.bfloat16, device="cuda")
        api.dsa_latent_project(olat, A, y0, st0, ws)
        torch.cuda.synchronize()
        assert int(st0.item()) == 0
        st1 = torch.zeros(1, dtype=torch.int32, device="cuda")
        y1 = torch.zeros_like(y0)
        api.dsa_set_option(api._lib.DSA_OPT_INJECT_STALL, 1)
        try:
            api.dsa_latent_project(olat, A, y1, st1, ws)
        finally:
            taken = api.dsa_get_option(api._lib.DSA_OPT_INJECT_STALL)
            api.dsa_set_option(api._lib.DSA_OPT_INJECT_STALL, 0)
        torch.cuda.synchronize()
        assert taken == 0
        assert int(st1.item()) & api._lib.DSA_STATUS_TIMEOUT
        st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
        y2 = torch.zeros_like(y0)
        api.dsa_latent_project(olat, A, y2, st2, ws)
        torch.cuda.synchronize()
        assert int(st2.item()) == 0
        assert torch.equal(y0, y2)


@pytest.mark.parametrize("rows,heads,hidden,frac", [(8, 64, 4096, 0.25), (64, 64, 4096, 0.25),
                                                    (70, 16, 256, 1.0), (20, 8, 128, 0.4)])
def test_project_after_l2_prefetch_is_identical(rows, heads, hidden, frac, proj_kernel):
    """Staging part of o_absorb in L2 (dsa_prefetch_l2) changes nothing in y: the
    tensor-core projection then also returns the staged lines to normal priority
    (an extra arrival on its ring), over one or several 64-row launches."""
    rng = np.random.default_rng(rows + heads + hidden)
    olat = torch.from_numpy(rng.standard_normal((rows, heads, 512)).astype(np.float32)).cuda()
    A = torch.from_numpy((rng.standard_normal((hidden, heads * 512)) * 0.02).astype(np.float32)
                         ).to(torch.bfloat16).cuda()
    ws = torch.zeros(max(1, api.dsa_latent_project_workspace(rows, heads, hidden)),
                     dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y0 = torch.zeros((rows, hidden), dtype=torch.bfloat16, device="cuda")
    api.dsa_latent_project(olat, A, y0, status, ws)
    y1 = torch.zeros_like(y0)
    api.dsa_prefetch_l2(A, int(A.numel() * 2 * frac))
    api.dsa_latent_project(olat, A, y1, status, ws)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(y0, y1)


def _paged_small_wl():
    return W.make_workload("paged-small-pf", 6, W.Geometry(**W.GLM53), [3000, 5000, 700, 4096],
                           block_size=64, max_seq_len=5120, invalid_per_seq=7)


@pytest.mark.parametrize("make", [W.tiny, _paged_small_wl], ids=["tiny", "paged"])
def test_step_with_l2_prefetch_branch_is_identical(make):
    """The step graph with the o_absorb prefetch on a forked branch equals the plain
    step bit for bit."""
    wl = make()
    plain = DsaDecodeLayer(wl, keep_olat=True, l2_prefetch_bytes=0)
    pf = DsaDecodeLayer(wl, keep_olat=True, l2_prefetch_bytes=wl.o_absorb.numel())  # half
    assert pf.l2_prefetch_bytes > 0 and pf.launches_per_step() == plain.launches_per_step() + 1
    for lay in (plain, pf):
        lay.compress()
        lay.capture()
        lay.graph.replay()
    torch.cuda.synchronize()
    assert int(pf.status.item()) == 0
    for k in ("pool_ids", "token_ids", "olat", "y"):
        assert torch.equal(getattr(pf, k), getattr(plain, k)), k
