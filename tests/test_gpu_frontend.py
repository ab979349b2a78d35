"""Projection front-end (dsa_frontend) against the oracle's frontend_row, and the
whole decode layer (front-end -> append -> step) under graph replay."""
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
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


F32_EPS = 2.0 ** -24


def _acc_bound(Wm, v):
    """Worst-case error of an f32 sum of the products W[n, k] v[k] (each product of
    two bf16 values is exact in f32): K * 2^-24 * sum |W v| per output."""
    return Wm.shape[1] * F32_EPS * (np.abs(Wm) @ np.abs(v))


def _check_rounded(gpu, exact, extra, what):
    """gpu is bf16 of (exact + e), |e| <= extra: within half an ulp plus extra."""
    lim = 0.5 * H.bf16_ulp(np.abs(exact) + extra) + extra + 1e-30
    err = np.abs(gpu - exact)
    assert (err <= lim).all(), f"{what}: max excess {(err - lim).max():.3e}"


def _check_frontend(layer, fe, rows):
    g = layer.geom
    f = lambda t: t.float().cpu().numpy().astype(np.float64)
    Wqa, Wkva, Wk, Wg, Wp = (f(t) for t in (fe.q_a_proj, fe.kv_a_proj, fe.wk, fe.compress_gate,
                                             fe.weights_proj))
    gq, gkv, Wqabs, Wqb = f(fe.q_a_norm), f(fe.kv_a_norm), f(fe.q_absorb), f(fe.wq_b)
    x_all = f(fe.x)
    got = {k: getattr(layer, n).float().cpu().numpy().astype(np.float64)
           for k, n in (("qlat", "qlat"), ("qidx", "qidx"), ("w", "w"), ("k_raw", "k_new"),
                        ("gate", "gate_new"), ("ckv", "ckv_new"))}
    for r in rows:
        x = x_all[r]
        ref = O.frontend_row(x, Wqa, gq, Wkva, gkv, Wk, Wg, Wp, Wqabs, Wqb, fe.eps, g.heads,
                             g.index_heads)
        # x projections: plain sums of exact products
        np.testing.assert_array_less(np.abs(got["w"][r] - Wp @ x), _acc_bound(Wp, x) + 1e-30)
        _check_rounded(got["k_raw"][r], Wk @ x, _acc_bound(Wk, x), f"k_raw {r}")
        _check_rounded(got["gate"][r], Wg @ x, _acc_bound(Wg, x), f"gate {r}")
        # norms: the f32 sums' error, relative error of the f32 norm, then bf16
        for name, Wm, gm in (("ckv", Wkva, gkv), ("q_lora", Wqa, gq)):
            y = Wm @ x
            ex = O.rms_norm(y, gm, fe.eps)
            rinv = 1.0 / np.sqrt((y * y).mean() + fe.eps)
            extra = np.abs(gm) * rinv * _acc_bound(Wm, x) * 2 + np.abs(ex) * 1e-5
            if name == "ckv":
                _check_rounded(got["ckv"][r], ex, extra, f"ckv {r}")
            else:
                ql_extra = extra
                ql_exact = ex
        # qlat, qidx from q_lora: the oracle's bf16 q_lora may differ from the
        # device's in a rare element whose exact value sits within ql_extra of a
        # rounding midpoint; allow two such flips per output.
        near = np.abs(np.abs(ql_exact - ref["q_lora"]) - 0.5 * H.bf16_ulp(ql_exact)) <= ql_extra
        flip = H.bf16_ulp(ql_exact) * near
        for name, Wm, shape in (("qlat", Wqabs, (g.heads, -1)), ("qidx", Wqb, (g.index_heads, -1))):
            pre = Wm @ ref["q_lora"]
            extra = _acc_bound(Wm, ref["q_lora"]) + 2 * (np.abs(Wm) * flip[None, :]).max(axis=1)
            _check_rounded(got[name][r].reshape(-1), pre, extra, f"{name} {r}")


FRONT_CASES = [
    # name, hidden, q_lora, heads, index_heads, ihd, rows
    ("small-r3", 512, 256, 4, 8, 64, 3),
    ("small-r70", 512, 256, 2, 4, 128, 70),
    ("glm-r8", 4096, 1536, 64, 32, 128, 8),
]


@pytest.mark.parametrize("case", FRONT_CASES, ids=[c[0] for c in FRONT_CASES])
def test_frontend_parity(case):
    name, hidden, ql, heads, hi, ihd, rows = case
    g = W.Geometry(index_kpool=4, index_heads=hi, index_head_dim=ihd, index_topk=64, heads=heads,
                   hidden=hidden)
    wl = W.make_workload(f"fe-{name}", 51, g, [300] * rows, with_raw=False, with_o_absorb=False)
    fe = W.make_frontend(g, rows, q_lora_rank=ql, seed=52)
    layer = DsaDecodeLayer(wl, with_o_absorb=False, keep_olat=True, frontend=fe)
    layer.status.zero_()
    for t in (layer.qlat, layer.qidx, layer.w, layer.k_new, layer.gate_new, layer.ckv_new):
        t.fill_(7)
    layer.frontend()
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    _check_frontend(layer, fe, range(rows))


def test_full_layer_graph_replay_matches_eager():
    """front-end -> append -> step, captured once: every replay equals the same calls
    made eagerly on a twin layer, bit for bit, and the step consumes exactly what
    the front-end produced."""
    g = W.Geometry(index_kpool=4, index_heads=32, index_head_dim=128, index_topk=256, heads=8,
                   hidden=512)
    wl = W.make_workload("fe-layer", 53, g, [300, 517, 77])
    fe = W.make_frontend(g, wl.rows, q_lora_rank=512, seed=54)
    L0 = wl.seq_lens.astype(np.int64) - 5
    a = DsaDecodeLayer(wl, keep_olat=True, decode_from=L0, frontend=fe)
    b = DsaDecodeLayer(wl, keep_olat=True, decode_from=L0, frontend=fe)
    for lay in (a, b):
        lay.status.zero_()
        lay.compress()
    a.capture_layer()
    for i in range(5):
        a.layer_graph.replay()
        b.layer_step()
        torch.cuda.synchronize()
        for k in ("qlat", "qidx", "w", "k_new", "ckv_new", "scores", "pool_ids", "token_ids",
                  "olat", "y", "seq_lens", "kpool"):
            assert torch.equal(getattr(a, k), getattr(b, k)), f"step {i}: {k}"
    assert int(a.status.item()) == 0 and a.seq_lens.tolist() == wl.seq_lens.tolist()
    # The appended rows are the front-end's outputs for the last step.
    for bi in range(wl.batch):
        t = int(wl.seq_lens[bi]) - 1
        row = int(a._token_rows(bi, t, t + 1)[0])
        assert torch.equal(a.k_raw.view(-1, 128)[row], a.k_new[bi])
        assert torch.equal(a.ckv.view(-1, 512)[row], a.ckv_new[bi])
    _check_frontend(a, fe, range(wl.rows))
