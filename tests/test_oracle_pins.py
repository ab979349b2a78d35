"""Pins for the CPU oracle: worked examples, closed forms, invariants and brute
force, each fixed independently of the oracle's own code. CPU only."""
import itertools
import math

import numpy as np
import pytest
import torch

from oracle import dsa_oracle as O
from sparse_attention_decode_kpool_gb300 import workloads as W
from tests._golden import load_kv, load_pairs


# ---------------------------------------------------------------------------
# bf16 rounding


def test_bf16_golden():
    for x, want in load_pairs("bf16_rne.txt"):
        got = float(O.bf16_round(np.array([x]))[0])
        assert got == want or (math.isinf(want) and got == want), (x, got, want)


def test_bf16_matches_library_on_float32_inputs():
    # For float32 inputs, rounding float64 -> bf16 directly equals the library's
    # float32 -> bf16 nearest-even conversion.
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(200000).astype(np.float32),
        (rng.standard_normal(20000) * 1e30).astype(np.float32),
        (rng.standard_normal(20000) * 1e-39).astype(np.float32),  # subnormals
        rng.integers(0, 2**32, 50000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ])
    x = x[np.isfinite(x)]
    lib = torch.from_numpy(x).to(torch.bfloat16).float().numpy().astype(np.float64)
    ours = O.bf16_round(x.astype(np.float64))
    np.testing.assert_array_equal(ours, lib)


def test_bf16_idempotent_and_signed_zero():
    v = O.bf16_round(np.random.default_rng(1).standard_normal(1000))
    np.testing.assert_array_equal(O.bf16_round(v), v)
    assert math.copysign(1.0, O.bf16_round(np.array([-0.0]))[0]) == -1.0


# ---------------------------------------------------------------------------
# LayerNorm with bias (k_norm)


def test_layernorm_golden():
    g = load_kv("layernorm.txt")
    for x, ga, be, ep, ex in zip(g["x"], g["gamma"], g["beta"], g["eps"], g["expect"]):
        got = O.layernorm_bias(x, ga, be, float(ep[0]))
        np.testing.assert_allclose(got, ex, rtol=0, atol=1e-14)


def test_layernorm_constant_row_gives_bias():
    rng = np.random.default_rng(2)
    beta = rng.standard_normal(64)
    gamma = rng.standard_normal(64)
    x = np.full(64, 3.25)
    np.testing.assert_array_equal(O.layernorm_bias(x, gamma, beta, 1e-6), beta)


def test_layernorm_moments_closed_form():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((10, 128)) * 3 + 1
    eps = 0.5
    y = O.layernorm_bias(x, np.ones(128), np.zeros(128), eps)
    var = x.var(axis=1)  # biased
    np.testing.assert_allclose(y.mean(axis=1), 0, atol=1e-12)
    np.testing.assert_allclose(y.var(axis=1), var / (var + eps), rtol=1e-12)


# ---------------------------------------------------------------------------
# kpool_compress


def _pool_golden():
    g = load_kv("kpool_compress.txt")
    kp = int(g["kpool"][0][0])
    fk = int(g["first_key"][0][0])
    k = g["k"][0].reshape(-1, 2)
    ape = g["ape"][0].reshape(kp, 2)
    return g, kp, fk, k, ape


def test_pool_golden():
    g, kp, fk, k, ape = _pool_golden()
    gate = np.zeros_like(k)
    keys, pv, pidx = O.kpool_compress(k, gate, np.ones(len(k), np.uint8), ape,
                                      np.ones(2), np.zeros(2), 0.0, fk, kp)
    np.testing.assert_allclose(keys, g["keys"][0].reshape(-1, 2), rtol=0, atol=1e-15)
    np.testing.assert_array_equal(pv, [1, 1])
    np.testing.assert_array_equal(pidx, g["pool_idx"][0].reshape(-1, 2))
    keys2, pv2, _ = O.kpool_compress(k, gate, g["valid_case2"][0].astype(np.uint8), ape,
                                     np.ones(2), np.zeros(2), 0.0, fk, kp)
    np.testing.assert_allclose(keys2, g["keys_case2"][0].reshape(-1, 2), rtol=0, atol=1e-15)
    np.testing.assert_array_equal(pv2, g["pool_valid_case2"][0])


def _rand_pool_inputs(S=64, ihd=16, kp=4, seed=5):
    rng = np.random.default_rng(seed)
    k = O.bf16_round(rng.standard_normal((S, ihd)))
    gate = O.bf16_round(rng.standard_normal((S, ihd)))
    ape = rng.standard_normal((kp, ihd)) * 0.1
    gam = O.bf16_round(1 + 0.1 * rng.standard_normal(ihd))
    bet = O.bf16_round(0.1 * rng.standard_normal(ihd))
    return k, gate, ape, gam, bet


def test_pool_kpool1_is_normalised_key():
    k, gate, _, gam, bet = _rand_pool_inputs(kp=1)
    ape = np.random.default_rng(9).standard_normal((1, 16))
    keys, pv, _ = O.kpool_compress(k, gate, np.ones(64, np.uint8), ape, gam, bet, 1e-6, 0, 1)
    np.testing.assert_array_equal(keys, O.bf16_round(O.layernorm_bias(k, gam, bet, 1e-6)))
    assert pv.all()


def test_pool_equal_logits_give_slot_mean():
    k, _, _, gam, bet = _rand_pool_inputs()
    # logits vary across channels but not across slots of a pool
    chan = np.linspace(-3, 3, 16)
    gate = np.tile(chan, (64, 1))
    ape = np.zeros((4, 16))
    keys, _, _ = O.kpool_compress(k, gate, np.ones(64, np.uint8), ape, gam, bet, 1e-6, 0, 4)
    kn = O.bf16_round(O.layernorm_bias(k, gam, bet, 1e-6)).reshape(16, 4, 16)
    np.testing.assert_allclose(keys, O.bf16_round(kn.mean(axis=1)), rtol=0, atol=0)


def test_pool_dominant_slot():
    k, gate, ape, gam, bet = _rand_pool_inputs()
    gate = np.zeros_like(gate)
    ape = np.zeros((4, 16))
    ape[2, :] = 60.0  # slot 2 dominates every channel by e^60
    keys, _, _ = O.kpool_compress(k, gate, np.ones(64, np.uint8), ape, gam, bet, 1e-6, 0, 4)
    kn = O.bf16_round(O.layernorm_bias(k, gam, bet, 1e-6)).reshape(16, 4, 16)
    np.testing.assert_array_equal(keys, kn[:, 2, :])


def test_pool_weights_are_convex():
    # identical normalised keys in all slots -> the pool equals that key for any logits
    rng = np.random.default_rng(11)
    row = rng.standard_normal(16)
    k = np.tile(row, (64, 1))
    gate = rng.standard_normal((64, 16)) * 3
    keys, _, _ = O.kpool_compress(k, gate, np.ones(64, np.uint8), rng.standard_normal((4, 16)),
                                  np.ones(16), np.zeros(16), 1e-6, 0, 4)
    kn = O.bf16_round(O.layernorm_bias(row, np.ones(16), np.zeros(16), 1e-6))
    np.testing.assert_allclose(keys, np.tile(kn, (16, 1)), rtol=0, atol=0)


def test_pool_softmax_shift_invariance():
    k, gate, ape, gam, bet = _rand_pool_inputs()
    base, _, _ = O.kpool_compress(k, gate, np.ones(64, np.uint8), ape, gam, bet, 1e-6, 0, 4)
    shifted = ape + np.linspace(-5, 5, 16)[None, :]  # same shift for every slot of a channel
    got, _, _ = O.kpool_compress(k, gate, np.ones(64, np.uint8), shifted, gam, bet, 1e-6, 0, 4)
    np.testing.assert_allclose(got, base, rtol=0, atol=2 ** -8 * np.abs(base).max())
    assert (got == base).mean() > 0.99


def test_pool_transposed_ape_differs():
    # ape is [slot, channel]: using it as [channel, slot] changes the result
    g, kp, fk, k, ape = _pool_golden()
    keys, _, _ = O.kpool_compress(k, np.zeros_like(k), np.ones(len(k), np.uint8), ape.T,
                                  np.ones(2), np.zeros(2), 0.0, fk, kp)
    assert not np.allclose(keys, g["keys"][0].reshape(-1, 2))


@pytest.mark.parametrize("S,fk,kp,P", [(2047, 0, 4, 511), (2048, 0, 4, 512), (5, 2, 4, 0),
                                       (10, 2, 4, 2), (3, 0, 4, 0), (0, 0, 4, 0), (13, 1, 3, 4)])
def test_pool_count_drops_partial(S, fk, kp, P):
    rng = np.random.default_rng(0)
    k = rng.standard_normal((S, 8))
    keys, pv, pidx = O.kpool_compress(k, k, np.ones(S, np.uint8), np.zeros((kp, 8)),
                                      np.ones(8), np.zeros(8), 1e-6, fk, kp)
    assert keys.shape == (P, 8) and pv.shape == (P,) and pidx.shape == (P, kp)
    if P:
        assert pidx[0, 0] == fk and pidx[-1, -1] == fk + P * kp - 1 <= S - 1


def test_pool_tiny_workload_validity():
    wl = W.tiny()
    v = wl.valid.numpy()[0]
    keys, pv, _ = O.kpool_compress(wl.k_raw.float().numpy()[0], wl.gate.float().numpy()[0], v,
                                   wl.ape.numpy(), wl.ln_w.float().numpy(), wl.ln_b.float().numpy(),
                                   wl.geom.eps, 0, 4)
    assert keys.shape == (512, 64)
    assert pv[:511].all() and pv[511] == 0 and pv.sum() == 511
    assert not keys[511].any()


# ---------------------------------------------------------------------------
# index_scores


def test_score_golden():
    g = load_kv("index_scores.txt")
    q = g["q"][0].reshape(2, 2)
    keys = g["keys"][0].reshape(-1, 2)
    pv = g["pool_valid"][0].astype(np.uint8)
    for w, ex in ((g["w"][0], g["expect"][0]), (g["w_neg"][0], g["expect_neg"][0])):
        got = O.index_scores(q, w, keys, pv, 17, 0, 4, 0.5, 6)
        np.testing.assert_array_equal(got, ex)


def test_score_orthogonal_is_zero_and_parallel_closed_form():
    rng = np.random.default_rng(4)
    a = rng.standard_normal(8)
    b = rng.standard_normal(8)
    b -= a * (a @ b) / (a @ a)  # b orthogonal to a
    s0 = O.index_scores(a[None], [1.0], b[None], [1], 4, 0, 4, 0.3)
    assert abs(s0[0]) < 1e-14
    s1 = O.index_scores(a[None], [0.7], (2.5 * a)[None], [1], 4, 0, 4, 0.3)
    np.testing.assert_allclose(s1[0], 0.7 * 0.3 * np.linalg.norm(a) * np.linalg.norm(2.5 * a),
                               rtol=1e-14)


def test_score_positive_homogeneity():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((4, 16))
    w = rng.random(4)
    keys = rng.standard_normal((30, 16))
    s = O.index_scores(q, w, keys, np.ones(30, np.uint8), 200, 0, 4, 0.25)
    s2 = O.index_scores(q, 2 * w, keys, np.ones(30, np.uint8), 200, 0, 4, 0.25)
    np.testing.assert_array_equal(s2, 2 * s)


@pytest.mark.parametrize("ctx,fk,kp,nvis", [(17, 0, 4, 4), (16, 0, 4, 4), (15, 0, 4, 3),
                                            (3, 0, 4, 0), (18, 2, 4, 4), (17, 2, 4, 3)])
def test_score_visibility(ctx, fk, kp, nvis):
    keys = np.ones((10, 2))
    s = O.index_scores(np.ones((1, 2)), [1.0], keys, np.ones(10, np.uint8), ctx, fk, kp, 1.0, 12)
    assert np.isfinite(s).sum() == nvis and np.isfinite(s[:nvis]).all()


def test_score_relu_zero_ties():
    # all dots negative -> every score exactly 0; top-k then keeps the lowest ids
    keys = -np.abs(np.random.default_rng(6).standard_normal((12, 4)))
    s = O.index_scores(np.ones((2, 4)), [1.0, 0.5], keys, np.ones(12, np.uint8), 48, 0, 4, 1.0)
    assert (s == 0).all()
    np.testing.assert_array_equal(O.topk_pools(s, 5), [0, 1, 2, 3, 4])


# ---------------------------------------------------------------------------
# top-k and expand


def test_select_k_and_out_width():
    assert O.select_k(2048, 4, 65536) == 512
    assert O.select_k(256, 4, 512) == 64
    assert O.select_k(256, 4, 50) == 50
    assert O.out_width(2048, 4) == 2048 and O.out_width(2048, 4, True) == 2051


def test_topk_golden():
    g = load_kv("topk_expand.txt")
    s = g["scores"][0]
    for key, sk in (("sk4", 4), ("sk6", 6), ("sk9", 9)):
        np.testing.assert_array_equal(O.topk_pools(s, sk), g[key][0])


def _brute_topk(s, sk):
    fin = [i for i in range(len(s)) if np.isfinite(s[i])]
    kk = min(sk, len(fin))

    def beats(i, j):
        return s[i] > s[j] or (s[i] == s[j] and i < j)

    sols = [c for c in itertools.combinations(fin, kk)
            if all(beats(i, j) for i in c for j in fin if j not in c)]
    assert len(sols) == 1
    return list(sols[0]) + [-1] * (sk - kk)


def test_topk_brute_force_tiny():
    rng = np.random.default_rng(8)
    vals = np.array([-np.inf, -1.0, -0.0, 0.0, 1.0, 2.0])
    for trial in range(400):
        P = int(rng.integers(0, 9))
        s = vals[rng.integers(0, len(vals), P)]
        for sk in range(0, P + 2):
            np.testing.assert_array_equal(O.topk_pools(s, sk), _brute_topk(s, sk))


def test_topk_all_equal_and_all_masked():
    np.testing.assert_array_equal(O.topk_pools(np.full(10, 0.5), 3), [0, 1, 2])
    np.testing.assert_array_equal(O.topk_pools(np.full(10, -np.inf), 3), [-1, -1, -1])


def test_expand_golden():
    g = load_kv("topk_expand.txt")
    got = O.expand_selection(g["pool_ids"][0].astype(int), 1, 4, 16)
    np.testing.assert_array_equal(got, g["tokens"][0])


def test_expand_properties():
    rng = np.random.default_rng(10)
    for _ in range(50):
        kp = int(rng.integers(1, 9))
        sk = int(rng.integers(0, 20))
        kk = int(rng.integers(0, sk + 1))
        ids = np.sort(rng.choice(100, kk, replace=False)).tolist() + [-1] * (sk - kk)
        fk = int(rng.integers(0, 5))
        width = sk * kp + int(rng.integers(0, 7))
        row = O.expand_selection(ids, fk, kp, width)
        assert row.shape == (width,)
        assert (row != -1).sum() == kk * kp
        sel = row[row != -1]
        assert (np.diff(sel) > 0).all()
        assert set(sel.tolist()) == {fk + p * kp + s for p in ids[:kk] for s in range(kp)}
    assert (O.expand_selection([-1, -1], 0, 4, 8) == -1).all()


def test_expand_tail_golden():
    g = load_kv("expand_tail.txt")
    assert len(g["case"]) == 6
    for c, pools, toks in zip(g["case"], g["pools"], g["tokens"]):
        ctx, fk, kp, topk = (int(v) for v in c)
        got = O.expand_selection_tail(pools.astype(int), fk, kp, topk, ctx)
        np.testing.assert_array_equal(got, toks)


def test_expand_tail_covers_every_seen_token_once():
    # Selecting every pool of a row: pools plus tail are exactly the tokens
    # [first_key, ctx), each once, and the tail fits the kpool - 1 extra slots.
    rng = np.random.default_rng(12)
    for _ in range(300):
        kp = int(rng.integers(1, 9))
        fk = int(rng.integers(0, 6))
        ctx = int(rng.integers(0, 60))
        P = max(0, (ctx - fk) // kp)
        topk = kp * (P + int(rng.integers(0, 3)))
        if topk == 0:
            topk = kp
        sk = O.select_k(topk, kp, P)
        ids = list(range(P))[:sk] + [-1] * (sk - min(sk, P))
        row = O.expand_selection_tail(ids, fk, kp, topk, ctx)
        assert row.shape == (O.out_width(topk, kp, True),)
        seen = row[row >= 0]
        assert sorted(seen.tolist()) == list(range(fk, max(fk, ctx)))
        assert (np.diff(seen) > 0).all()
        tail = row[topk:]
        n_tail = (ctx - fk) % kp if ctx > fk else 0
        assert (tail >= 0).sum() == n_tail
    # Without a selection the tail still comes through, and nothing else does.
    row = O.expand_selection_tail([-1, -1], 0, 4, 8, 7)
    np.testing.assert_array_equal(row, [-1] * 8 + [4, 5, 6])


def test_dense_equivalence_with_tail():
    # With always_select_tail and index_topk covering every candidate pool, sparse
    # attention equals dense masked attention over the tokens of candidate pools
    # plus every token past the last whole pool.
    g = W.Geometry(index_kpool=4, index_heads=4, index_head_dim=32, index_topk=4 * 64,
                   heads=3, hidden=64, kv_lora_rank=32)
    L, fk = 206, 3
    wl = W.make_workload("t", 23, g, [L], invalid_per_seq=9)
    k = wl.k_raw.float().numpy()[0]
    keys, pv, _ = O.kpool_compress(k, wl.gate.float().numpy()[0], wl.valid.numpy()[0],
                                   wl.ape.numpy(), wl.ln_w.float().numpy(),
                                   wl.ln_b.float().numpy(), g.eps, fk, 4)
    ckv = wl.ckv.float().numpy()[0]
    r = O.decode_row(wl.qidx.float().numpy()[0], wl.w.numpy()[0], keys, pv, L, fk, 4,
                     g.index_scale, g.index_topk, wl.p_stride, wl.qlat.float().numpy()[0],
                     ckv, g.softmax_scale, always_select_tail=True)
    mask = np.zeros(L, bool)
    for t in range(fk, L):
        p = (t - fk) // 4
        mask[t] = p >= len(pv) or bool(pv[p])
    assert len(pv) == 50 and mask[fk + 200:].all() and mask[fk + 200:].sum() == 3
    dense = O.dense_masked_attention(wl.qlat.float().numpy()[0], ckv, mask, g.softmax_scale)
    np.testing.assert_allclose(r["olat"], dense, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# projection front-end


def test_rms_norm_golden_and_closed_forms():
    g = load_kv("rms_norm.txt")
    x, gamma = g["x"][0], g["gamma"][0]
    np.testing.assert_allclose(O.rms_norm(x, gamma, 0.0), g["eps0"][0], rtol=1e-15)
    np.testing.assert_allclose(O.rms_norm(x, gamma, 0.5), g["eps05"][0], rtol=1e-15)
    rng = np.random.default_rng(16)
    v = rng.normal(size=(5, 33))
    gm = rng.normal(size=33)
    # constant row -> sign * gamma; positive scale invariance; unit mean square
    np.testing.assert_allclose(O.rms_norm(np.full(33, -2.5), gm, 0.0), -gm, rtol=1e-14)
    np.testing.assert_allclose(O.rms_norm(7.0 * v, gm, 0.0), O.rms_norm(v, gm, 0.0), rtol=1e-13)
    np.testing.assert_allclose((O.rms_norm(v, np.ones(33), 0.0) ** 2).mean(axis=1), 1.0,
                               rtol=1e-13)


def test_frontend_row_on_basis_vectors():
    # With x a scaled basis vector every projection picks one weight column, and with
    # q_absorb and wq_b the identity qlat and qidx are q_lora itself: each output is
    # fixed without retyping the composition.
    rng = np.random.default_rng(17)
    hidden, ql, kvl, ihd, Hi, H = 64, 96, 32, 16, 6, 3
    W = lambda n, k: rng.normal(size=(n, k))
    q_a, kv_a, wk, gate, wp = W(ql, hidden), W(kvl, hidden), W(ihd, hidden), W(ihd, hidden), W(Hi, hidden)
    gq, gkv = rng.normal(size=ql), rng.normal(size=kvl)
    eye = np.eye(ql)
    for j, sc in ((5, 1.5), (63, -0.25)):
        x = np.zeros(hidden)
        x[j] = sc
        out = O.frontend_row(x, q_a, gq, kv_a, gkv, wk, gate, wp, eye, eye, 1e-6, H, Hi)
        np.testing.assert_array_equal(out["w"], sc * wp[:, j])
        np.testing.assert_array_equal(out["k_raw"], O.bf16_round(sc * wk[:, j]))
        np.testing.assert_array_equal(out["gate"], O.bf16_round(sc * gate[:, j]))
        np.testing.assert_array_equal(out["ckv"], O.bf16_round(O.rms_norm(sc * kv_a[:, j], gkv, 1e-6)))
        ql_ref = O.bf16_round(O.rms_norm(sc * q_a[:, j], gq, 1e-6))
        np.testing.assert_array_equal(out["q_lora"], ql_ref)
        np.testing.assert_array_equal(out["qlat"], ql_ref.reshape(H, kvl))
        np.testing.assert_array_equal(out["qidx"], ql_ref.reshape(Hi, ihd))
    # the norms are not interchangeable, and q uses q_lora, not x (distinct widths)
    out = O.frontend_row(x, q_a, gq, kv_a, gkv, wk, gate, wp, eye, eye, 1e-6, H, Hi)
    assert out["q_lora"].shape == (ql,) and out["ckv"].shape == (kvl,)


# ---------------------------------------------------------------------------
# FP8 latent cache


def test_e4m3_golden():
    g = load_kv("fp8_e4m3.txt")
    for v, c in g["code"]:
        assert O.e4m3_round(v) == v
        assert int(O.e4m3_encode(np.array([v]))[0]) == int(c), v
        assert O.e4m3_decode(np.array([int(c)]))[0] == v
    for v, r in g["round"]:
        assert O.e4m3_round(v) == r, v
    for a, k in g["scale"]:
        assert int(O.fp8_scale_exponent(a)) == int(k), a
    assert int(O.fp8_scale_exponent(2.0 ** -130)) == -126


def test_e4m3_matches_library_codec():
    f8 = getattr(torch, "float8_e4m3fn", None)
    if f8 is None:
        pytest.skip("torch without float8_e4m3fn")
    codes = np.arange(256)
    lib = torch.from_numpy(codes.astype(np.uint8)).view(f8).float().numpy().astype(np.float64)
    mine = O.e4m3_decode(codes)
    np.testing.assert_array_equal(np.isnan(mine), np.isnan(lib))
    fin = ~np.isnan(mine)
    np.testing.assert_array_equal(mine[fin], lib[fin])
    np.testing.assert_array_equal(O.e4m3_encode(mine[fin]), codes[fin].astype(np.uint8))
    rng = np.random.default_rng(14)
    x = np.concatenate([rng.uniform(-448, 448, 20000), rng.normal(0, 1e-2, 20000),
                        rng.normal(0, 3e-3, 5000), mine[fin],
                        (mine[fin][1:] + mine[fin][:-1]) / 2]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    want = torch.from_numpy(x).to(f8)
    got = O.e4m3_encode(O.e4m3_round(x.astype(np.float64)))
    np.testing.assert_array_equal(got, want.view(torch.uint8).numpy())


def test_fp8_scale_and_quantize_properties():
    rng = np.random.default_rng(15)
    amax = np.abs(rng.normal(0, 1, 5000)) * np.exp2(rng.integers(-40, 40, 5000))
    k = O.fp8_scale_exponent(amax)
    assert (amax <= 448 * np.exp2(k.astype(np.float64))).all()
    assert ((k == -126) | (amax > 448 * np.exp2(k - 1.0))).all()
    x = O.bf16_round(rng.normal(0, 1, (40, 512)) * np.exp2(rng.integers(-6, 6, (40, 1))))
    x[3, 128:256] = 0.0  # an all-zero group
    codes, scales = O.quantize_latent_fp8(x)
    assert codes.dtype == np.uint8 and scales.shape == (40, 4)
    assert scales[3, 1] == 1.0 and (codes[3, 128:256] == 0).all()
    deq = O.dequantize_latent_fp8(codes, scales)
    # each element within half an E4M3 spacing (at its binade) of the input, times the scale
    g = np.abs(x).reshape(40, 4, 128).max(axis=2)
    assert (np.abs(deq.reshape(40, 4, 128)).max(axis=2) <= 448 * scales).all()
    rel = np.abs(deq - x) / np.maximum(np.abs(x), 2.0 ** -6 * np.repeat(scales, 128, axis=1))
    assert rel.max() <= 2.0 ** -4 + 1e-12
    assert (g <= 448 * scales).all()
    # E4M3 values times a power of two come back exactly
    back_codes, back_scales = O.quantize_latent_fp8(deq)
    np.testing.assert_array_equal(O.dequantize_latent_fp8(back_codes, back_scales), deq)


# ---------------------------------------------------------------------------
# decode-time append and geometry


def test_append_geometry_golden():
    g = load_kv("append_geom.txt")
    assert len(g["completed"]) == 8
    for v in g["completed"]:
        prev, new, fk, kp, lo, hi = (int(x) for x in v)
        assert O.pools_completed(prev, new, fk, kp) == range(lo, hi), v
    for v in g["maxctx"]:
        assert O.max_dsa_context(int(v[0]), int(v[1])) == int(v[2])
    np.testing.assert_array_equal(
        O.write_geom(g["geom_seq_lens"][0].astype(int), g["geom_row_seq"][0].astype(int)),
        g["geom_row_ctx"][0])


def test_pools_completed_partition_the_whole_pools():
    # Over any sequence of appends the completed ranges are disjoint, contiguous,
    # and together are exactly the pools whole at the final length.
    rng = np.random.default_rng(13)
    for _ in range(300):
        kp = int(rng.integers(1, 9))
        fk = int(rng.integers(0, 7))
        lens = np.cumsum(rng.integers(0, 6, size=int(rng.integers(1, 12))))
        seen = []
        prev = 0
        for L in lens:
            r = O.pools_completed(prev, int(L), fk, kp)
            assert r.start == (len(seen) if seen else 0) or len(r) == 0
            seen.extend(r)
            prev = int(L)
        P = max(0, (prev - fk) // kp)
        assert seen == list(range(P))


def test_store_then_incremental_compress_equals_one_shot():
    g = W.Geometry(index_kpool=4, index_heads=4, index_head_dim=32, index_topk=64, heads=2,
                   hidden=32, kv_lora_rank=32)
    wl = W.make_workload("t", 31, g, [61], invalid_per_seq=5)
    k = wl.k_raw.float().numpy()[0]
    gt = wl.gate.float().numpy()[0]
    v = wl.valid.numpy()[0]
    ln = (wl.ape.numpy(), wl.ln_w.float().numpy(), wl.ln_b.float().numpy(), g.eps)
    for fk in (0, 3):
        L0 = 17
        kc, gc, vc = np.zeros_like(k), np.zeros_like(gt), np.zeros_like(v)
        kc[:L0], gc[:L0], vc[:L0] = k[:L0], gt[:L0], v[:L0]
        keys = np.full((64, k.shape[1]), np.nan)
        pv = np.full(64, 7, dtype=np.uint8)
        O.compress_append(kc, gc, vc, *ln, fk, 4, 0, L0, keys, pv)
        L = L0
        for t in range(L0, 61):
            L = O.indexer_store(kc, gc, vc, L, k[t], gt[t], capacity=61)
            if not v[t]:
                vc[t] = 0  # the workload's own invalid tokens stay invalid
            O.compress_append(kc, gc, vc, *ln, fk, 4, L - 1, L, keys, pv)
        assert L == 61
        ref_k, ref_v, _ = O.kpool_compress(k, gt, v, *ln, fk, 4)
        P = ref_k.shape[0]
        np.testing.assert_array_equal(keys[:P], ref_k)
        np.testing.assert_array_equal(pv[:P], ref_v)
        assert np.isnan(keys[P:]).all() and (pv[P:] == 7).all()  # untouched
    # A full cache is left as it is.
    kc = np.zeros((3, 2))
    assert O.indexer_store(kc, kc.copy(), np.zeros(3), 3, [1, 1], [1, 1], capacity=3) == 3
    assert (kc == 0).all()


# ---------------------------------------------------------------------------
# sparse latent MLA


def test_attention_golden():
    g = load_kv("sparse_mla.txt")
    q = g["q"][0].reshape(1, 2)
    ckv = g["ckv"][0].reshape(-1, 2)
    ids = g["token_ids"][0].astype(int)
    A = g["o_absorb"][0].reshape(2, 2)
    olat, y, yb = O.sparse_mla_decode_row(q, ckv, ids, 1.0, A)
    np.testing.assert_allclose(olat[0], g["olat"][0], rtol=1e-15)
    np.testing.assert_allclose(y, g["y"][0], rtol=1e-14)
    np.testing.assert_array_equal(yb, g["y_bf16"][0])
    olat2, _, _ = O.sparse_mla_decode_row(q, g["ckv_half"][0].reshape(-1, 2), ids, 0.5)
    np.testing.assert_allclose(olat2[0], g["olat_half"][0], rtol=1e-15)
    dense = O.dense_masked_attention(q, ckv, [True, True, False], 1.0)
    np.testing.assert_allclose(dense[0], g["olat"][0], rtol=1e-15)


def test_attention_single_token_and_empty():
    rng = np.random.default_rng(12)
    q = rng.standard_normal((3, 16))
    ckv = rng.standard_normal((10, 16))
    olat, _, _ = O.sparse_mla_decode_row(q, ckv, [-1, 7, -1], 0.3)
    np.testing.assert_allclose(olat, np.tile(ckv[7], (3, 1)), rtol=1e-15)
    olat, y, yb = O.sparse_mla_decode_row(q, ckv, [-1, -1], 0.3, rng.standard_normal((5, 48)))
    assert not olat.any() and not y.any() and not yb.any()


def test_attention_permutation_invariance():
    rng = np.random.default_rng(13)
    q = rng.standard_normal((4, 32))
    ckv = rng.standard_normal((50, 32))
    ids = rng.choice(50, 20, replace=False)
    a, _, _ = O.sparse_mla_decode_row(q, ckv, ids, 0.2)
    b, _, _ = O.sparse_mla_decode_row(q, ckv, rng.permutation(ids), 0.2)
    np.testing.assert_allclose(a, b, rtol=1e-12)


def test_dense_equivalence_when_topk_covers_all_candidates():
    # With index_topk >= kpool * #candidates, sparse attention over the selected
    # tokens equals dense masked attention over the tokens of candidate pools.
    g = W.Geometry(index_kpool=4, index_heads=4, index_head_dim=32, index_topk=4 * 64,
                   heads=3, hidden=64, kv_lora_rank=32)
    wl = W.make_workload("t", 21, g, [203], invalid_per_seq=9)
    k = wl.k_raw.float().numpy()[0]
    keys, pv, _ = O.kpool_compress(k, wl.gate.float().numpy()[0], wl.valid.numpy()[0],
                                   wl.ape.numpy(), wl.ln_w.float().numpy(),
                                   wl.ln_b.float().numpy(), g.eps, 0, 4)
    ckv = wl.ckv.float().numpy()[0]
    r = O.decode_row(wl.qidx.float().numpy()[0], wl.w.numpy()[0], keys, pv, 203, 0, 4,
                     g.index_scale, g.index_topk, wl.p_stride, wl.qlat.float().numpy()[0],
                     ckv, g.softmax_scale)
    mask = np.zeros(203, bool)
    for p in np.nonzero(pv)[0]:
        mask[4 * p: 4 * p + 4] = True
    assert mask.sum() == 4 * pv.sum() and pv.sum() < 50
    dense = O.dense_masked_attention(wl.qlat.float().numpy()[0], ckv, mask, g.softmax_scale)
    np.testing.assert_allclose(r["olat"], dense, rtol=1e-12, atol=1e-13)


def test_absorption_equivalence():
    # absorbed latent attention == unabsorbed MLA that decompresses the latent
    # through kv_b_proj, for every head, to float64 rounding.
    rng = np.random.default_rng(14)
    H, nope, vd, kvl, ql, hidden, T = 3, 5, 4, 7, 6, 8, 9
    q_b = rng.standard_normal((H * nope, ql))
    kv_b = rng.standard_normal((H * (nope + vd), kvl))
    o_proj = rng.standard_normal((hidden, H * vd))
    q_lora = rng.standard_normal(ql)
    ckv = rng.standard_normal((T, kvl))
    scale = nope ** -0.5
    ref = O.mla_unabsorbed(q_lora, q_b, kv_b, o_proj, ckv, H, nope, vd, kvl, scale)
    qlat = (O.absorb_q(q_b, kv_b, H, nope, vd, kvl, ql) @ q_lora).reshape(H, kvl)
    A = O.absorb_o(o_proj, kv_b, H, nope, vd, kvl, hidden)
    _, y, _ = O.sparse_mla_decode_row(qlat, ckv, np.arange(T), scale, A)
    np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-12)


def test_absorb_golden():
    # absorb_q / absorb_o against values worked by hand from the build.rs index
    # expressions (tests/golden/absorb.txt): a K/V half swap, a transposed operand
    # or a head offset error changes them.
    G = load_kv("absorb.txt")
    q_b, kv_b, o_proj = (np.vstack(G[k]) for k in ("q_b", "kv_b", "o_proj"))
    qa = O.absorb_q(q_b, kv_b, heads=2, nope=2, vd=1, kvl=2, ql=2)
    oa = O.absorb_o(o_proj, kv_b, heads=2, nope=2, vd=1, kvl=2, hidden=2)
    np.testing.assert_array_equal(qa, np.vstack(G["q_absorb"]))
    np.testing.assert_array_equal(oa, np.vstack(G["o_absorb"]))
    # the unabsorbed form with the same weights distinguishes the halves too: one
    # latent row, so the softmax weight is 1 and y = o_proj . V_h(ckv) per head
    ckv = np.array([[1.0, 2.0]])
    y = O.mla_unabsorbed(np.array([1.0, 1.0]), q_b, kv_b, o_proj, ckv, 2, 2, 1, 2, 0.5)
    # V_0(ckv) = 0*1 + 3*2 = 6, V_1(ckv) = 2*1 - 2*2 = -2; y = o_proj . (6, -2)
    np.testing.assert_array_equal(y, [1 * 6 + 2 * -2, -1 * 6 + 3 * -2])


def test_unabsorbed_reduces_to_plain_attention():
    # kv_b halves = identity, o_proj = identity: MLA is plain attention with
    # keys = values = latent rows.
    rng = np.random.default_rng(15)
    H, d, T = 2, 6, 7
    kv_b = np.tile(np.vstack([np.eye(d), np.eye(d)]), (H, 1))
    q_b = rng.standard_normal((H * d, 4))
    q_lora = rng.standard_normal(4)
    ckv = rng.standard_normal((T, d))
    y = O.mla_unabsorbed(q_lora, q_b, kv_b, np.eye(H * d), ckv, H, d, d, d, 0.4)
    dense = O.dense_masked_attention((q_b @ q_lora).reshape(H, d), ckv, np.ones(T, bool), 0.4)
    np.testing.assert_allclose(y, dense.reshape(-1), rtol=1e-12)


# ---------------------------------------------------------------------------
# cache addressing


def test_paged_and_contiguous_views_agree():
    g = W.Geometry(index_kpool=4, index_heads=4, index_head_dim=32, index_topk=64,
                   heads=2, hidden=64, kv_lora_rank=32)
    lens = [100, 37, 64]
    a = W.make_workload("c", 31, g, lens, max_seq_len=128, direct_kpool=True)
    b = W.make_workload("p", 31, g, lens, block_size=16, max_seq_len=128, direct_kpool=True)
    for s, L in enumerate(lens):
        for name in ("k_raw", "gate", "ckv"):
            x = O.sequence_tokens(getattr(a, name).float().numpy(), s, L)
            y = O.sequence_tokens(getattr(b, name).float().numpy(), s, L,
                                  b.block_table.numpy(), 16)
            np.testing.assert_array_equal(x, y)
        np.testing.assert_array_equal(
            O.sequence_tokens(a.valid.numpy(), s, L),
            O.sequence_tokens(b.valid.numpy(), s, L, b.block_table.numpy(), 16))
        P = L // 4
        np.testing.assert_array_equal(
            O.sequence_pools(a.kpool_keys.float().numpy(), s, P),
            O.sequence_pools(b.kpool_keys.float().numpy(), s, P, b.block_table.numpy(), 4))
