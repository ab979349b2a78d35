"""Decode-time append and graph replay while the sequences grow: dsa_indexer_store ->
dsa_write_geom -> dsa_compress_append -> the step, captured once and replayed while
the sequences grow. Each step is checked against the oracle at the grown length,
the replayed graph against an eager twin bit for bit, and the incrementally built
pooled-key cache against a one-shot dsa_compress of the final caches bit for bit."""
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


CASES = [
    # name, seq_lens, block_size, first_key, steps, always_select_tail, graph layer's append
    # fused (the eager twin takes the other form, so the two forms are compared bit for bit)
    ("contig", [300, 517, 77], None, 0, 9, False, True),
    ("contig-fk3-tail", [300, 517, 77], None, 3, 9, True, False),
    ("paged-fk4-tail", [300, 517, 130], 64, 4, 9, True, True),
]


def _seq(wl, name, b):
    """Host logical [L, ...] rows of sequence b of a workload token cache (float64)."""
    t = getattr(wl, name)
    bt = None if wl.block_table is None else wl.block_table.numpy()
    raw = t.view(torch.int16).numpy() if t.dtype == torch.bfloat16 else t.numpy()
    rows = O.sequence_tokens(raw, b, int(wl.seq_lens[b]), bt, wl.block_size or 0)
    if t.dtype == torch.bfloat16:
        return torch.from_numpy(np.ascontiguousarray(rows)).view(torch.bfloat16).double().numpy()
    return rows


def _snapshot(layer):
    return {k: getattr(layer, k).clone() for k in ("scores", "pool_ids", "token_ids", "olat", "y",
                                                     "seq_lens", "row_ctx")}


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_append_graph_replay(case):
    name, lens, bs, fk, n, tail, fused = case
    g = W.Geometry(index_kpool=4, index_heads=32, index_head_dim=128, index_topk=256, heads=8,
                   hidden=256, first_key=fk, always_select_tail=tail)
    wl = W.make_workload(f"append-{name}", 41, g, lens, block_size=bs,
                         max_seq_len=576 if bs else None, invalid_per_seq=3)
    L0 = wl.seq_lens.astype(np.int64) - n
    graph_layer = DsaDecodeLayer(wl, keep_olat=True, decode_from=L0, fuse_append=fused)
    twin = DsaDecodeLayer(wl, keep_olat=True, decode_from=L0, fuse_append=not fused)
    for lay in (graph_layer, twin):
        lay.status.zero_()
        lay.compress()

    # Graph layer: step 0 eagerly, then one capture replayed for steps 1..n-1.
    got = []
    for i in range(n):
        graph_layer.stage(i)
        if i == 0:
            graph_layer.append_step()
        else:
            if graph_layer.append_graph is None:
                graph_layer.capture_append()
            graph_layer.append_graph.replay()
        torch.cuda.synchronize()
        got.append(_snapshot(graph_layer))
    assert int(graph_layer.status.item()) == 0

    # Oracle inputs: the workload's rows; appended tokens are marked valid.
    ape, lnw, lnb = wl.ape.numpy(), H.f(wl.ln_w), H.f(wl.ln_b)
    A = H.f(wl.o_absorb)
    seqs = {b: dict(k=_seq(wl, "k_raw", b), gate=_seq(wl, "gate", b),
                    valid=_seq(wl, "valid", b).copy(), ckv=_seq(wl, "ckv", b))
            for b in range(wl.batch)}
    for b in range(wl.batch):
        seqs[b]["valid"][int(L0[b]):] = 1
    bt = None if wl.block_table is None else wl.block_table.numpy()
    ppb = (wl.block_size or 0) // g.index_kpool
    sk = twin.sk
    kinds = {"gap": 0, "band": 0}
    for i in range(n):
        twin.stage(i)
        twin.append_step()
        torch.cuda.synchronize()
        assert int(twin.status.item()) == 0
        mine = _snapshot(twin)
        for k, v in mine.items():
            assert torch.equal(v, got[i][k]), f"step {i}: graph replay differs from eager in {k}"
        L = L0 + i + 1
        np.testing.assert_array_equal(mine["seq_lens"].cpu().numpy(), L)
        np.testing.assert_array_equal(mine["row_ctx"].cpu().numpy(), O.write_geom(L))
        scores = mine["scores"].cpu().numpy().astype(np.float64)
        ids = mine["pool_ids"].cpu().numpy()
        tok = mine["token_ids"].cpu().numpy()
        kp_dev = twin.kpool.float().cpu().numpy()
        pv_dev = twin.pool_valid.cpu().numpy()
        redo = {}
        for b in range(wl.batch):
            Lb = int(L[b])
            s = seqs[b]
            keys, pv, _ = O.kpool_compress(s["k"][:Lb], s["gate"][:Lb], s["valid"][:Lb], ape,
                                           lnw, lnb, g.eps, fk, g.index_kpool)
            P = keys.shape[0]
            gk = O.sequence_pools(kp_dev, b, P, bt, ppb).astype(np.float64)
            np.testing.assert_array_equal(O.sequence_pools(pv_dev, b, P, bt, ppb), pv)
            toks = fk + np.arange(P)[:, None] * g.index_kpool + np.arange(g.index_kpool)
            kn = O.bf16_round(O.layernorm_bias(s["k"][toks], lnw, lnb, g.eps))
            H.check_kpool(gk, keys, H.bf16_ulp(kn).max(axis=1), f"step {i} seq {b} kpool")
            ref_s = O.index_scores(H.f(wl.qidx[b]), wl.w[b].numpy().astype(np.float64), keys, pv,
                                   Lb, fk, g.index_kpool, g.index_scale, wl.p_stride)
            extra = H.score_input_bound(H.f(wl.qidx[b]), wl.w[b].numpy(), gk - keys,
                                        g.index_scale, wl.p_stride)
            H.check_scores(scores[b], ref_s, f"step {i} row {b}", extra=extra)
            np.testing.assert_array_equal(ids[b], O.topk_pools(scores[b], sk))
            kinds[H.check_selection(ids[b], ref_s, sk)] += 1
            ref_ids = O.topk_pools(ref_s, sk)
            if tail:
                ref_tok = O.expand_selection_tail(ref_ids, fk, g.index_kpool, g.index_topk, Lb)
            else:
                ref_tok = O.expand_selection(ref_ids, fk, g.index_kpool, g.out_width)
            o_, y_, _ = O.sparse_mla_decode_row(H.f(wl.qlat[b]), s["ckv"][:Lb], ref_tok,
                                                g.softmax_scale, A)
            if np.array_equal(ref_tok, tok[b]):
                H.check_attention(mine["olat"][b].cpu().numpy().reshape(1, -1),
                                  o_.reshape(1, -1), f"step {i} olat {b}")
                H.check_attention(mine["y"][b].float().cpu().numpy()[None], y_[None],
                                  f"step {i} y {b}")
            else:
                redo[b] = (ref_tok, o_, y_)
        if redo:  # selections that differ inside the tie band: attention on the oracle's ids
            for b, (t, _, _) in redo.items():
                twin.token_ids[b] = torch.from_numpy(t.astype(np.int32)).cuda()
            twin.attend()
            twin.project()
            torch.cuda.synchronize()
            for b, (_, o_, y_) in redo.items():
                H.check_attention(twin.olat[b].cpu().numpy().reshape(1, -1), o_.reshape(1, -1),
                                  f"step {i} olat {b} (oracle ids)")
                H.check_attention(twin.y[b].float().cpu().numpy()[None], y_[None],
                                  f"step {i} y {b} (oracle ids)")
    assert kinds["gap"] + kinds["band"] == n * wl.batch

    # The incrementally built pooled cache is what one dsa_compress of the final
    # caches writes, bit for bit.
    fresh_k = torch.zeros_like(twin.kpool)
    fresh_v = torch.zeros_like(twin.pool_valid)
    api.dsa_compress(twin.k_raw, twin.gate, twin.valid, twin.ape, twin.ln_w, twin.ln_b, g.eps,
                     twin.pg, fk, g.index_kpool, fresh_k, fresh_v, status=twin.status)
    torch.cuda.synchronize()
    for b in range(wl.batch):
        P = max(0, (int(wl.seq_lens[b]) - fk) // g.index_kpool)
        a = O.sequence_pools(twin.kpool.view(torch.int16).cpu().numpy(), b, P, bt, ppb)
        c = O.sequence_pools(fresh_k.view(torch.int16).cpu().numpy(), b, P, bt, ppb)
        np.testing.assert_array_equal(a, c, err_msg=f"seq {b} keys")
        np.testing.assert_array_equal(O.sequence_pools(twin.pool_valid.cpu().numpy(), b, P, bt, ppb),
                                      O.sequence_pools(fresh_v.cpu().numpy(), b, P, bt, ppb))
    assert torch.equal(graph_layer.kpool, twin.kpool)
    assert torch.equal(graph_layer.seq_lens, twin.seq_lens)


def test_indexer_store_rows_and_full_cache():
    """Rows land at the live length (contiguous and paged), the token is marked
    valid, the length grows by one; a full cache sets the status bit and stores
    nothing."""
    for bs in (None, 64):
        g = W.Geometry(index_kpool=4, index_heads=4, index_head_dim=64, index_topk=64, heads=2,
                       hidden=64)
        wl = W.make_workload("store", 5, g, [128, 70], block_size=bs, max_seq_len=128)
        lay = DsaDecodeLayer(wl, decode_from=[127, 60])
        k0, g0, v0, c0 = (lay.k_raw.clone(), lay.gate.clone(), lay.valid.clone(), lay.ckv.clone())
        lay.k_new.copy_(torch.randn_like(lay.k_new, dtype=torch.float32).to(torch.bfloat16))
        lay.gate_new.copy_(torch.randn_like(lay.gate_new, dtype=torch.float32).to(torch.bfloat16))
        lay.ckv_new.copy_(torch.randn_like(lay.ckv_new, dtype=torch.float32).to(torch.bfloat16))
        lay.status.zero_()
        api.dsa_indexer_store(lay.k_new, lay.gate_new, lay.pg, lay.seq_lens, lay.k_raw, lay.gate,
                              lay.valid, lay.ckv_new, lay.ckv, lay.status)
        torch.cuda.synchronize()
        assert lay.seq_lens.tolist() == [128, 61] and int(lay.status.item()) == 0
        for b, t in ((0, 127), (1, 60)):
            row = int(lay._token_rows(b, t, t + 1)[0])
            assert torch.equal(lay.k_raw.view(-1, 64)[row], lay.k_new[b])
            assert torch.equal(lay.gate.view(-1, 64)[row], lay.gate_new[b])
            assert torch.equal(lay.ckv.view(-1, 512)[row], lay.ckv_new[b])
            assert int(lay.valid.view(-1)[row]) == 1
            for full, before in ((lay.k_raw, k0), (lay.gate, g0), (lay.valid, v0), (lay.ckv, c0)):
                w = full.shape[-1] if full.dim() == 3 else 1
                diff = (full.view(-1, w) != before.view(-1, w)).any(dim=1).nonzero().flatten()
                assert set(diff.tolist()) <= {int(lay._token_rows(0, 127, 128)[0]),
                                              int(lay._token_rows(1, 60, 61)[0])}
        # Sequence 0 is now full: a second store leaves it and flags the status.
        k1 = lay.k_raw.clone()
        api.dsa_indexer_store(lay.k_new, lay.gate_new, lay.pg, lay.seq_lens, lay.k_raw, lay.gate,
                              lay.valid, None, None, lay.status)
        torch.cuda.synchronize()
        assert lay.seq_lens.tolist() == [128, 62]
        assert int(lay.status.item()) == 8  # DSA_STATUS_CACHE_FULL
        row = int(lay._token_rows(1, 61, 62)[0])
        changed = (lay.k_raw.view(-1, 64) != k1.view(-1, 64)).any(dim=1).nonzero().flatten()
        assert set(changed.tolist()) <= {row}


def test_write_geom_and_compress_append_ranges():
    """write_geom maps rows to their sequence's live length (bad indices flagged);
    compress_append with several new tokens writes exactly the completed pools."""
    seq_lens = torch.tensor([5, 9, 2], dtype=torch.int32, device="cuda")
    row_seq = torch.tensor([2, 0, 0, 1, 3], dtype=torch.int32, device="cuda")
    row_ctx = torch.full((5,), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.dsa_write_geom(seq_lens, row_seq, row_ctx, status)
    torch.cuda.synchronize()
    assert row_ctx.tolist() == [2, 5, 5, 9, 0] and int(status.item()) == 1
    assert O.write_geom([5, 9, 2], [2, 0, 0, 1]).tolist() == [2, 5, 5, 9]

    g = W.Geometry(index_kpool=4, index_heads=4, index_head_dim=128, index_topk=64, heads=2,
                   hidden=64, first_key=1)
    wl = W.make_workload("append-range", 6, g, [200, 57, 13], max_seq_len=200)
    full = DsaDecodeLayer(wl)
    full.compress()
    lay = DsaDecodeLayer(wl)
    lay.kpool.fill_(7)
    lay.pool_valid.fill_(9)
    for new, prev in ((11, [189, 46, 2]),):
        api.dsa_compress_append(lay.k_raw, lay.gate, lay.valid, lay.ape, lay.ln_w, lay.ln_b,
                                g.eps, lay.pg, 1, 4, new, lay.kpool, lay.pool_valid,
                                status=lay.status)
        torch.cuda.synchronize()
        for b in range(3):
            rng = O.pools_completed(prev[b], int(wl.seq_lens[b]), 1, 4)
            pc = wl.max_seq_len // 4
            got_k = lay.kpool.view(3, pc, 128)[b]
            got_v = lay.pool_valid.view(3, pc)[b]
            ref_k = full.kpool.view(3, pc, 128)[b]
            ref_v = full.pool_valid.view(3, pc)[b]
            inside = torch.zeros(pc, dtype=torch.bool, device="cuda")
            inside[rng.start:rng.stop] = True
            assert torch.equal(got_k[inside], ref_k[inside]), f"seq {b}"
            assert torch.equal(got_v[inside], ref_v[inside])
            assert (got_k[~inside].view(torch.int16) == torch.tensor(7, dtype=torch.bfloat16,
                                                                      device="cuda").view(torch.int16)).all()
            assert (got_v[~inside] == 9).all()


def test_decode_append_full_cache_matches_separate_calls():
    """At the capacity the fused append flags the status, stores nothing, keeps the
    length and writes it to row_ctx, as the three separate calls do."""
    g = W.Geometry(index_kpool=4, index_heads=4, index_head_dim=128, index_topk=64, heads=2,
                   hidden=64)
    wl = W.make_workload("append-full", 8, g, [128, 100], max_seq_len=128)
    out = []
    for fused in (True, False):
        lay = DsaDecodeLayer(wl, decode_from=[127, 97], fuse_append=fused)
        lay.compress()
        lay.stage(0)
        lay.status.zero_()
        for _ in range(3):  # sequence 0 fills at the first append
            lay.append()
        torch.cuda.synchronize()
        out.append((lay.seq_lens.clone(), lay.row_ctx.clone(), int(lay.status.item()),
                    lay.k_raw.clone(), lay.kpool.clone(), lay.pool_valid.clone(), lay.valid.clone()))
    (a, b) = out
    assert a[0].tolist() == [128, 100] and a[1].tolist() == [128, 100] and a[2] == 8
    assert b[2] == a[2]
    for x, y in zip(a[:2] + a[3:], b[:2] + b[3:]):
        assert torch.equal(x, y)


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "three-call"])
def test_append_bad_block_entry_sets_status(fused):
    """A block-table entry outside [0, num_blocks) at the append position: the token is
    not stored, the length stays, DSA_STATUS_BAD_BLOCK is set; other sequences append."""
    g = W.Geometry(index_kpool=4, index_heads=4, index_head_dim=128, index_topk=64, heads=2,
                   hidden=64)
    wl = W.make_workload("append-badblock", 9, g, [300, 200], block_size=64, max_seq_len=320)
    lay = DsaDecodeLayer(wl, decode_from=[290, 190], fuse_append=fused)
    lay.compress()
    lay.stage(0)
    blk = 290 // 64
    lay.block_table[0, blk] = -1
    k0 = lay.k_raw.clone()
    lay.status.zero_()
    lay.append()
    torch.cuda.synchronize()
    assert int(lay.status.item()) & 2
    assert lay.seq_lens.tolist() == [290, 191]
    row = int(lay._token_rows(1, 190, 191)[0])
    changed = (lay.k_raw.view(-1, 128) != k0.view(-1, 128)).any(dim=1).nonzero().flatten()
    assert set(changed.tolist()) <= {row}
    assert torch.equal(lay.k_raw.view(-1, 128)[row], lay.k_new[1])
