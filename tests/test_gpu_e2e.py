"""End-to-end parity of the decode step (compress -> score -> select -> expand ->
sparse MLA) on the named workloads, at full size, in the launch configuration the
benchmark times. Oracle rows are computed one by one on the host."""
import numpy as np
import pytest
import torch

from oracle import dsa_oracle as O
from sparse_attention_decode_kpool_gb300 import api, workloads as W
from sparse_attention_decode_kpool_gb300.pipeline import DsaDecodeLayer
from tests import _harness as H

pytestmark = pytest.mark.gpu


def _run(wl, rows_to_check, with_o_absorb=True):
    g = wl.geom
    layer = DsaDecodeLayer(wl, with_o_absorb=with_o_absorb, keep_olat=True)
    layer.status.zero_()
    layer.compress()
    layer.step()
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    oq = H.OracleSeq(wl)
    kp = layer.kpool.float().cpu().numpy()
    pv = layer.pool_valid.cpu().numpy()
    scores = layer.scores.cpu().numpy().astype(np.float64)
    ids = layer.pool_ids.cpu().numpy()
    tok = layer.token_ids.cpu().numpy()
    olat = layer.olat.cpu().numpy()
    y = layer.y.float().cpu().numpy() if layer.y is not None else None
    A = H.f(wl.o_absorb) if with_o_absorb else None
    bt = None if wl.block_table is None else wl.block_table.numpy()
    ppb = (wl.block_size or 0) // g.index_kpool
    kinds = {"gap": 0, "band": 0}
    dkeys = {}
    redo_rows = []
    for r in rows_to_check:
        b = int(wl.row_seq[r])
        keys, rpv, _ = oq.pools(b)
        P = keys.shape[0]
        if b not in dkeys:
            np.testing.assert_array_equal(O.sequence_pools(pv, b, P, bt, ppb), rpv)
            gk = O.sequence_pools(kp, b, P, bt, ppb)
            H.check_kpool(gk, keys, oq.kn_ulp(b), f"{wl.name} seq {b}")
            dkeys[b] = gk - keys
        ref_s = oq.scores(r, wl.p_stride)
        # The GPU scored its own pooled keys: widen the bound by what their (checked)
        # difference from the oracle's keys can move each score.
        extra = H.score_input_bound(H.f(wl.qidx[r]), wl.w[r].numpy(), dkeys[b], g.index_scale,
                                    wl.p_stride)
        H.check_scores(scores[r], ref_s, f"{wl.name} row {r}", extra=extra)
        # S1: the GPU's selection is the exact top-k of its own score row.
        np.testing.assert_array_equal(ids[r], O.topk_pools(scores[r], layer.sk))
        # S3: against the oracle's scores, exact outside the near-tie band.
        kinds[H.check_selection(ids[r], ref_s, layer.sk)] += 1
        ref_ids = O.topk_pools(ref_s, layer.sk)
        if g.always_select_tail:
            ref_tok = O.expand_selection_tail(ref_ids, g.first_key, g.index_kpool, g.index_topk,
                                              int(wl.row_ctx[r]))
        else:
            ref_tok = O.expand_selection(ref_ids, g.first_key, g.index_kpool, g.out_width)
        assert ref_tok.shape == (g.out_width,)
        if np.array_equal(ref_tok, tok[r]):
            o_, y_, _ = O.sparse_mla_decode_row(H.f(wl.qlat[r]), oq.ckv(b), ref_tok,
                                                g.softmax_scale, A)
            H.check_attention(olat[r].reshape(1, -1), o_.reshape(1, -1), f"olat row {r}")
            if A is not None:
                H.check_attention(y[r][None], y_[None], f"y row {r}")
        else:
            redo_rows.append((r, ref_tok))
    # Rows whose selection differs inside the tie band: attention parity on the
    # oracle's token ids (stage isolation).
    if redo_rows:
        tok_ref = layer.token_ids.clone()
        for r, t in redo_rows:
            tok_ref[r] = torch.from_numpy(t.astype(np.int32)).cuda()
        layer.token_ids.copy_(tok_ref)
        layer.attend()
        torch.cuda.synchronize()
        olat = layer.olat.cpu().numpy()
        y = layer.y.float().cpu().numpy() if layer.y is not None else None
        for r, t in redo_rows:
            b = int(wl.row_seq[r])
            o_, y_, _ = O.sparse_mla_decode_row(H.f(wl.qlat[r]), oq.ckv(b), t, g.softmax_scale, A)
            H.check_attention(olat[r].reshape(1, -1), o_.reshape(1, -1), f"olat row {r} (oracle ids)")
            if A is not None:
                H.check_attention(y[r][None], y_[None], f"y row {r} (oracle ids)")
    return kinds


def test_tiny_end_to_end():
    wl = W.tiny()
    kinds = _run(wl, range(wl.rows))
    assert sum(kinds.values()) == 1


def test_tiny_graph_replay_matches_eager():
    wl = W.tiny()
    layer = DsaDecodeLayer(wl)
    layer.compress()
    layer.step()
    torch.cuda.synchronize()
    y0 = layer.y.clone()
    ids0 = layer.pool_ids.clone()
    layer.capture()
    layer.y.zero_()
    layer.pool_ids.zero_()
    layer.replay()
    torch.cuda.synchronize()
    assert torch.equal(layer.pool_ids, ids0)
    assert torch.equal(layer.y, y0)


def test_second_step_input_buffer_matches():
    # use_step_inputs: a graph captured over a second input buffer (holding the same
    # inputs) gives the same outputs bit for bit, and writing the first buffer does
    # not reach it.
    wl = W.tiny()
    layer = DsaDecodeLayer(wl)
    layer.compress()
    layer.step()
    torch.cuda.synchronize()
    y0, tok0 = layer.y.clone(), layer.token_ids.clone()
    first = layer.step_inputs
    second = first.clone()
    layer.use_step_inputs(second)
    layer.capture()
    first.zero_()  # the captured graph reads the second buffer only
    layer.y.zero_()
    layer.replay()
    torch.cuda.synchronize()
    assert torch.equal(layer.y, y0) and torch.equal(layer.token_ids, tok0)
    with pytest.raises(ValueError):
        layer.use_step_inputs(second[:-1])


def _tail_workload(paged: bool):
    # always_select_tail on lengths that leave every remainder mod kpool past
    # first_key, plus a sequence with no whole pool (6 tokens) and one that ends
    # before first_key (2 tokens: empty selection). The paged layout wants
    # first_key on a pool boundary, so it takes 4; the contiguous one takes 3.
    fk = 4 if paged else 3
    g = W.Geometry(**W.GLM53, first_key=fk, always_select_tail=True)
    return W.make_workload(f"tail-{'paged' if paged else 'contig'}-fk{fk}", 11, g,
                           [4097, 5002, 1023, 6, 2050, 9000, 2],
                           block_size=64 if paged else None, max_seq_len=9024,
                           invalid_per_seq=5)


@pytest.mark.parametrize("paged", [False, True], ids=["contig", "paged"])
@pytest.mark.parametrize("fuse", [True, False], ids=["fused", "two-call"])
def test_always_select_tail_end_to_end(fuse, paged, monkeypatch):
    wl = _tail_workload(paged)
    assert wl.geom.out_width == 2048 + 3
    orig = DsaDecodeLayer.__init__

    def init(self, *a, **k):
        k["fuse_expand"] = fuse
        orig(self, *a, **k)

    monkeypatch.setattr(DsaDecodeLayer, "__init__", init)
    _run(wl, range(wl.rows))


@pytest.mark.slow
def test_single_32k_end_to_end():
    wl = W.single_32k()
    _run(wl, [0])


@pytest.mark.slow
def test_paged_batch_end_to_end_sampled():
    wl = W.paged_batch()
    _run(wl, [0, 1, 17, 40, 63])


@pytest.mark.slow
def test_long_262k_end_to_end_sampled():
    wl = W.long_262k()
    _run(wl, [0, 5])


@pytest.mark.slow
def test_prefill_chunk_sampled_rows():
    wl = W.prefill_chunk(with_o_absorb=False)
    _run(wl, [0, 1, 2, 1000, 2047, 3333, 4094, 4095], with_o_absorb=False)
