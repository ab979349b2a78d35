"""FP8 latent cache: dsa_quantize_latent against the oracle's encoder (codes and
scales bit for bit), and dsa_sparse_mla_decode_fp8 against the oracle on the
decoded cache and, bit for bit, against dsa_sparse_mla_decode run on that decoded
cache stored as bf16 (decoding is exact in bf16, and the attention arithmetic after
the gather is shared)."""
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


@pytest.fixture(autouse=True)
def _mma_kernel():
    with api.mla_kernel("mma"):  # the bf16 twin runs the same split kernel
        yield


def _host_quant(x_bf16: torch.Tensor):
    rows = x_bf16.float().numpy().reshape(-1, x_bf16.shape[-1]).astype(np.float64)
    return O.quantize_latent_fp8(rows)


def test_quantize_latent_parity():
    rng = np.random.default_rng(21)
    x = rng.normal(0, 1, (300, 512)) * np.exp2(rng.integers(-20, 20, (300, 1)))
    x[0] = 0.0                                   # all-zero row
    x[1, :128] = 0.0                             # one all-zero group
    x[2, 5] = -0.0
    x[3] = rng.normal(0, 1, 512) * 2.0 ** -128   # tiny: the -126 clamp
    x[4, 7] = 448.0 * 2 ** 10                    # a group maximum on a boundary
    x[5] = np.where(np.arange(512) % 2, 1.0625, -1.1875)  # E4M3 ties
    x[6] = rng.normal(0, 1e30, 512)
    xb = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    codes = torch.full((300, 512), 0xAA, dtype=torch.uint8, device="cuda")
    scales = torch.full((300, 4), -1.0, dtype=torch.float32, device="cuda")
    api.dsa_quantize_latent(xb.cuda(), codes, scales)
    torch.cuda.synchronize()
    want_c, want_s = _host_quant(xb)
    np.testing.assert_array_equal(codes.cpu().numpy(), want_c)
    np.testing.assert_array_equal(scales.cpu().numpy().astype(np.float64), want_s)


FP8_CASES = [
    # name, heads, hidden, lens, block_size, out_width, o_absorb
    ("h4-tiny", 4, 1024, [2048], None, 256, True),
    ("h64-b1", 64, 512, [5000], None, 2048, True),
    ("h64-b3-paged", 64, 256, [3000, 700, 4097], 64, 512, True),
    ("h20-ragged", 20, 128, [999, 400], None, 300, True),
    ("h16-olat-only", 16, 0, [1500, 1500], None, 700, False),
    ("h96-two-groups", 96, 64, [800], None, 200, True),
    ("h64-r40-two-chunks", 64, 128, [3000] * 40, None, 1024, False),
]


@pytest.mark.parametrize("form", ["mma", "tcgen05"])
@pytest.mark.parametrize("case", FP8_CASES, ids=[c[0] for c in FP8_CASES])
def test_fp8_attention_parity(case, form):
    """Both attention kernels on the FP8 cache (the tcgen05 one, 64 heads, decodes in its
    gather warps) equal the same kernel on the decoded cache stored as bf16, bit for bit."""
    name, heads, hidden, lens, bs, ow, with_o = case
    if form == "tcgen05" and heads != 64:
        pytest.skip("the tcgen05 attention serves 64 heads")
    with api.mla_kernel(form):
        _fp8_attention_parity(case)


def _fp8_attention_parity(case):
    name, heads, hidden, lens, bs, ow, with_o = case
    g = W.Geometry(index_kpool=4, index_heads=32, index_head_dim=128, index_topk=ow, heads=heads,
                   hidden=max(hidden, 32))
    wl = W.make_workload(name, 310, g, lens, block_size=bs, with_raw=False, with_o_absorb=with_o)
    layer = DsaDecodeLayer(wl, with_o_absorb=with_o, keep_olat=True, latent_fp8=True)
    torch.cuda.synchronize()
    # The device cache's codes and scales are the oracle's encoding of the bf16 cache.
    want_c, want_s = _host_quant(wl.ckv)
    np.testing.assert_array_equal(layer.ckv_codes.cpu().numpy().reshape(-1, 512), want_c)
    np.testing.assert_array_equal(layer.ckv_scales.cpu().numpy().reshape(-1, 4), want_s)
    deq = O.dequantize_latent_fp8(want_c, want_s)  # exact bf16 values
    deq_dev = torch.from_numpy(deq.astype(np.float32)).to(torch.bfloat16).view(
        wl.ckv.shape).cuda()
    assert np.array_equal(deq_dev.float().cpu().numpy().reshape(-1, 512), deq)

    rng = np.random.default_rng(heads + ow + 7)
    ids = np.full((wl.rows, ow), -1, dtype=np.int32)
    for r in range(wl.rows):
        L = int(wl.seq_lens[int(wl.row_seq[r])])
        if r == 1:
            continue  # an empty selection
        k = int(rng.integers(1, min(ow, L) + 1))
        pos = np.sort(rng.choice(ow, k, replace=False))
        ids[r, pos] = rng.choice(L, k, replace=False)
    tok = torch.from_numpy(ids).cuda()
    outs = []
    for fp8 in (True, False):
        olat = H.Guarded((wl.rows, heads, 512), torch.float32, 555.0)
        y = H.Guarded((wl.rows, g.hidden), torch.bfloat16, 3.0) if with_o else None
        if fp8:
            api.dsa_sparse_mla_decode_fp8(layer.qlat, layer.row_seq, layer.ckv_codes,
                                          layer.ckv_scales, layer.pg, tok, g.softmax_scale,
                                          layer.o_absorb, None if y is None else y.t, olat.t,
                                          layer.status, layer.fused_workspace())
        else:
            api.dsa_sparse_mla_decode(layer.qlat, layer.row_seq, deq_dev, layer.pg, tok,
                                      g.softmax_scale, layer.o_absorb, None if y is None else y.t,
                                      olat.t, layer.status, layer.fused_workspace())
        torch.cuda.synchronize()
        olat.check()
        if y is not None:
            y.check()
        outs.append((olat.t.clone(), None if y is None else y.t.clone()))
    assert int(layer.status.item()) == 0
    assert torch.equal(outs[0][0], outs[1][0]), "FP8 olat differs from bf16 on the decoded cache"
    if with_o:
        assert torch.equal(outs[0][1], outs[1][1])

    bt = None if wl.block_table is None else wl.block_table.numpy()
    deq_cache = deq.reshape(tuple(wl.ckv.shape))
    A = H.f(wl.o_absorb) if with_o else None
    ro, ry = [], []
    for r in range(wl.rows):
        b = int(wl.row_seq[r])
        ckv_seq = O.sequence_tokens(deq_cache, b, int(wl.seq_lens[b]), bt, wl.block_size or 0)
        o_, y_, _ = O.sparse_mla_decode_row(H.f(wl.qlat[r]), ckv_seq, ids[r], g.softmax_scale, A)
        ro.append(o_.reshape(-1))
        if with_o:
            ry.append(y_)
    H.check_attention(outs[0][0].cpu().numpy().reshape(wl.rows, -1), np.array(ro), f"{name} olat")
    if with_o:
        H.check_attention(outs[0][1].float().cpu().numpy(), np.array(ry), f"{name} y")


def _paged_small():
    return W.make_workload("paged-small", 5, W.Geometry(**W.GLM53), [3000, 5000, 700, 4096],
                           block_size=64, max_seq_len=5120, invalid_per_seq=7)


@pytest.mark.parametrize("make", [W.tiny, _paged_small], ids=["tiny", "paged"])
def test_fp8_decode_step_equals_bf16_step_on_decoded_cache(make):
    """The whole step with the FP8 cache equals the bf16 step over the decoded cache,
    bit for bit (scores and selection do not read the latent cache)."""
    wl = make()
    fp8 = DsaDecodeLayer(wl, keep_olat=True, latent_fp8=True)
    ref = DsaDecodeLayer(wl, keep_olat=True)
    c, sc = _host_quant(wl.ckv)
    ref.ckv.copy_(torch.from_numpy(O.dequantize_latent_fp8(c, sc).astype(np.float32))
                  .to(torch.bfloat16).view(wl.ckv.shape))
    for lay in (fp8, ref):
        lay.compress()
        lay.step()
    torch.cuda.synchronize()
    assert int(fp8.status.item()) == 0
    assert torch.equal(fp8.pool_ids, ref.pool_ids)
    assert torch.equal(fp8.olat, ref.olat)
    assert torch.equal(fp8.y, ref.y)


@pytest.mark.parametrize("paged", [False, True], ids=["contig", "paged"])
def test_fp8_decode_append(paged):
    """dsa_decode_append_fp8 grows the FP8 cache one token per sequence (eager, then a
    replayed graph). Afterwards every cache row's codes and scales equal the oracle's
    encoding of the workload's bf16 row, and the last step equals, bit for bit, the
    step of a layer whose FP8 cache was encoded in one piece at the full length."""
    g = W.Geometry(index_kpool=4, index_heads=32, index_head_dim=128, index_topk=256, heads=8,
                   hidden=256)
    n = 7
    wl = W.make_workload(f"fp8-append-{int(paged)}", 43, g, [300, 517, 130],
                         block_size=64 if paged else None, max_seq_len=576 if paged else None,
                         invalid_per_seq=3)
    L0 = wl.seq_lens.astype(np.int64) - n
    grow = DsaDecodeLayer(wl, keep_olat=True, decode_from=L0, latent_fp8=True)
    grow.compress()
    for i in range(n):
        grow.stage(i)
        if i == 0:
            grow.append_step()
        else:
            if grow.append_graph is None:
                grow.capture_append()
            grow.append_graph.replay()
    torch.cuda.synchronize()
    assert int(grow.status.item()) == 0
    np.testing.assert_array_equal(grow.seq_lens.cpu().numpy(), wl.seq_lens)

    codes = grow.ckv_codes.view(-1, g.kv_lora_rank).cpu().numpy()
    scales = grow.ckv_scales.view(-1, g.kv_lora_rank // 128).cpu().numpy()
    src = wl.ckv.reshape(-1, g.kv_lora_rank)
    for b in range(wl.batch):
        rows = grow._token_rows(b, 0, int(wl.seq_lens[b]))
        c, sc = _host_quant(src[torch.from_numpy(rows)])
        np.testing.assert_array_equal(codes[rows], c, err_msg=f"seq {b} codes")
        np.testing.assert_array_equal(scales[rows], sc, err_msg=f"seq {b} scales")

    # The one-piece twin: appended tokens count as valid, as the append marks them.
    whole = DsaDecodeLayer(wl, keep_olat=True, latent_fp8=True)
    for b in range(wl.batch):
        rows = torch.from_numpy(whole._token_rows(b, int(L0[b]), int(wl.seq_lens[b])))
        whole.valid.view(-1)[rows.to(whole.valid.device)] = 1
    whole.compress()
    whole.step()
    torch.cuda.synchronize()
    assert int(whole.status.item()) == 0
    assert torch.equal(grow.kpool, whole.kpool)
    for k in ("scores", "pool_ids", "token_ids", "olat", "y"):
        assert torch.equal(getattr(grow, k), getattr(whole, k)), k


def test_fp8_decode_append_rejects_bad_rank():
    """kv_lora_rank must be a multiple of 128 for the FP8 cache (no launch)."""
    g = W.Geometry(index_kpool=4, index_heads=32, index_head_dim=128, index_topk=256, heads=8,
                   hidden=256)
    wl = W.make_workload("fp8-append-bad", 44, g, [300], invalid_per_seq=0)
    lay = DsaDecodeLayer(wl, decode_from=[290], latent_fp8=True)
    ckv_new = torch.zeros((1, 200), dtype=torch.bfloat16, device="cuda")
    codes = torch.zeros((wl.max_seq_len, 200), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((wl.max_seq_len, 1), dtype=torch.float32, device="cuda")
    with pytest.raises(Exception, match="multiple of"):
        api.dsa_decode_append_fp8(lay.k_new, lay.gate_new, ckv_new, lay.ape, lay.ln_w, lay.ln_b,
                                  g.eps, lay.pg, lay.seq_lens, g.first_key, g.index_kpool,
                                  lay.k_raw, lay.gate, lay.valid, codes, scales, lay.kpool,
                                  lay.pool_valid, status=lay.status)
