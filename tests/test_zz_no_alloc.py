"""The no-allocation variant of the sparse latent MLA entry point.

dsa_sparse_mla_decode_noalloc serves callers that cannot allocate device memory
(a host framework that owns every allocation, or a loop that must never call
cudaMalloc/cudaFree because they can synchronise the device): it takes no
workspace and uses the library's fixed scratch array instead. Here it must give
the same results as dsa_sparse_mla_decode with a caller-provided workspace, on
two calls in a row with different problems, so that the previous call's scratch
contents cannot leak into the next one. This file is collected last on purpose:
it runs both alone in a fresh process and after every other test.
"""
import numpy as np
import pytest
import torch

from sparse_attention_decode_kpool_gb300 import api, workloads as W
from sparse_attention_decode_kpool_gb300._lib import DSA_ERR_UNSUPPORTED, DsaError
from sparse_attention_decode_kpool_gb300.pipeline import DsaDecodeLayer
from tests import _harness as H

pytestmark = pytest.mark.gpu


def _problem(seed, rows, heads, lens, ow, block_size=None):
    g = W.Geometry(index_kpool=4, index_heads=8, index_head_dim=128, index_topk=ow,
                   heads=heads, hidden=512)
    wl = W.make_workload(f"noalloc-{seed}", seed, g, lens, block_size=block_size,
                         with_raw=False)
    layer = DsaDecodeLayer(wl, keep_olat=True)
    rng = np.random.default_rng(seed)
    ids = np.full((wl.rows, ow), -1, dtype=np.int32)
    for r in range(wl.rows):
        L = int(wl.seq_lens[r])
        k = int(rng.integers(1, min(ow, L) + 1))
        ids[r, :k] = np.sort(rng.choice(L, k, replace=False))
    layer.token_ids.copy_(torch.from_numpy(ids))
    return wl, layer


def _with_workspace(wl, layer):
    y = torch.full_like(layer.y, 7.0)
    olat = torch.full_like(layer.olat, 7.0)
    api.dsa_sparse_mla_decode(layer.qlat, layer.row_seq, layer.ckv, layer.pg, layer.token_ids,
                              wl.geom.softmax_scale, layer.o_absorb, y, olat,
                              layer.status, layer.fused_workspace())
    torch.cuda.synchronize()
    return y, olat


def _no_alloc(wl, layer):
    y = torch.full_like(layer.y, 9.0)
    olat = torch.full_like(layer.olat, 9.0)
    api.dsa_sparse_mla_decode_noalloc(layer.qlat, layer.row_seq, layer.ckv, layer.pg,
                                      layer.token_ids, wl.geom.softmax_scale, layer.o_absorb,
                                      y, olat, layer.status)
    torch.cuda.synchronize()
    return y, olat


def _same(got, ref, what):
    """The two entry points run the same kernels with the same launch plan on the
    same inputs, so their results must agree bit for bit (a scratch value left by an
    earlier call could hide inside a tolerance); the oracle-tolerance check is kept
    as a readable report if they do not."""
    (gy, go), (ry, ro) = got, ref
    if not (torch.equal(gy, ry) and torch.equal(go, ro)):
        H.check_attention(gy.float().cpu().numpy(), ry.float().cpu().numpy(), f"y ({what})")
        H.check_attention(go.cpu().numpy().reshape(go.shape[0], -1),
                          ro.cpu().numpy().reshape(ro.shape[0], -1), f"olat ({what})")
        pytest.fail(f"{what}: no-alloc result differs from the workspace entry point's")


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    assert torch.cuda.is_available()
    # Different problems back to back: many splits per row (scratch holds split
    # partials and GEMV partials), then a paged batch with other sizes, then the
    # first problem again after the second has overwritten the scratch.
    first = _problem(11, rows=4, heads=64, lens=[3000, 2500, 4000, 1800], ow=1024)
    second = _problem(12, rows=3, heads=16, lens=[700, 900, 650], ow=256, block_size=64)
    got = [_no_alloc(*first), _no_alloc(*second), _no_alloc(*first)]
    ref = [_with_workspace(*first), _with_workspace(*second)]
    _same(got[0], ref[0], "first problem")
    _same(got[1], ref[1], "second problem")
    _same(got[2], ref[0], "first problem again, after the second")
    assert int(first[1].status.item()) == 0 and int(second[1].status.item()) == 0


def test_noalloc_tensor_core_kernel_on_shared_scratch():
    # The tcgen05 split kernel (64 heads, forced) writes its per-split partials into
    # the shared array; run it after a different problem has left its own partials
    # there, and twice in a row.
    other = _problem(14, rows=5, heads=32, lens=[2000, 1500, 2500, 1200, 900], ow=512)
    tc = _problem(15, rows=4, heads=64, lens=[3000, 2600, 2048, 4000], ow=1024)
    with api.mla_kernel("tcgen05"):
        _no_alloc(*other)
        got = [_no_alloc(*tc), _no_alloc(*tc)]
        ref = _with_workspace(*tc)
    _same(got[0], ref, "tcgen05 kernel, after another problem")
    _same(got[1], ref, "tcgen05 kernel, second call")
    assert int(tc[1].status.item()) == 0


def test_noalloc_refuses_problems_larger_than_its_scratch():
    wl, layer = _problem(13, rows=2, heads=8, lens=[500, 500], ow=128)
    need = api.dsa_sparse_mla_decode_workspace(4096, 64, 2048, 4096, True)
    assert need > (48 << 20)
    big_q = torch.zeros((4096, 64, 512), dtype=torch.bfloat16, device="cuda")
    big_tok = torch.full((4096, 2048), -1, dtype=torch.int32, device="cuda")
    row_seq = torch.zeros(4096, dtype=torch.int32, device="cuda")
    oabs = torch.zeros((4096, 64 * 512), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((4096, 4096), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(DsaError) as e:
        api.dsa_sparse_mla_decode_noalloc(big_q, row_seq, layer.ckv, layer.pg, big_tok,
                                          0.0625, oabs, y)
    assert e.value.code == DSA_ERR_UNSUPPORTED
    assert "scratch" in str(e.value)
