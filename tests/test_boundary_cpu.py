"""The C ABI on the host, without a GPU: the library loads and exports every symbol
include/dsa.h declares, host-visible argument errors come back as the documented
codes before anything touches CUDA, the paging struct matches the C layout, and the
product path refuses to run without the library."""
import ctypes
import os
import subprocess
import sys
import tempfile

import pytest

from sparse_attention_decode_kpool_gb300 import _build, _lib
from sparse_attention_decode_kpool_gb300._lib import (DSA_ERR_CONFIG, DSA_ERR_INVALID_ARG,
                                                       DSA_ERR_UNSUPPORTED, DSA_OK, DsaPaging)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 0x10000  # a non-NULL device address the host never dereferences


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return _lib.load()


def _err(lib):
    return lib.dsa_last_error().decode()


def test_exports_every_declared_symbol(lib):
    names = _lib.header_functions()
    assert len(names) >= 11
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert set(_lib.SIGNATURES) == set(names)
    assert lib.dsa_abi_version() == _lib.DSA_ABI_VERSION


def test_header_constants_match_the_binding():
    """Every integer DSA_* macro of include/dsa.h that the Python binding names has the
    same value there, and the binding names no DSA_* constant the header lacks."""
    import re
    text = open(os.path.join(ROOT, "include", "dsa.h")).read()
    header = {m.group(1): int(m.group(2))
              for m in re.finditer(r"^#define\s+(DSA_[A-Z0-9_]+)\s+(-?\d+)\b", text, re.M)}
    binding = {k: v for k, v in vars(_lib).items() if k.startswith("DSA_") and isinstance(v, int)}
    assert len(binding) >= 20
    assert not set(binding) - set(header), sorted(set(binding) - set(header))
    wrong = {k: (binding[k], header[k]) for k in binding if binding[k] != header[k]}
    assert not wrong, wrong


@pytest.mark.parametrize("args,code", [
    ((4, 2048, 512, 64), DSA_OK),
    ((0, 2048, 512, 64), DSA_ERR_CONFIG),
    ((4, 0, 512, 64), DSA_ERR_CONFIG),
    ((4, 2050, 512, 64), DSA_ERR_CONFIG),
    ((32, 64, 512, 64), DSA_ERR_UNSUPPORTED),
    ((16, 64, 512, 64), DSA_OK),
    ((4, 2048, 0, 64), DSA_ERR_CONFIG),
    ((4, 2048, 576, 64), DSA_ERR_UNSUPPORTED),
    ((4, 2048, 512, 0), DSA_ERR_CONFIG),
])
def test_validate_config_rules(lib, args, code):
    rc = lib.dsa_validate_config(*args)
    assert rc == code
    if code:
        assert _err(lib)


def test_prefetch_l2_argument_errors(lib):
    assert lib.dsa_prefetch_l2(None, 0, None) == DSA_OK  # nothing to do: no launch
    assert lib.dsa_prefetch_l2(FAKE, 0, None) == DSA_OK
    assert lib.dsa_prefetch_l2(FAKE, 8, None) == DSA_OK  # below one 16-byte unit
    assert lib.dsa_prefetch_l2(None, 1 << 20, None) == DSA_ERR_INVALID_ARG
    assert lib.dsa_prefetch_l2(FAKE + 8, 1 << 20, None) == DSA_ERR_INVALID_ARG
    assert "aligned" in _err(lib)


def test_launch_options(lib):
    from sparse_attention_decode_kpool_gb300._lib import (DSA_MLA_KERNEL_AUTO,
                                                           DSA_MLA_KERNEL_MMA,
                                                           DSA_MLA_KERNEL_TCGEN05,
                                                           DSA_OPT_MLA_KERNEL, DSA_OPT_PDL)
    assert lib.dsa_get_option(DSA_OPT_PDL) == 1
    assert lib.dsa_get_option(DSA_OPT_MLA_KERNEL) == DSA_MLA_KERNEL_AUTO
    assert lib.dsa_get_option(99) == -1
    try:
        for v in (DSA_MLA_KERNEL_TCGEN05, DSA_MLA_KERNEL_MMA, DSA_MLA_KERNEL_AUTO):
            assert lib.dsa_set_option(DSA_OPT_MLA_KERNEL, v) == DSA_OK
            assert lib.dsa_get_option(DSA_OPT_MLA_KERNEL) == v
        assert lib.dsa_set_option(DSA_OPT_MLA_KERNEL, 3) == DSA_OK
        assert lib.dsa_set_option(DSA_OPT_MLA_KERNEL, 4) == DSA_ERR_INVALID_ARG
        assert "DSA_OPT_MLA_KERNEL" in _err(lib)
        assert lib.dsa_set_option(DSA_OPT_PDL, 0) == DSA_OK
        assert lib.dsa_get_option(DSA_OPT_PDL) == 0
        assert lib.dsa_set_option(DSA_OPT_PDL, 2) == DSA_ERR_INVALID_ARG
        assert lib.dsa_set_option(2, 1) == DSA_OK  # DSA_OPT_SELECT_KERNEL, radix
        assert lib.dsa_get_option(2) == 1
        assert lib.dsa_set_option(2, 2) == DSA_ERR_INVALID_ARG
        assert lib.dsa_set_option(7, 0) == DSA_ERR_INVALID_ARG
        # DSA_OPT_INJECT_STALL: off by default, 0 or 1 only
        assert lib.dsa_get_option(4) == 0
        assert lib.dsa_set_option(4, 2) == DSA_ERR_INVALID_ARG
        assert lib.dsa_set_option(4, 1) == DSA_OK
        assert lib.dsa_get_option(4) == 1
        assert lib.dsa_set_option(4, 0) == DSA_OK
    finally:
        lib.dsa_set_option(DSA_OPT_PDL, 1)
        lib.dsa_set_option(DSA_OPT_MLA_KERNEL, DSA_MLA_KERNEL_AUTO)
        lib.dsa_set_option(2, 0)
    # nothing in the library reads the environment
    src = os.path.join(ROOT, "sparse_attention_decode_kpool_gb300", "csrc")
    for f in os.listdir(src):
        assert "getenv" not in open(os.path.join(src, f)).read(), f


def test_select_k(lib):
    assert lib.dsa_select_k(2048, 4, 65536) == 512
    assert lib.dsa_select_k(256, 4, 50) == 50
    assert lib.dsa_select_k(0, 4, 50) == -1


def _paging(batch=1, max_seq_len=1024, block_table=None, max_blocks=0, block_size=0, nb=0):
    pg = DsaPaging()
    pg.batch, pg.max_seq_len, pg.seq_lens = batch, max_seq_len, FAKE
    pg.block_table, pg.max_blocks, pg.block_size, pg.num_blocks = block_table, max_blocks, block_size, nb
    return pg


def test_compress_argument_errors(lib):
    pg = _paging()
    call = lambda kp, ihd, pgp=ctypes.byref(pg), fk=0: lib.dsa_compress(
        FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1e-6, pgp, fk, kp, ihd, FAKE, FAKE, None, None, None)
    assert call(17, 128) == DSA_ERR_UNSUPPORTED
    assert call(0, 128) == DSA_ERR_UNSUPPORTED
    assert call(4, 96) == DSA_ERR_UNSUPPORTED
    assert call(4, 128, None) == DSA_ERR_INVALID_ARG
    assert call(4, 128, ctypes.byref(pg), -1) == DSA_ERR_INVALID_ARG
    paged = _paging(block_table=FAKE, max_blocks=16, block_size=64, nb=8)
    assert call(3, 128, ctypes.byref(paged)) == DSA_ERR_UNSUPPORTED  # 64 % 3 != 0
    assert call(4, 128, ctypes.byref(paged), 2) == DSA_ERR_UNSUPPORTED  # first_key % kpool
    short = _paging(max_seq_len=2048, block_table=FAKE, max_blocks=16, block_size=64, nb=8)
    assert call(4, 128, ctypes.byref(short)) == DSA_ERR_INVALID_ARG  # 16*64 < 2048
    assert "paging" in _err(lib)


def test_append_entry_argument_errors(lib):
    pg = _paging()
    ca = lambda n, kp=4, ihd=128: lib.dsa_compress_append(
        FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1e-6, ctypes.byref(pg), 0, kp, ihd, n, FAKE, FAKE,
        None, None, None)
    assert ca(0) == DSA_ERR_INVALID_ARG and "new_tokens" in _err(lib)
    assert ca(1, 17) == DSA_ERR_UNSUPPORTED
    assert ca(1, 4, 96) == DSA_ERR_UNSUPPORTED
    # dsa_indexer_store(k_new, gate_new, ckv_new, ihd, kvl, pg, seq_lens, k_raw, gate, valid,
    #                   ckv, status, stream)
    st = lambda ihd=128, kvl=512, ckv_new=FAKE, ckv=FAKE, sl=FAKE, pgp=ctypes.byref(pg): \
        lib.dsa_indexer_store(FAKE, FAKE, ckv_new, ihd, kvl, pgp, sl, FAKE, FAKE, FAKE, ckv,
                              None, None)
    assert st(ihd=96) == DSA_ERR_UNSUPPORTED
    assert st(ckv=None) == DSA_ERR_INVALID_ARG and "together" in _err(lib)
    assert st(kvl=500) == DSA_ERR_INVALID_ARG
    assert st(sl=FAKE + 64) == DSA_ERR_INVALID_ARG and "seq_lens" in _err(lib)
    assert st(sl=None) == DSA_ERR_INVALID_ARG
    assert st(pgp=None) == DSA_ERR_INVALID_ARG
    assert lib.dsa_indexer_store(FAKE + 8, FAKE, None, 128, 0, ctypes.byref(pg), FAKE, FAKE,
                                 FAKE, FAKE, None, None, None) == DSA_ERR_INVALID_ARG  # align
    # dsa_decode_append(k_new, gate_new, ckv_new, ape, ln_w, ln_b, eps, pg, seq_lens, fk,
    #                   kpool, ihd, kvl, k_raw, gate, valid, ckv, kpool_out, pool_valid,
    #                   pool_idx, row_ctx, status, stream)
    da = lambda kp=4, ihd=128, kvl=512, ckv=FAKE, sl=FAKE, fk=0, pgp=ctypes.byref(pg): \
        lib.dsa_decode_append(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1e-6, pgp, sl, fk, kp, ihd, kvl,
                              FAKE, FAKE, FAKE, ckv, FAKE, FAKE, None, None, None, None)
    assert da(kp=17) == DSA_ERR_UNSUPPORTED
    assert da(ihd=96) == DSA_ERR_UNSUPPORTED
    assert da(fk=-1) == DSA_ERR_INVALID_ARG
    assert da(ckv=None) == DSA_ERR_INVALID_ARG and "together" in _err(lib)
    assert da(kvl=12) == DSA_ERR_INVALID_ARG
    assert da(sl=FAKE + 4) == DSA_ERR_INVALID_ARG and "seq_lens" in _err(lib)
    assert da(pgp=None) == DSA_ERR_INVALID_ARG
    paged = _paging(block_table=FAKE, max_blocks=16, block_size=64, nb=8)
    assert da(fk=2, pgp=ctypes.byref(paged)) == DSA_ERR_UNSUPPORTED  # first_key % kpool
    # dsa_decode_append_fp8: as dsa_decode_append plus ckv_codes, ckv_scales after ckv
    d8 = lambda kvl=512, codes=FAKE, scales=FAKE, ckv_new=FAKE, ckv=None: \
        lib.dsa_decode_append_fp8(FAKE, FAKE, ckv_new, FAKE, FAKE, FAKE, 1e-6, ctypes.byref(pg),
                                  FAKE, 0, 4, 128, kvl, FAKE, FAKE, FAKE, ckv, codes, scales,
                                  FAKE, FAKE, None, None, None, None)
    assert d8(codes=None) == DSA_ERR_INVALID_ARG and "FP8" in _err(lib)
    assert d8(scales=None) == DSA_ERR_INVALID_ARG
    assert d8(ckv_new=None) == DSA_ERR_INVALID_ARG and "together" in _err(lib)
    assert d8(kvl=196) == DSA_ERR_INVALID_ARG and "multiple of 8" in _err(lib)
    assert d8(kvl=192) == DSA_ERR_INVALID_ARG and "multiple of 128" in _err(lib)
    assert d8(codes=FAKE + 8) == DSA_ERR_INVALID_ARG and "aligned" in _err(lib)
    assert lib.dsa_write_geom(FAKE, 0, None, 4, FAKE, None, None) == DSA_ERR_INVALID_ARG
    assert lib.dsa_write_geom(FAKE, 2, None, -1, FAKE, None, None) == DSA_ERR_INVALID_ARG
    assert lib.dsa_write_geom(FAKE, 2, None, 0, None, None, None) == DSA_OK
    assert lib.dsa_write_geom(None, 2, None, 3, FAKE, None, None) == DSA_ERR_INVALID_ARG


def test_score_select_expand_argument_errors(lib):
    pg = _paging()
    score = lambda heads, ihd, kp=4: lib.dsa_score(FAKE, FAKE, 1, heads, ihd, None, None, FAKE,
                                                   FAKE, ctypes.byref(pg), 0, kp, 0.1, FAKE, 16,
                                                   None, None)
    assert score(65, 128) == DSA_ERR_UNSUPPORTED
    assert score(32, 96) == DSA_ERR_UNSUPPORTED
    assert score(32, 128, 0) == DSA_ERR_UNSUPPORTED
    assert lib.dsa_score(FAKE, FAKE, 0, 32, 128, None, None, FAKE, FAKE, ctypes.byref(pg), 0, 4,
                         0.1, FAKE, 16, None, None) == DSA_OK  # nothing to do
    assert lib.dsa_select(FAKE, 1, 100, 0, 4, FAKE, None) == DSA_ERR_CONFIG
    assert lib.dsa_select(FAKE, 1, 327681, 2048, 4, FAKE, None) == DSA_ERR_UNSUPPORTED
    assert lib.dsa_select(FAKE, 0, 100, 2048, 4, FAKE, None) == DSA_OK
    assert lib.dsa_select(None, 1, 100, 2048, 4, FAKE, None) == DSA_ERR_INVALID_ARG
    assert lib.dsa_expand(FAKE, 2, 64, 0, 4, 255, FAKE, None) == DSA_ERR_INVALID_ARG
    assert lib.dsa_expand(FAKE, 0, 64, 0, 4, 256, FAKE, None) == DSA_OK
    assert lib.dsa_expand(FAKE, 2, 64, -1, 4, 256, FAKE, None) == DSA_ERR_INVALID_ARG


def test_tail_entry_argument_errors(lib):
    # dsa_expand_tail(pool_ids, rows, sk, first_key, kpool, index_topk, row_ctx,
    #                 out_width, token_ids, stream): out_width >= index_topk + kpool - 1.
    et = lib.dsa_expand_tail
    assert et(FAKE, 2, 64, 0, 4, 256, FAKE, 258, FAKE, None) == DSA_ERR_INVALID_ARG
    assert "index_topk + kpool - 1" in _err(lib)
    assert et(FAKE, 2, 65, 0, 4, 256, FAKE, 259, FAKE, None) == DSA_ERR_INVALID_ARG
    assert et(FAKE, 2, 64, 0, 4, 256, None, 259, FAKE, None) == DSA_ERR_INVALID_ARG
    assert et(FAKE, 2, 64, 0, 0, 256, FAKE, 259, FAKE, None) == DSA_ERR_INVALID_ARG
    assert et(FAKE, 0, 64, 0, 4, 256, FAKE, 259, FAKE, None) == DSA_OK
    st = lib.dsa_select_expand_tail
    assert st(FAKE, 1, 100, 256, 4, 0, FAKE, 258, FAKE, FAKE, None) == DSA_ERR_INVALID_ARG
    assert st(FAKE, 1, 100, 256, 4, 0, None, 259, FAKE, FAKE, None) == DSA_ERR_INVALID_ARG
    assert st(FAKE, 1, 100, 0, 4, 0, FAKE, 259, FAKE, FAKE, None) == DSA_ERR_CONFIG
    assert st(FAKE, 1, 100, 256, 17, 0, FAKE, 400, FAKE, FAKE, None) == DSA_ERR_UNSUPPORTED
    assert st(None, 1, 100, 256, 4, 0, FAKE, 259, FAKE, FAKE, None) == DSA_ERR_INVALID_ARG
    assert st(FAKE, 0, 100, 256, 4, 0, FAKE, 259, FAKE, FAKE, None) == DSA_OK


def test_score_prefill_argument_errors(lib):
    pg = _paging(batch=2)

    def pf(heads=32, ihd=128, seq=0, kp=4, pgp=None, rows=8, q=FAKE, fk=0):
        return lib.dsa_score_prefill(q, FAKE, rows, heads, ihd, seq, None, FAKE, FAKE,
                                     pgp or ctypes.byref(pg), fk, kp, 0.1, FAKE, 64, None, None)

    assert pf(heads=20) == DSA_ERR_UNSUPPORTED
    assert "dsa_score" in _err(lib)
    assert pf(heads=256) == DSA_ERR_UNSUPPORTED
    assert pf(ihd=96) == DSA_ERR_UNSUPPORTED
    assert pf(kp=17) == DSA_ERR_UNSUPPORTED
    assert pf(seq=2) == DSA_ERR_INVALID_ARG
    assert pf(seq=-1) == DSA_ERR_INVALID_ARG
    assert pf(rows=-1) == DSA_ERR_INVALID_ARG
    assert pf(fk=-1) == DSA_ERR_INVALID_ARG
    assert pf(q=FAKE + 8) == DSA_ERR_INVALID_ARG  # misaligned
    assert pf(q=None) == DSA_ERR_INVALID_ARG
    paged = _paging(block_table=FAKE, max_blocks=16, block_size=64, nb=8)
    assert pf(pgp=ctypes.byref(paged)) == DSA_ERR_UNSUPPORTED
    assert "paged" in _err(lib)
    assert pf(rows=0) == DSA_OK  # nothing to do


def test_sparse_mla_argument_errors(lib):
    pg = _paging()

    def mla(kvl=512, hidden=4096, oabs=FAKE, y=FAKE, heads=64):
        return lib.dsa_sparse_mla_decode(FAKE, 1, heads, kvl, None, FAKE, ctypes.byref(pg), FAKE,
                                         2048, 0.0625, oabs, hidden, y, None, None, FAKE, 1 << 20,
                                         None)

    assert mla(kvl=576) == DSA_ERR_UNSUPPORTED
    assert mla(kvl=0) == DSA_ERR_CONFIG
    assert mla(hidden=100) == DSA_ERR_UNSUPPORTED
    assert mla(y=None) == DSA_ERR_INVALID_ARG
    assert mla(heads=0) == DSA_ERR_INVALID_ARG
    n = ctypes.c_size_t()
    assert lib.dsa_sparse_mla_decode_workspace(1, 64, 576, 2048, 4096, 1, ctypes.byref(n)) == \
        DSA_ERR_UNSUPPORTED
    assert lib.dsa_sparse_mla_decode_noalloc(FAKE, 1, 64, 576, None, FAKE, ctypes.byref(pg), FAKE,
                                             2048, 0.0625, FAKE, 4096, FAKE, None, None,
                                             None) == DSA_ERR_UNSUPPORTED


def test_paging_struct_matches_c_layout(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "dsa.h"\nint main(void){'
                   'printf("%zu %zu %zu %zu %zu %zu %zu %zu\\n", sizeof(dsa_paging),'
                   'offsetof(dsa_paging,batch),offsetof(dsa_paging,max_seq_len),'
                   'offsetof(dsa_paging,seq_lens),offsetof(dsa_paging,block_table),'
                   'offsetof(dsa_paging,max_blocks),offsetof(dsa_paging,block_size),'
                   'offsetof(dsa_paging,num_blocks));return 0;}\n')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    c = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True).stdout.split()]
    py = [ctypes.sizeof(DsaPaging)] + [getattr(DsaPaging, f).offset for f, _ in DsaPaging._fields_]
    assert c == py


def test_missing_library_fails_loudly(monkeypatch):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", "/nonexistent/libdsa.so")
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        _lib.load()
