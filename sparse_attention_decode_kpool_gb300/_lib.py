"""ctypes view of libdsa.so (the C ABI declared in include/dsa.h).

Loading fails loudly when the library is missing: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsa.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "dsa.h")

DSA_OK = 0
DSA_ERR_INVALID_ARG = 1
DSA_ERR_UNSUPPORTED = 2
DSA_ERR_CONFIG = 3
DSA_ERR_CUDA = 4
DSA_STATUS_BAD_TOKEN = 1
DSA_STATUS_BAD_BLOCK = 2
DSA_STATUS_TIMEOUT = 4
DSA_STATUS_CACHE_FULL = 8
DSA_ABI_VERSION = 8
DSA_OPT_PDL = 0
DSA_OPT_MLA_KERNEL = 1
DSA_MLA_KERNEL_AUTO = 0
DSA_MLA_KERNEL_TCGEN05 = 1
DSA_MLA_KERNEL_MMA = 2
DSA_MLA_KERNEL_CLUSTER = 3
DSA_OPT_SELECT_KERNEL = 2
DSA_SELECT_KERNEL_MERGE = 0
DSA_SELECT_KERNEL_RADIX = 1
DSA_OPT_PROJECT_KERNEL = 3
DSA_PROJECT_KERNEL_AUTO = 0
DSA_PROJECT_KERNEL_TCGEN05 = 1
DSA_PROJECT_KERNEL_MMA = 2
DSA_OPT_INJECT_STALL = 4


class DsaPaging(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("max_seq_len", ctypes.c_int32),
        ("seq_lens", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p),
        ("max_blocks", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_blocks", ctypes.c_int64),
    ]


_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t
_PG = ctypes.POINTER(DsaPaging)

# name -> (restype, argtypes), in header order
SIGNATURES = {
    "dsa_last_error": (ctypes.c_char_p, []),
    "dsa_abi_version": (_I, []),
    "dsa_set_option": (_I, [_I, _I]),
    "dsa_prefetch_l2": (_I, [_P, _SZ, _P]),
    "dsa_get_option": (_I, [_I]),
    "dsa_validate_config": (_I, [_I, _I, _I, _I]),
    "dsa_select_k": (_I, [_I, _I, _I]),
    "dsa_compress": (_I, [_P, _P, _P, _P, _P, _P, _F, _PG, _I, _I, _I, _P, _P, _P, _P, _P]),
    "dsa_compress_append": (_I, [_P, _P, _P, _P, _P, _P, _F, _PG, _I, _I, _I, _I, _P, _P, _P, _P,
                                 _P]),
    "dsa_indexer_store": (_I, [_P, _P, _P, _I, _I, _PG, _P, _P, _P, _P, _P, _P, _P]),
    "dsa_write_geom": (_I, [_P, _I, _P, _I, _P, _P, _P]),
    "dsa_decode_append": (_I, [_P, _P, _P, _P, _P, _P, _F, _PG, _P, _I, _I, _I, _I, _P, _P, _P,
                               _P, _P, _P, _P, _P, _P, _P]),
    "dsa_decode_append_fp8": (_I, [_P, _P, _P, _P, _P, _P, _F, _PG, _P, _I, _I, _I, _I, _P, _P,
                                   _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "dsa_score": (_I, [_P, _P, _I, _I, _I, _P, _P, _P, _P, _PG, _I, _I, _F, _P, _I, _P, _P]),
    "dsa_score_prefill": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _PG, _I, _I, _F, _P, _I, _P,
                               _P]),
    "dsa_select": (_I, [_P, _I, _I, _I, _I, _P, _P]),
    "dsa_expand": (_I, [_P, _I, _I, _I, _I, _I, _P, _P]),
    "dsa_select_expand": (_I, [_P, _I, _I, _I, _I, _I, _I, _P, _P, _P]),
    "dsa_expand_tail": (_I, [_P, _I, _I, _I, _I, _I, _P, _I, _P, _P]),
    "dsa_select_expand_tail": (_I, [_P, _I, _I, _I, _I, _I, _P, _I, _P, _P, _P]),
    "dsa_sparse_mla_decode_workspace": (_I, [_I, _I, _I, _I, _I, _I, ctypes.POINTER(_SZ)]),
    "dsa_sparse_mla_decode": (_I, [_P, _I, _I, _I, _P, _P, _PG, _P, _I, _F, _P, _I, _P, _P, _P,
                                   _P, _SZ, _P]),
    "dsa_quantize_latent": (_I, [_P, ctypes.c_longlong, _I, _P, _P, _P]),
    "dsa_sparse_mla_decode_fp8": (_I, [_P, _I, _I, _I, _P, _P, _P, _PG, _P, _I, _F, _P, _I, _P,
                                       _P, _P, _P, _SZ, _P]),
    "dsa_frontend_workspace": (_I, [_I, _I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(_SZ)]),
    "dsa_frontend": (_I, [_P, _I, _I, _P, _I, _I, _I, _I, _I, _P, _P, _F, _P, _I, _P, _P, _P,
                          _P, _P, _P, _P, _P, _SZ, _P]),
    "dsa_latent_project_workspace": (_I, [_I, _I, _I, _I, ctypes.POINTER(_SZ)]),
    "dsa_latent_project": (_I, [_P, _I, _I, _I, _P, _I, _P, _P, _P, _SZ, _P]),
    "dsa_sparse_mla_decode_noalloc": (_I, [_P, _I, _I, _I, _P, _P, _PG, _P, _I, _F, _P, _I, _P,
                                           _P, _P, _P]),
}

_lib = None


def header_functions() -> list[str]:
    """Function names declared in include/dsa.h."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return re.findall(r"\b(dsa_[a-z0-9_]+)\s*\(", src)


def load() -> ctypes.CDLL:
    """Load libdsa.so (built by ``_build.build()``); raise if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (no CPU fallback exists)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if lib.dsa_abi_version() != DSA_ABI_VERSION:
        raise RuntimeError("libdsa.so ABI version mismatch; rebuild it")
    _lib = lib
    return lib


class DsaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[dsa error {code}] {msg}")
        self.code = code


def check(code: int) -> None:
    if code != DSA_OK:
        raise DsaError(code, load().dsa_last_error().decode())
