"""ctypes loader for ``librcp.so``: signatures of the C ABI in ``include/rcp.h``.

Argument marshalling only.  Loading fails loudly if the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "librcp.so")

RCP_OK = 0
RCP_ERR_INVALID_ARG = 1
RCP_ERR_UNSUPPORTED = 2
RCP_ERR_CAPACITY = 3
RCP_ERR_WORKSPACE = 4
RCP_ERR_CUDA = 5

RCP_DEVERR_BAD_SLOT = 1
RCP_DEVERR_BAD_BLOCK = 2
RCP_DEVERR_BAD_LEN = 4
RCP_DEVERR_TIMEOUT = 8


class CacheConfig(ctypes.Structure):
    _fields_ = [("num_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("rank_k", ctypes.c_int32), ("rank_v", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("num_blocks", ctypes.c_int64),
                ("page_format", ctypes.c_int32)]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64P = ctypes.POINTER(ctypes.c_int64)
_SIG = {
    "rcp_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "rcp_config_supported": (ctypes.c_int, [ctypes.POINTER(CacheConfig)]),
    "rcp_create_cache": (ctypes.c_int, [ctypes.POINTER(CacheConfig), _P, _P, _P, _P, _P,
                                        ctypes.POINTER(_P)]),
    "rcp_destroy_cache": (ctypes.c_int, [_P]),
    "rcp_alloc_blocks": (ctypes.c_int, [_P, _I32, ctypes.POINTER(ctypes.c_int32)]),
    "rcp_free_blocks": (ctypes.c_int, [_P, _I32, ctypes.POINTER(ctypes.c_int32)]),
    "rcp_num_free_blocks": (ctypes.c_int, [_P, _I64P]),
    "rcp_workspace_size": (ctypes.c_int, [_P, _I32, ctypes.POINTER(ctypes.c_size_t)]),
    "rcp_append_kv": (ctypes.c_int, [_P, _P, _P, _P, _I32, _P]),
    "rcp_decode_attn": (ctypes.c_int, [_P, _P, _P, _I32, _P, _I32, _P, _P, ctypes.c_size_t, _P]),
    "rcp_decode_attn_sparse": (ctypes.c_int, [_P, _P, _P, _I32, _P, _I32, ctypes.c_float, _P,
                                              _P, _P, ctypes.c_size_t, _P]),
    "rcp_decode_step": (ctypes.c_int, [_P, _P, _P, _P, _I32, _P, _P, _I32, _P, _I32, _P, _P,
                                       ctypes.c_size_t, _P]),
    "rcp_prefill_attn": (ctypes.c_int, [_P, _P, _P, _I32, _P, _I32, _P, _I32, _P, _P,
                                        ctypes.c_size_t, _P]),
    "rcp_prefill_attn_reconstruct": (ctypes.c_int, [_P, _P, _P, _I32, _P, _I32, _P, _I32, _P,
                                                    _P, ctypes.c_size_t, _P]),
    "rcp_prefill_step": (ctypes.c_int, [_P, _P, _P, _P, _I32, _P, _P, _I32, _P, _I32, _P, _I32,
                                        _I32, _P, _P, ctypes.c_size_t, _P]),
    "rcp_prefill_reconstruct_workspace_size": (ctypes.c_int, [_P, _I32, _I32, _I32,
                                                              ctypes.POINTER(ctypes.c_size_t)]),
    "rcp_prefill_crossover_rows": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_int32)]),
    "rcp_set_profile_events": (ctypes.c_int, [_P, _P, _P]),
    "rcp_decode_attn_noalloc": (ctypes.c_int, [_P, _P, _P, _I32, _P, _I32, _P, _P]),
}

RCP_NOALLOC_SCRATCH_BYTES = 64 << 20
RCP_PAGES_FP16 = 0
RCP_PAGES_FP8_E4M3 = 1
RCP_PAGES_INT4 = 2

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library once; raise if it is missing (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -m rank_compressed_paged_gb300.build` "
            "(the CUDA library is the only implementation)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIG.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load().rcp_status_string(code).decode()


class RcpError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {status_string(code)} ({code})")
        self.code = code


def check(fn: str, code: int) -> None:
    if code != RCP_OK:
        raise RcpError(fn, code)
