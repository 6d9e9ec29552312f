"""The C-ABI library: loads, exports every declared symbol, validates on the host (no GPU).

None of these tests launches a kernel: every call here returns before any CUDA call
(argument checks, block pool, workspace arithmetic).  Pointers are fake but aligned.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from rank_compressed_paged_gb300 import build
    build.build()
    from rank_compressed_paged_gb300 import _lib
    return _lib.load()


def _declared_symbols():
    src = open(os.path.join(ROOT, "include", "rcp.h")).read()
    return sorted(set(re.findall(r"^(?:const char\*|rcp_status)\s+(rcp_\w+)\(", src, re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_symbols()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), n


def _cfg(_lib, H=32, d=128, rk=64, R=1024, bs=16, nb=100, fmt=0):
    return _lib.CacheConfig(H, d, rk, R, bs, nb, fmt)


def _create(lib, _lib, cfg, ptrs=(0x10000, 0x20000, 0x30000, 0x40000, 0x50000)):
    h = ctypes.c_void_p()
    st = lib.rcp_create_cache(ctypes.byref(cfg), *ptrs, ctypes.byref(h))
    return st, h


def test_config_support_and_status_strings(lib):
    from rank_compressed_paged_gb300 import _lib
    assert lib.rcp_config_supported(ctypes.byref(_cfg(_lib))) == _lib.RCP_OK
    assert lib.rcp_config_supported(ctypes.byref(_cfg(_lib, 4, 64, 16, 64))) == _lib.RCP_OK
    assert lib.rcp_config_supported(ctypes.byref(_cfg(_lib, bs=32))) == _lib.RCP_ERR_UNSUPPORTED
    assert lib.rcp_config_supported(ctypes.byref(_cfg(_lib, rk=48))) == _lib.RCP_ERR_UNSUPPORTED
    assert lib.rcp_config_supported(ctypes.byref(_cfg(_lib, fmt=_lib.RCP_PAGES_FP8_E4M3))) == \
        _lib.RCP_OK
    assert lib.rcp_config_supported(ctypes.byref(_cfg(_lib, fmt=_lib.RCP_PAGES_INT4))) == \
        _lib.RCP_OK
    assert lib.rcp_config_supported(ctypes.byref(_cfg(_lib, fmt=3))) == _lib.RCP_ERR_UNSUPPORTED
    assert lib.rcp_config_supported(None) == _lib.RCP_ERR_INVALID_ARG
    for code in range(6):
        assert lib.rcp_status_string(code)
    assert b"workspace" in lib.rcp_status_string(_lib.RCP_ERR_WORKSPACE)


def test_create_cache_rejects_bad_arguments(lib):
    from rank_compressed_paged_gb300 import _lib
    st, _ = _create(lib, _lib, _cfg(_lib, rk=48))
    assert st == _lib.RCP_ERR_UNSUPPORTED
    st, _ = _create(lib, _lib, _cfg(_lib, nb=0))
    assert st == _lib.RCP_ERR_INVALID_ARG
    st, _ = _create(lib, _lib, _cfg(_lib), ptrs=(0x10008, 0x20000, 0x30000, 0x40000, 0x50000))
    assert st == _lib.RCP_ERR_INVALID_ARG            # misaligned K pages
    st, _ = _create(lib, _lib, _cfg(_lib), ptrs=(0x10000, None, 0x30000, 0x40000, 0x50000))
    assert st == _lib.RCP_ERR_INVALID_ARG            # null V pages
    st, h = _create(lib, _lib, _cfg(_lib))
    assert st == _lib.RCP_OK and h.value
    assert lib.rcp_destroy_cache(h) == _lib.RCP_OK


def test_block_pool_alloc_free(lib):
    from rank_compressed_paged_gb300 import _lib
    st, h = _create(lib, _lib, _cfg(_lib, nb=10))
    assert st == _lib.RCP_OK
    n = ctypes.c_int64()
    lib.rcp_num_free_blocks(h, ctypes.byref(n))
    assert n.value == 10
    ids = (ctypes.c_int32 * 10)()
    assert lib.rcp_alloc_blocks(h, 7, ids) == _lib.RCP_OK
    got = [ids[i] for i in range(7)]
    assert len(set(got)) == 7 and all(0 <= i < 10 for i in got)
    assert lib.rcp_alloc_blocks(h, 4, ids) == _lib.RCP_ERR_CAPACITY     # only 3 left
    lib.rcp_num_free_blocks(h, ctypes.byref(n))
    assert n.value == 3                                                # unchanged on failure
    bad = (ctypes.c_int32 * 2)(got[0], got[0])
    assert lib.rcp_free_blocks(h, 2, bad) == _lib.RCP_ERR_CAPACITY       # duplicate in list
    oob = (ctypes.c_int32 * 1)(10)
    assert lib.rcp_free_blocks(h, 1, oob) == _lib.RCP_ERR_CAPACITY       # out of range
    fr = (ctypes.c_int32 * 2)(got[0], got[1])
    assert lib.rcp_free_blocks(h, 2, fr) == _lib.RCP_OK
    assert lib.rcp_free_blocks(h, 1, fr) == _lib.RCP_ERR_CAPACITY        # double free
    lib.rcp_num_free_blocks(h, ctypes.byref(n))
    assert n.value == 5
    assert lib.rcp_alloc_blocks(h, 5, ids) == _lib.RCP_OK
    assert sorted(ids[i] for i in range(5)) == sorted(set(range(10)) - set(got[2:]))
    lib.rcp_destroy_cache(h)


def test_workspace_size_and_host_checks(lib):
    from rank_compressed_paged_gb300 import _lib
    st, h = _create(lib, _lib, _cfg(_lib))
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.rcp_workspace_size(h, 16, ctypes.byref(a)) == _lib.RCP_OK
    assert lib.rcp_workspace_size(h, 64, ctypes.byref(b)) == _lib.RCP_OK
    assert b.value > a.value > 0 and a.value % 256 == 0
    assert lib.rcp_workspace_size(h, -1, ctypes.byref(a)) == _lib.RCP_ERR_INVALID_ARG
    ws = 0x100000
    # too-small workspace is rejected before any launch
    assert lib.rcp_decode_attn(h, 0x1000, 0x2000, 64, 0x3000, 16, 0x4000, ws, 1024, None) \
        == _lib.RCP_ERR_WORKSPACE
    # misaligned q, null table, bad max_blocks
    assert lib.rcp_decode_attn(h, 0x1008, 0x2000, 64, 0x3000, 16, 0x4000, ws, b.value, None) \
        == _lib.RCP_ERR_INVALID_ARG
    assert lib.rcp_decode_attn(h, 0x1000, None, 64, 0x3000, 16, 0x4000, ws, b.value, None) \
        == _lib.RCP_ERR_INVALID_ARG
    assert lib.rcp_decode_attn(h, 0x1000, 0x2000, 0, 0x3000, 16, 0x4000, ws, b.value, None) \
        == _lib.RCP_ERR_INVALID_ARG
    assert lib.rcp_decode_attn(h, 0x1000, 0x2000, 64, 0x3000, 0, 0x4000, ws, b.value, None) \
        == _lib.RCP_OK                                               # empty batch: no work
    assert lib.rcp_prefill_attn(h, 0x1000, None, 8, 0x2000, 64, 0x3000, 2, 0x4000, ws, b.value,
                                None) == _lib.RCP_ERR_INVALID_ARG
    assert lib.rcp_append_kv(h, 0x1000, 0x2000, 0x3004, 4, None) == _lib.RCP_ERR_INVALID_ARG
    assert lib.rcp_append_kv(h, 0x1000, 0x2000, 0x3000, 0, None) == _lib.RCP_OK
    assert lib.rcp_append_kv(h, 0x1000, 0x2000, 0x3000, -1, None) == _lib.RCP_ERR_INVALID_ARG
    lib.rcp_destroy_cache(h)


def test_prefill_step_host_checks(lib):
    """rcp_prefill_step refuses bad arguments before any CUDA call, as the append and the
    prefill calls it stands for do; with no tokens and no query rows it has nothing to do."""
    from rank_compressed_paged_gb300 import _lib
    st, h = _create(lib, _lib, _cfg(_lib))
    b = ctypes.c_size_t()
    assert lib.rcp_prefill_reconstruct_workspace_size(h, 8, 2, 64, ctypes.byref(b)) == _lib.RCP_OK
    ws = 0x100000

    def step(k=0x1000, T=8, cu=0x5000, nq=8, recon=1, ws_bytes=None):
        return lib.rcp_prefill_step(h, k, 0x2000, 0x3000, T, 0x4000, cu, nq, 0x6000, 64, 0x7000,
                                    2, recon, 0x8000, ws, b.value if ws_bytes is None else ws_bytes,
                                    None)

    assert step(recon=2) == _lib.RCP_ERR_INVALID_ARG          # neither variant
    assert step(recon=-1) == _lib.RCP_ERR_INVALID_ARG
    assert step(cu=None) == _lib.RCP_ERR_INVALID_ARG          # a prefill needs chunk offsets
    assert step(T=-1) == _lib.RCP_ERR_INVALID_ARG
    assert step(k=0x1008) == _lib.RCP_ERR_INVALID_ARG         # misaligned keys of the append
    assert step(ws_bytes=1024) == _lib.RCP_ERR_WORKSPACE      # workspace of the prefill call
    assert step(T=0, nq=0) == _lib.RCP_OK                     # nothing to append or attend
    lib.rcp_destroy_cache(h)


def test_python_layer_fails_loudly_without_library(tmp_path):
    from rank_compressed_paged_gb300 import _lib
    saved = _lib._lib
    _lib._lib = None
    try:
        with pytest.raises(RuntimeError, match="missing"):
            _lib.load(str(tmp_path / "nope.so"))
    finally:
        _lib._lib = saved


def test_prefill_crossover_and_reconstruct_workspace(lib):
    from rank_compressed_paged_gb300 import _lib
    st, h = _create(lib, _lib, _cfg(_lib))
    assert st == _lib.RCP_OK
    rows = ctypes.c_int32()
    assert lib.rcp_prefill_crossover_rows(h, ctypes.byref(rows)) == _lib.RCP_OK
    assert rows.value == 147                 # ceil(1024 * 128 / (1024 - 128))
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    # V^ (2 * H * d bytes per key) dominates once pages outnumber the query rows
    assert lib.rcp_prefill_reconstruct_workspace_size(h, 64, 16, 272, ctypes.byref(a)) == 0
    assert lib.rcp_prefill_reconstruct_workspace_size(h, 64, 16, 273, ctypes.byref(b)) == 0
    assert b.value - a.value >= 16 * 16 * 32 * 128 * 2   # one more page per request
    assert a.value >= 16 * 272 * 16 * 32 * 128 * 2
    small = ctypes.c_size_t()
    assert lib.rcp_workspace_size(h, 64, ctypes.byref(small)) == 0
    assert a.value > small.value
    assert lib.rcp_prefill_reconstruct_workspace_size(h, -1, 16, 272, ctypes.byref(a)) == \
        _lib.RCP_ERR_INVALID_ARG
    lib.rcp_destroy_cache(h)
    st, h = _create(lib, _lib, _cfg(_lib, 4, 64, 16, 64))
    assert lib.rcp_prefill_crossover_rows(h, ctypes.byref(rows)) == _lib.RCP_OK
    assert rows.value == 2**31 - 1           # R <= d: rank space is never dearer
    lib.rcp_destroy_cache(h)


def test_sparse_decode_host_checks(lib):
    """Threshold range and workspace are checked before any CUDA call, for every page
    format."""
    from rank_compressed_paged_gb300 import _lib
    st, h = _create(lib, _lib, _cfg(_lib))
    b = ctypes.c_size_t()
    assert lib.rcp_workspace_size(h, 16, ctypes.byref(b)) == _lib.RCP_OK
    ws = 0x100000
    args = (h, 0x1000, 0x2000, 64, 0x3000, 16)
    for bad in (1.0, -0.25, float("nan"), float("inf")):
        assert lib.rcp_decode_attn_sparse(*args, bad, None, 0x4000, ws, b.value, None) \
            == _lib.RCP_ERR_INVALID_ARG, bad
    assert lib.rcp_decode_attn_sparse(*args, 0.01, None, 0x4000, ws, 1024, None) \
        == _lib.RCP_ERR_WORKSPACE
    assert lib.rcp_decode_attn_sparse(h, 0x1000, 0x2000, 64, 0x3000, 0, 0.01, None, 0x4000, ws,
                                      b.value, None) == _lib.RCP_OK   # empty batch
    lib.rcp_destroy_cache(h)
    for fmt in (_lib.RCP_PAGES_FP8_E4M3, _lib.RCP_PAGES_INT4):
        # every page format is accepted: the same host checks, no CUDA call for an empty batch
        st, hq = _create(lib, _lib, _cfg(_lib, fmt=fmt))
        assert st == _lib.RCP_OK
        assert lib.rcp_decode_attn_sparse(hq, 0x1000, 0x2000, 64, 0x3000, 16, 2.0, None, 0x4000,
                                          ws, b.value, None) == _lib.RCP_ERR_INVALID_ARG
        assert lib.rcp_decode_attn_sparse(hq, 0x1000, 0x2000, 64, 0x3000, 16, 0.01, None, 0x4000,
                                          ws, 1024, None) == _lib.RCP_ERR_WORKSPACE
        assert lib.rcp_decode_attn_sparse(hq, 0x1000, 0x2000, 64, 0x3000, 0, 0.01, None, 0x4000,
                                          ws, b.value, None) == _lib.RCP_OK
        lib.rcp_destroy_cache(hq)


def test_reconstruct_workspace_grows_by_the_widened_pages_for_e4m3(lib):
    """E4M3 pages: the reconstructing prefill's workspace also holds fp16 copies of the
    pages the batch can reach (2 * 16 * (H r_k + R) bytes each) and their table (4 bytes)."""
    from rank_compressed_paged_gb300 import _lib
    st, h16 = _create(lib, _lib, _cfg(_lib))
    st8, h8 = _create(lib, _lib, _cfg(_lib, fmt=_lib.RCP_PAGES_FP8_E4M3))
    assert st == st8 == _lib.RCP_OK
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.rcp_prefill_reconstruct_workspace_size(h16, 64, 16, 272, ctypes.byref(a)) == 0
    assert lib.rcp_prefill_reconstruct_workspace_size(h8, 64, 16, 272, ctypes.byref(b)) == 0
    pages = 16 * 272
    extra = pages * 2 * 16 * (32 * 64 + 1024) + pages * 4
    assert extra <= b.value - a.value <= extra + 3 * 256
    # the rank-space prefill on quantized pages widens them too: the query-row workspace
    # alone is refused before any launch (E4M3 and 4-bit alike)
    st4, h4 = _create(lib, _lib, _cfg(_lib, fmt=_lib.RCP_PAGES_INT4))
    assert st4 == _lib.RCP_OK
    small = ctypes.c_size_t()
    for h in (h8, h4):
        assert lib.rcp_workspace_size(h, 64, ctypes.byref(small)) == 0
        assert small.value < b.value
        assert lib.rcp_prefill_attn(h, 0x1000, 0x5000, 64, 0x2000, 272, 0x3000, 16, 0x4000,
                                    0x100000, small.value, None) == _lib.RCP_ERR_WORKSPACE
    lib.rcp_destroy_cache(h16)
    lib.rcp_destroy_cache(h8)
    lib.rcp_destroy_cache(h4)


def _declared_param_counts():
    """Parameter count of every function the header declares (comments stripped)."""
    src = open(os.path.join(ROOT, "include", "rcp.h")).read()
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    out = {}
    for m in re.finditer(r"^(?:const char\*|rcp_status)\s+(rcp_\w+)\(([^)]*)\)\s*;", src,
                         re.M | re.S):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_signatures_match_the_header():
    """Every ctypes prototype the binding declares has the header's parameter count."""
    from rank_compressed_paged_gb300 import _lib
    decl = _declared_param_counts()
    assert set(decl) == set(_declared_symbols())
    assert set(_lib._SIG) == set(decl)            # and the binding covers all of them
    for name, (_, args) in _lib._SIG.items():
        assert len(args) == decl[name], (name, len(args), decl[name])
