"""GPU chunked prefill step (rcp_prefill_step): the append of the chunk's keys and values and
the chunk attention queued as one step, against the same two calls made one after the other
and against the oracle (needs a GB300)."""
import numpy as np
import pytest

import workloads as wl
from oracle import rcp_oracle as orc
from tests.gpu_util import assert_close, make_cache, t

pytestmark = pytest.mark.gpu

TINY = wl.SHAPES["tiny"]
MAIN = wl.SHAPES["mha32"]
VARIANTS = ["rank", "reconstruct"]


def _both(inp, variant, page_format="fp16", U=None, W=None, kp=None, vp=None):
    """Outputs and pages of (a) append_kv + prefill_attn and (b) prefill_step, each on its
    own device copy of the same starting pages."""
    import torch
    from rank_compressed_paged_gb300 import PagedCoeffCache
    c = inp.cache
    U = inp.U_k if U is None else U
    W = inp.W_v if W is None else W
    kp = c.k_pages if kp is None else kp
    vp = c.v_pages if vp is None else vp
    res = []
    for fused in (False, True):
        sh = inp.shape
        cache = PagedCoeffCache(sh["num_heads"], sh["head_dim"], sh["rank_k"], sh["rank_v"],
                                kp.shape[0], t(U), t(W), k_pages=t(kp), v_pages=t(vp),
                                page_format=page_format)
        args = (t(inp.q), t(inp.cu_chunk_lens), t(c.block_table), t(inp.seq_lens_after))
        if fused:
            out = cache.prefill_step(t(inp.k), t(inp.v), t(inp.slot_mapping), *args,
                                     variant=variant)
        else:
            cache.append_kv(t(inp.k), t(inp.v), t(inp.slot_mapping))
            out = cache.prefill_attn(*args, variant=variant)
        torch.cuda.synchronize()
        assert cache.read_device_error() == 0
        res.append((out.cpu().numpy(), cache.k_pages.cpu().numpy(), cache.v_pages.cpu().numpy()))
    return res


def _check_same(res, what):
    (o1, k1, v1), (o2, k2, v2) = res
    assert np.array_equal(k1.view(np.uint8), k2.view(np.uint8)), f"{what}: K pages differ"
    assert np.array_equal(v1.view(np.uint8), v2.view(np.uint8)), f"{what}: V pages differ"
    assert np.array_equal(o1.view(np.uint16), o2.view(np.uint16)), f"{what}: outputs differ"


@pytest.mark.parametrize("variant", VARIANTS)
def test_tiny_prefill_step_equals_append_then_prefill(variant):
    inp = wl.make_prefill_inputs(TINY, [0, 37, 64, 5], [40, 21, 16, 0], seed=141, fill=np.nan)
    res = _both(inp, variant)
    _check_same(res, f"tiny ({variant})")
    c = inp.cache
    kp, vp = orc.append_kv(c.k_pages, c.v_pages, inp.U_k, inp.W_v, inp.k, inp.v,
                           inp.slot_mapping, 16)
    ref = orc.prefill_attn(inp.q, inp.cu_chunk_lens, kp, vp, inp.U_k, inp.W_v, c.block_table,
                           inp.seq_lens_after, 16)
    assert_close(res[1][0], ref, what=f"tiny prefill step ({variant})")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("prior,chunk", [([100, 256], [48, 64]),            # 112 rows: 64-row tiles
                                         ([300, 0, 17, 40], [200, 130, 0, 129]),   # 459: 256-row
                                         ([33], [7])])                       # 7 rows: 16-row tiles
def test_main_prefill_step_equals_append_then_prefill(variant, prior, chunk):
    """The query projection takes the append launch's tile size (16, 64 or 256 rows); each
    query's projection is the same sum of products either way, so the results are equal bit
    for bit, and both match the oracle."""
    inp = wl.make_prefill_inputs(MAIN, prior, chunk, seed=142 + sum(chunk), fill=np.nan)
    res = _both(inp, variant)
    _check_same(res, f"main {chunk} ({variant})")
    c = inp.cache
    kp, vp = orc.append_kv(c.k_pages, c.v_pages, inp.U_k, inp.W_v, inp.k, inp.v,
                           inp.slot_mapping, 16)
    ref = orc.prefill_attn(inp.q, inp.cu_chunk_lens, kp, vp, inp.U_k, inp.W_v, c.block_table,
                           inp.seq_lens_after, 16)
    assert_close(res[1][0], ref, what=f"main prefill step {chunk} ({variant})")


def test_fp8_prefill_step_equals_append_then_prefill():
    """E4M3 pages (the step widens them after its append)."""
    inp = wl.make_prefill_inputs(MAIN, [500, 64, 0], [100, 33, 16], seed=190, fill=np.nan)
    c = inp.cache
    U, W = wl.selection_factors(np.random.default_rng(191), 32, 128, 64, 1024)
    kp8 = orc.e4m3_encode(np.asarray(c.k_pages, np.float64))
    vp8 = orc.e4m3_encode(np.asarray(c.v_pages, np.float64))
    res = _both(inp, "reconstruct", page_format="fp8_e4m3", U=U, W=W, kp=kp8, vp=vp8)
    _check_same(res, "fp8")
    ko, vo = orc.append_kv_fp8(kp8, vp8, U, W, inp.k, inp.v, inp.slot_mapping, 16)
    ref = orc.prefill_attn(inp.q, inp.cu_chunk_lens, orc.e4m3_decode(ko), orc.e4m3_decode(vo),
                           U, W, c.block_table, inp.seq_lens_after, 16)
    assert_close(res[1][0], ref, what="fp8 prefill step")


def test_prefill_step_rejects_an_unknown_variant_code():
    """reconstruct must be 0 or 1: refused before any launch."""
    import ctypes
    from rank_compressed_paged_gb300 import _lib
    inp = wl.make_prefill_inputs(TINY, [8], [8], seed=143)
    c = inp.cache
    cache = make_cache(TINY, inp.U_k, inp.W_v, c.k_pages, c.v_pages)
    q, k, v = t(inp.q), t(inp.k), t(inp.v)
    sl, cu, bt, ln = (t(inp.slot_mapping), t(inp.cu_chunk_lens), t(c.block_table),
                      t(inp.seq_lens_after))
    out = q.clone()
    ws = cache.workspace(8, cache.reconstruct_workspace_bytes(8, 1, int(bt.shape[1])))
    st = cache._lib.rcp_prefill_step(
        cache._h, k.data_ptr(), v.data_ptr(), sl.data_ptr(), 8, q.data_ptr(), cu.data_ptr(), 8,
        bt.data_ptr(), int(bt.shape[1]), ln.data_ptr(), 1, 2, out.data_ptr(), ws.data_ptr(),
        ctypes.c_size_t(ws.numel()), None)
    assert st == _lib.RCP_ERR_INVALID_ARG
