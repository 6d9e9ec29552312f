"""GPU chunked-prefill attention vs the oracle, through the C ABI (needs a GB300)."""
import numpy as np
import pytest

import workloads as wl
from oracle import rcp_oracle as orc
from tests.gpu_util import assert_close, make_cache, t

pytestmark = pytest.mark.gpu

TINY = wl.SHAPES["tiny"]
MAIN = wl.SHAPES["mha32"]


VARIANTS = ["rank", "reconstruct"]


def _run(inp, variant="rank"):
    import torch
    c = inp.cache
    cache = make_cache(inp.shape, inp.U_k, inp.W_v, c.k_pages, c.v_pages)
    cache.append_kv(t(inp.k), t(inp.v), t(inp.slot_mapping))
    out = cache.prefill_attn(t(inp.q), t(inp.cu_chunk_lens), t(c.block_table),
                             t(inp.seq_lens_after), variant=variant)
    torch.cuda.synchronize()
    assert cache.read_device_error() == 0
    kp, vp = orc.append_kv(c.k_pages, c.v_pages, inp.U_k, inp.W_v, inp.k, inp.v,
                           inp.slot_mapping, 16)
    ref = orc.prefill_attn(inp.q, inp.cu_chunk_lens, kp, vp, inp.U_k, inp.W_v, c.block_table,
                           inp.seq_lens_after, 16)
    return out.cpu().numpy(), ref


@pytest.mark.parametrize("variant", VARIANTS)
def test_tiny_prefill_ragged_chunks(variant):
    inp = wl.make_prefill_inputs(TINY, [0, 37, 64, 5], [40, 21, 16, 0], seed=41, fill=np.nan)
    out, ref = _run(inp, variant)
    assert_close(out, ref, what=f"tiny prefill ({variant})")


@pytest.mark.parametrize("variant", VARIANTS)
def test_main_prefill_small(variant):
    inp = wl.make_prefill_inputs(MAIN, [100, 256], [48, 64], seed=42, fill=np.nan)
    out, ref = _run(inp, variant)
    assert_close(out, ref, what=f"main prefill ({variant})")


@pytest.mark.parametrize("variant", VARIANTS)
def test_main_prefill_multi_tile_chunks(variant):
    """Chunks longer than one 128-row tile, priors off block boundaries, a zero chunk."""
    inp = wl.make_prefill_inputs(MAIN, [300, 0, 17, 40], [200, 130, 0, 129], seed=43,
                                 fill=np.nan)
    out, ref = _run(inp, variant)
    assert_close(out, ref, what=f"main prefill multi-tile ({variant})")


@pytest.mark.parametrize("variant", VARIANTS)
def test_prefill_is_deterministic(variant):
    inp = wl.make_prefill_inputs(MAIN, [64, 250], [100, 37], seed=44)
    a, _ = _run(inp, variant)
    b, _ = _run(inp, variant)
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))


def test_prefill_variants_agree_on_a_long_chunk():
    """Above the crossover both formulations give the oracle's result."""
    inp = wl.make_prefill_inputs(MAIN, [512, 77], [300, 260], seed=45, fill=np.nan)
    a, ref = _run(inp, "rank")
    b, _ = _run(inp, "reconstruct")
    assert_close(a, ref, what="rank")
    assert_close(b, ref, what="reconstruct")


@pytest.mark.parametrize("variant", VARIANTS)
def test_prefill_rejects_decreasing_chunk_offsets(variant):
    """cu_chunk_lens = [0, 10, 5, 20]: request 2 would start inside request 0's rows.  The
    plan refuses the whole batch: the length error bit is set and no output row is
    written (the rows keep their NaN fill)."""
    import torch
    from rank_compressed_paged_gb300 import _lib
    inp = wl.make_prefill_inputs(MAIN, [40, 40, 40], [10, 0, 10], seed=46)
    c = inp.cache
    cache = make_cache(inp.shape, inp.U_k, inp.W_v, c.k_pages, c.v_pages)
    q = t(wl.fp16(np.random.default_rng(47).standard_normal((20, 32, 128))))
    cu = t(np.array([0, 10, 5, 20], np.int32))
    lens = t(np.array([50, 40, 50], np.int32))      # within each request's valid blocks
    table = t(c.block_table)
    out = torch.full_like(q, float("nan"))
    cache.prefill_attn(q, cu, table, lens, out=out, variant=variant)
    torch.cuda.synchronize()
    assert cache.read_device_error() & _lib.RCP_DEVERR_BAD_LEN
    assert torch.isnan(out).all()


@pytest.mark.parametrize("variant", VARIANTS)
def test_prefill_rejects_bad_block_ids_on_device(variant):
    """A prior page of request 1 names a block past the pool: the device error word gets
    the bad-block bit, and request 0 (which reads none of request 1's pages) still matches
    the oracle.  (The reconstructing variant copies such a page from row -16, all out of
    bounds, so every stage still completes on its fixed byte count.)"""
    import torch
    from rank_compressed_paged_gb300 import _lib
    inp = wl.make_prefill_inputs(MAIN, [300, 200], [64, 40], seed=47)
    c = inp.cache
    cache = make_cache(inp.shape, inp.U_k, inp.W_v, c.k_pages, c.v_pages)
    cache.append_kv(t(inp.k), t(inp.v), t(inp.slot_mapping))
    table = c.block_table.copy()
    table[1, 2] = c.k_pages.shape[0] + 7              # out of range physical id
    out = cache.prefill_attn(t(inp.q), t(inp.cu_chunk_lens), t(table), t(inp.seq_lens_after),
                             variant=variant)
    torch.cuda.synchronize()
    assert cache.read_device_error() & _lib.RCP_DEVERR_BAD_BLOCK
    kp, vp = orc.append_kv(c.k_pages, c.v_pages, inp.U_k, inp.W_v, inp.k, inp.v,
                           inp.slot_mapping, 16)
    n0 = int(inp.cu_chunk_lens[1])
    ref0 = orc.prefill_attn(inp.q[:n0], inp.cu_chunk_lens[:2], kp, vp, inp.U_k, inp.W_v,
                            c.block_table[:1], inp.seq_lens_after[:1], 16)
    assert_close(out.cpu().numpy()[:n0], ref0, what=f"unaffected request ({variant})")
