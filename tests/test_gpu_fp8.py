"""E4M3 coefficient pages on the GPU vs the oracle, through the C ABI (needs a GB300).

The caches hold E4M3 roundings (oracle encoder) of the seeded fp16 pages; the oracle
decodes the same codes, so decode parity is held to the fp16 path's tolerances."""
import numpy as np
import pytest

import workloads as wl
from oracle import rcp_oracle as orc
from tests.gpu_util import assert_close, t

pytestmark = pytest.mark.gpu

TINY = wl.SHAPES["tiny"]
MAIN = wl.SHAPES["mha32"]


def _fp8_cache(shape, U, W, kp8, vp8):
    from rank_compressed_paged_gb300 import PagedCoeffCache
    return PagedCoeffCache(shape["num_heads"], shape["head_dim"], shape["rank_k"],
                           shape["rank_v"], kp8.shape[0], t(U), t(W), k_pages=t(kp8),
                           v_pages=t(vp8), page_format="fp8_e4m3")


def _codes(pages):
    return orc.e4m3_encode(np.asarray(pages, np.float64))   # NaN slots -> 0x7F


def _decode_case(shape, lens, seed, **kw):
    import torch
    inp = wl.make_decode_inputs(shape, lens, seed=seed, fill=np.nan, **kw)
    c = inp.cache
    kp8, vp8 = _codes(c.k_pages), _codes(c.v_pages)
    cache = _fp8_cache(shape, inp.U_k, inp.W_v, kp8, vp8)
    out = cache.decode_attn(t(inp.q), t(c.block_table), t(c.seq_lens))
    torch.cuda.synchronize()
    assert cache.read_device_error() == 0
    ref = orc.decode_attn(inp.q, orc.e4m3_decode(kp8), orc.e4m3_decode(vp8), inp.U_k, inp.W_v,
                          c.block_table, c.seq_lens, 16)
    return out.cpu().numpy(), ref


def test_fp8_tiny_decode_ragged():
    out, ref = _decode_case(TINY, [0, 1, 15, 16, 17, 100, 256], 81, spare_blocks=3)
    assert np.all(out[0] == 0)
    assert_close(out, ref, what="fp8 tiny")


def test_fp8_main_decode_ragged():
    rng = np.random.default_rng(82)
    lens = list(rng.integers(1, 900, size=9)) + [0, 16, 1024]
    out, ref = _decode_case(MAIN, lens, 82)
    assert_close(out, ref, what="fp8 main ragged")


def test_fp8_one_long_request_over_every_partition():
    out, ref = _decode_case(MAIN, [0, 9000], 83)
    assert_close(out, ref, what="fp8 long request")


def test_fp8_append_matches_the_oracle_codes():
    import torch
    inp = wl.make_decode_inputs(MAIN, [300, 17, 1024, 40], seed=84, append=True, spare_blocks=2)
    c = inp.cache
    kp8, vp8 = _codes(c.k_pages), _codes(c.v_pages)
    cache = _fp8_cache(MAIN, inp.U_k, inp.W_v, kp8, vp8)
    slots = inp.slot_mapping.copy()
    slots[1] = -1
    cache.append_kv(t(inp.new_k), t(inp.new_v), t(slots))
    torch.cuda.synchronize()
    assert cache.read_device_error() == 0
    kg, vg = cache.k_pages.cpu().numpy(), cache.v_pages.cpu().numpy()
    ko, vo = orc.append_kv_fp8(kp8, vp8, inp.U_k, inp.W_v, inp.new_k, inp.new_v, slots, 16)
    for g, o in ((kg, ko), (vg, vo)):
        diff = g != o
        # fp32 accumulation on the GPU vs fp64 here: a code may differ only next to a
        # rounding boundary, and then by one step
        assert diff.mean() < 0.01, diff.mean()
        dg, do = orc.e4m3_decode(g[diff]), orc.e4m3_decode(o[diff])
        step = np.maximum(np.abs(do), 2.0 ** -6) * 2.0 ** -3
        assert np.all(np.abs(dg - do) <= step + 1e-12)
    # untouched slots are bit-exact
    written = {int(s) for s in slots if s >= 0}
    for blk in range(kg.shape[0]):
        for off in range(16):
            if blk * 16 + off not in written:
                assert np.array_equal(kg[blk, :, off], kp8[blk, :, off])
                assert np.array_equal(vg[blk, off], vp8[blk, off])


def test_fp8_append_with_selection_factors_is_bit_exact():
    import torch
    H, d, rk, R = 4, 64, 16, 64
    rng = np.random.default_rng(85)
    U, W = wl.selection_factors(rng, H, d, rk, R)
    k = wl.fp16(rng.standard_normal((40, H, d)) * 200)   # some values saturate at 448
    v = wl.fp16(rng.standard_normal((40, H, d)))
    slots = rng.permutation(6 * 16)[:40].astype(np.int64)
    kp8 = np.full((6, H, 16, rk), 0x55, np.uint8)
    vp8 = np.full((6, 16, R), 0x55, np.uint8)
    cache = _fp8_cache(TINY, U, W, kp8, vp8)
    cache.append_kv(t(k), t(v), t(slots))
    torch.cuda.synchronize()
    ko, vo = orc.append_kv_fp8(kp8, vp8, U, W, k, v, slots, 16)
    assert np.array_equal(cache.k_pages.cpu().numpy(), ko)
    assert np.array_equal(cache.v_pages.cpu().numpy(), vo)


@pytest.mark.parametrize("shape_name,T,nb", [("tiny", 40, 6), ("mha32", 64, 80),
                                             ("mha32", 300, 40)])
def test_fp8_append_pair_sum_factors_round_to_nearest_even_bit_exact(shape_name, T, nb):
    """Pair-sum factors on narrow-range inputs: every fp32 sum the kernel forms is exact,
    so its conversion to E4M3 is the only rounding and the codes must equal the oracle's
    fp64 -> E4M3 round-to-nearest-even codes bit for bit (split-K cluster path at T = 64,
    256-token tiles at T = 300)."""
    import torch
    shape = wl.SHAPES[shape_name]
    H, d, rk, R = shape["num_heads"], shape["head_dim"], shape["rank_k"], shape["rank_v"]
    rng = np.random.default_rng(91 + T)
    U, W = wl.pair_sum_factors(rng, H, d, rk, R)
    k = wl.fp16_narrow(rng, (T, H, d))
    v = wl.fp16_narrow(rng, (T, H, d))
    slots = np.array([int(s) if i % 9 else -1 for i, s in
                      enumerate(rng.permutation(nb * 16)[:T])], np.int64)
    kp8 = np.full((nb, H, 16, rk), 0x55, np.uint8)
    vp8 = np.full((nb, 16, R), 0x55, np.uint8)
    cache = _fp8_cache(shape, U, W, kp8, vp8)
    cache.append_kv(t(k), t(v), t(slots))
    torch.cuda.synchronize()
    assert cache.read_device_error() == 0
    ko, vo = orc.append_kv_fp8(kp8, vp8, U, W, k, v, slots, 16)
    # the case exercises rounding: most exact sums fall between two E4M3 codes
    ex = np.einsum("hkd,thd->thk", U.astype(np.float64), k.astype(np.float64))
    assert np.mean(orc.e4m3_decode(orc.e4m3_encode(ex)) != ex) > 0.5
    assert np.array_equal(cache.k_pages.cpu().numpy(), ko)
    assert np.array_equal(cache.v_pages.cpu().numpy(), vo)


def test_fp8_decode_step_equals_append_then_decode():
    import torch
    inp = wl.make_decode_inputs(MAIN, [300, 17, 1024, 0], seed=86, append=True)
    c = inp.cache
    kp8, vp8 = _codes(c.k_pages), _codes(c.v_pages)
    # coordinate-selection factors: the appended codes are exact on both sides, so the
    # oracle's own append gives the GPU's pages
    U, W = wl.selection_factors(np.random.default_rng(186), 32, 128, 64, 1024)
    a = _fp8_cache(MAIN, U, W, kp8, vp8)
    a.append_kv(t(inp.new_k), t(inp.new_v), t(inp.slot_mapping))
    oa = a.decode_attn(t(inp.q), t(c.block_table), t(c.seq_lens))
    b = _fp8_cache(MAIN, U, W, kp8, vp8)
    ob = b.decode_step(t(inp.new_k), t(inp.new_v), t(inp.slot_mapping), t(inp.q),
                       t(c.block_table), t(c.seq_lens))
    torch.cuda.synchronize()
    assert np.array_equal(oa.cpu().numpy().view(np.uint16), ob.cpu().numpy().view(np.uint16))
    ko, vo = orc.append_kv_fp8(kp8, vp8, U, W, inp.new_k, inp.new_v, inp.slot_mapping, 16)
    ref = orc.decode_attn(inp.q, orc.e4m3_decode(ko), orc.e4m3_decode(vo), U, W,
                          c.block_table, c.seq_lens, 16)
    assert_close(ob.cpu().numpy(), ref, what="fp8 step")


def test_fp8_rank_space_prefill_on_oracle_pages():
    """The rank-space variant on E4M3 pages: the pages it reads are widened into the
    workspace first; the result is the oracle's on the decoded codes."""
    import torch
    inp = wl.make_prefill_inputs(MAIN, [300, 0, 1024, 17], [64, 130, 3, 1], seed=87, fill=np.nan)
    c = inp.cache
    ko, vo = orc.append_kv_fp8(_codes(c.k_pages), _codes(c.v_pages), inp.U_k, inp.W_v, inp.k,
                               inp.v, inp.slot_mapping, 16)
    cache = _fp8_cache(MAIN, inp.U_k, inp.W_v, ko, vo)
    out = cache.prefill_attn(t(inp.q), t(inp.cu_chunk_lens), t(c.block_table),
                             t(inp.seq_lens_after), variant="rank")
    torch.cuda.synchronize()
    assert cache.read_device_error() == 0
    ref = orc.prefill_attn(inp.q, inp.cu_chunk_lens, orc.e4m3_decode(ko), orc.e4m3_decode(vo),
                           inp.U_k, inp.W_v, c.block_table, inp.seq_lens_after, 16)
    assert_close(out.cpu().numpy(), ref, what="fp8 rank-space prefill")


@pytest.mark.parametrize("shape,prior,chunk,seed", [
    (TINY, [37, 0, 100, 5], [21, 16, 40, 0], 88),
    (MAIN, [300, 0, 1024, 17], [64, 130, 3, 1], 89),
])
def test_fp8_prefill_on_oracle_pages(shape, prior, chunk, seed):
    """Every page, the chunk's included, holds the oracle's own E4M3 codes; the GPU runs
    the prefill alone (widening pass, reconstruction, attention)."""
    import torch
    inp = wl.make_prefill_inputs(shape, prior, chunk, seed=seed, fill=np.nan)
    c = inp.cache
    ko, vo = orc.append_kv_fp8(_codes(c.k_pages), _codes(c.v_pages), inp.U_k, inp.W_v, inp.k,
                               inp.v, inp.slot_mapping, 16)
    cache = _fp8_cache(shape, inp.U_k, inp.W_v, ko, vo)
    out = cache.prefill_attn(t(inp.q), t(inp.cu_chunk_lens), t(c.block_table),
                             t(inp.seq_lens_after))
    torch.cuda.synchronize()
    assert cache.read_device_error() == 0
    ref = orc.prefill_attn(inp.q, inp.cu_chunk_lens, orc.e4m3_decode(ko), orc.e4m3_decode(vo),
                           inp.U_k, inp.W_v, c.block_table, inp.seq_lens_after, 16)
    assert_close(out.cpu().numpy(), ref, what="fp8 prefill")
    # the pages themselves are untouched by the widening pass
    assert np.array_equal(cache.k_pages.cpu().numpy(), ko)
    assert np.array_equal(cache.v_pages.cpu().numpy(), vo)


def test_fp8_prefill_after_its_own_append():
    """Chunk appended by the GPU (selection factors: exact codes), then the prefill."""
    import torch
    inp = wl.make_prefill_inputs(MAIN, [500, 64, 0], [100, 33, 16], seed=90, fill=np.nan)
    c = inp.cache
    U, W = wl.selection_factors(np.random.default_rng(190), 32, 128, 64, 1024)
    kp8, vp8 = _codes(c.k_pages), _codes(c.v_pages)
    cache = _fp8_cache(MAIN, U, W, kp8, vp8)
    cache.append_kv(t(inp.k), t(inp.v), t(inp.slot_mapping))
    out = cache.prefill_attn(t(inp.q), t(inp.cu_chunk_lens), t(c.block_table),
                             t(inp.seq_lens_after))
    torch.cuda.synchronize()
    assert cache.read_device_error() == 0
    ko, vo = orc.append_kv_fp8(kp8, vp8, U, W, inp.k, inp.v, inp.slot_mapping, 16)
    ref = orc.prefill_attn(inp.q, inp.cu_chunk_lens, orc.e4m3_decode(ko), orc.e4m3_decode(vo),
                           U, W, c.block_table, inp.seq_lens_after, 16)
    assert_close(out.cpu().numpy(), ref, what="fp8 prefill after append")
