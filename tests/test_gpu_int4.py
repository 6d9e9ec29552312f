"""4-bit coefficient pages on the GPU vs the oracle, through the C ABI (needs a GB300).

The pages hold the oracle's own 4-bit encoding (codes and fp16 scales) of the seeded
coefficients; the oracle reads the same bytes back as code * scale, so decode parity is
held to the fp16 path's tolerances.  Appends are compared byte for byte where every fp32
sum the kernel forms is exact (selection and pair-sum factors), and within one code step
elsewhere."""
import numpy as np
import pytest

import workloads as wl
from oracle import rcp_oracle as orc
from tests.gpu_util import assert_close, t

pytestmark = pytest.mark.gpu

TINY = wl.SHAPES["tiny"]
MAIN = wl.SHAPES["mha32"]


def _dims(shape):
    return shape["num_heads"], shape["head_dim"], shape["rank_k"], shape["rank_v"]


def _int4_cache(shape, U, W, kb, vb):
    from rank_compressed_paged_gb300 import PagedCoeffCache
    H, d, rk, R = _dims(shape)
    return PagedCoeffCache(H, d, rk, R, kb.shape[0], t(U), t(W), k_pages=t(kb), v_pages=t(vb),
                           page_format="int4")


def _bytes(shape, k_pages, v_pages):
    """Byte pages holding the oracle's 4-bit encoding of fp16/fp64 coefficient pages; a slot
    filled with NaN gets codes 0 and a NaN scale, so reading it would poison the output."""
    with np.errstate(invalid="ignore"):
        kc, ks, vc, vs = orc.int4_pages(k_pages, v_pages)
    return orc.int4_pack_pages(kc, ks, vc, vs)


def _values(shape, kb, vb):
    H, _, rk, R = _dims(shape)
    return orc.int4_page_coefficients(kb, vb, H, rk, R)


def test_int4_page_bytes_match_the_oracle_layout():
    from rank_compressed_paged_gb300 import int4_page_bytes
    for shape in (TINY, MAIN):
        H, _, rk, R = _dims(shape)
        assert int4_page_bytes(H, rk, R) == orc.int4_page_bytes(H, rk, R)


def _decode_case(shape, lens, seed, **kw):
    import torch
    inp = wl.make_decode_inputs(shape, lens, seed=seed, fill=np.nan, **kw)
    c = inp.cache
    kb, vb = _bytes(shape, c.k_pages, c.v_pages)
    cache = _int4_cache(shape, inp.U_k, inp.W_v, kb, vb)
    out = cache.decode_attn(t(inp.q), t(c.block_table), t(c.seq_lens))
    torch.cuda.synchronize()
    assert cache.read_device_error() == 0
    kv, vv = _values(shape, kb, vb)
    ref = orc.decode_attn(inp.q, kv, vv, inp.U_k, inp.W_v, c.block_table, c.seq_lens, 16)
    return out.cpu().numpy(), ref


def test_int4_tiny_decode_ragged():
    out, ref = _decode_case(TINY, [0, 1, 15, 16, 17, 100, 256], 181, spare_blocks=3)
    assert np.all(out[0] == 0)
    assert_close(out, ref, what="int4 tiny")


def test_int4_main_decode_ragged():
    rng = np.random.default_rng(182)
    lens = list(rng.integers(1, 900, size=9)) + [0, 16, 1024]
    out, ref = _decode_case(MAIN, lens, 182)
    assert_close(out, ref, what="int4 main ragged")


def test_int4_one_long_request_over_every_partition():
    out, ref = _decode_case(MAIN, [0, 9000], 183)
    assert_close(out, ref, what="int4 long request")


def _append_case(shape, U, W, k, v, slots, nb, seed):
    """Pages of random bytes (finite scales), an append on the GPU and the oracle's."""
    import torch
    H, _, rk, R = _dims(shape)
    kbytes, vbytes = orc.int4_page_bytes(H, rk, R)
    rng = np.random.default_rng(seed)
    kb = rng.integers(0, 256, size=(nb, kbytes), dtype=np.uint8)
    vb = rng.integers(0, 256, size=(nb, vbytes), dtype=np.uint8)
    kc, ks, vc, vs = orc.int4_unpack_pages(kb, vb, H, rk, R)
    kb, vb = orc.int4_pack_pages(kc, np.full_like(ks, 0.5), vc, np.full_like(vs, 0.25))
    cache = _int4_cache(shape, U, W, kb, vb)
    cache.append_kv(t(k), t(v), t(slots))
    torch.cuda.synchronize()
    assert cache.read_device_error() == 0
    ko, vo = orc.append_kv_int4(kb, vb, U, W, k, v, slots, 16)
    return cache.k_pages.cpu().numpy(), cache.v_pages.cpu().numpy(), ko, vo, kb, vb


def test_int4_append_with_selection_factors_is_bit_exact():
    H, d, rk, R = _dims(TINY)
    rng = np.random.default_rng(185)
    U, W = wl.selection_factors(rng, H, d, rk, R)
    k = wl.fp16(rng.standard_normal((40, H, d)) * 3)
    v = wl.fp16(rng.standard_normal((40, H, d)))
    k[3] = 0.0                                     # an all-zero group: scale 0, codes 0
    slots = rng.permutation(6 * 16)[:40].astype(np.int64)
    slots[5] = -1
    kg, vg, ko, vo, _, _ = _append_case(TINY, U, W, k, v, slots, 6, 1185)
    assert np.array_equal(kg, ko)
    assert np.array_equal(vg, vo)


@pytest.mark.parametrize("shape_name,T,nb", [("tiny", 40, 6), ("mha32", 16, 20),
                                             ("mha32", 64, 80), ("mha32", 300, 40)])
def test_int4_append_pair_sum_factors_bit_exact(shape_name, T, nb):
    """Pair-sum factors on narrow-range inputs: the group maxima and the quotients are exact
    on both sides, so scales (smallest fp16 with 7 * scale >= max |x|) and codes (nearest,
    ties to even) must match the oracle byte for byte: 16-token tiles at T = 16, the
    split-K cluster path at T = 64, 256-token tiles at T = 300."""
    shape = wl.SHAPES[shape_name]
    H, d, rk, R = _dims(shape)
    rng = np.random.default_rng(191 + T)
    U, W = wl.pair_sum_factors(rng, H, d, rk, R)
    k = wl.fp16_narrow(rng, (T, H, d))
    v = wl.fp16_narrow(rng, (T, H, d))
    slots = np.array([int(s) if i % 9 else -1 for i, s in
                      enumerate(rng.permutation(nb * 16)[:T])], np.int64)
    kg, vg, ko, vo, _, _ = _append_case(shape, U, W, k, v, slots, nb, 1191 + T)
    assert np.array_equal(kg, ko)
    assert np.array_equal(vg, vo)


def test_int4_append_random_factors_within_one_code_step():
    """Seeded low-rank factors: the GPU sums in fp32, the oracle in fp64, so a code may differ
    by one step next to a rounding boundary and a scale by one fp16 step next to a binade
    of 7 * scale; everything else is equal."""
    inp = wl.make_decode_inputs(MAIN, [300, 17, 1024, 40], seed=184, append=True,
                                spare_blocks=2)
    H, _, rk, R = _dims(MAIN)
    nb = inp.cache.k_pages.shape[0]
    slots = inp.slot_mapping.copy()
    slots[1] = -1
    kg, vg, ko, vo, _, _ = _append_case(MAIN, inp.U_k, inp.W_v, inp.new_k, inp.new_v, slots,
                                        nb, 1184)
    gk = orc.int4_unpack_pages(kg, vg, H, rk, R)
    ok = orc.int4_unpack_pages(ko, vo, H, rk, R)
    for g, o in zip(gk, ok):
        if g.dtype == np.float16:
            ulp = np.abs(g.view(np.int16).astype(np.int32) - o.view(np.int16).astype(np.int32))
            assert ulp.max() <= 1 and ulp.mean() < 0.01, (ulp.max(), ulp.mean())
        else:
            diff = np.abs(g.astype(np.int32) - o.astype(np.int32))
            assert diff.max() <= 1 and diff.mean() < 0.01, (diff.max(), diff.mean())


def test_int4_decode_step_equals_append_then_decode():
    import torch
    inp = wl.make_decode_inputs(MAIN, [300, 17, 1024, 0], seed=186, append=True)
    c = inp.cache
    kb, vb = _bytes(MAIN, c.k_pages, c.v_pages)
    # pair-sum factors on narrow inputs: the appended bytes are exact on both sides, so the
    # oracle's own append gives the GPU's pages.  Inputs below 1 keep the appended
    # coefficients at the magnitude of the others (the kernel widens each value to
    # fp16(code * scale), a relative rounding of 2^-12 that the tolerance is set for).
    rng = np.random.default_rng(286)
    U, W = wl.pair_sum_factors(rng, 32, 128, 64, 1024)
    nk = wl.fp16_narrow(rng, inp.new_k.shape, emin=-6, emax=-1)
    nv = wl.fp16_narrow(rng, inp.new_v.shape, emin=-6, emax=-1)
    a = _int4_cache(MAIN, U, W, kb, vb)
    a.append_kv(t(nk), t(nv), t(inp.slot_mapping))
    oa = a.decode_attn(t(inp.q), t(c.block_table), t(c.seq_lens))
    b = _int4_cache(MAIN, U, W, kb, vb)
    ob = b.decode_step(t(nk), t(nv), t(inp.slot_mapping), t(inp.q), t(c.block_table),
                       t(c.seq_lens))
    torch.cuda.synchronize()
    assert b.read_device_error() == 0
    assert np.array_equal(oa.cpu().numpy().view(np.uint16), ob.cpu().numpy().view(np.uint16))
    ko, vo = orc.append_kv_int4(kb, vb, U, W, nk, nv, inp.slot_mapping, 16)
    assert np.array_equal(b.k_pages.cpu().numpy(), ko)
    assert np.array_equal(b.v_pages.cpu().numpy(), vo)
    kv, vv = _values(MAIN, ko, vo)
    ref = orc.decode_attn(inp.q, kv, vv, U, W, c.block_table, c.seq_lens, 16)
    assert_close(ob.cpu().numpy(), ref, what="int4 step")


@pytest.mark.parametrize("variant", ["reconstruct", "rank"])
@pytest.mark.parametrize("shape,prior,chunk,seed", [
    (TINY, [37, 0, 100, 5], [21, 16, 40, 0], 188),
    (MAIN, [300, 0, 1024, 17], [64, 130, 3, 1], 189),
])
def test_int4_prefill_on_oracle_pages(shape, prior, chunk, seed, variant):
    """Every page, the chunk's included, holds the oracle's 4-bit encoding (its own append of
    the chunk); the GPU runs the prefill alone (widening pass, then the reconstruction and
    attention, or the rank-space attention) and the oracle attends the values code x
    scale."""
    import torch
    inp = wl.make_prefill_inputs(shape, prior, chunk, seed=seed, fill=np.nan)
    c = inp.cache
    kb, vb = _bytes(shape, c.k_pages, c.v_pages)
    ko, vo = orc.append_kv_int4(kb, vb, inp.U_k, inp.W_v, inp.k, inp.v, inp.slot_mapping, 16)
    cache = _int4_cache(shape, inp.U_k, inp.W_v, ko, vo)
    out = cache.prefill_attn(t(inp.q), t(inp.cu_chunk_lens), t(c.block_table),
                             t(inp.seq_lens_after), variant=variant)
    torch.cuda.synchronize()
    assert cache.read_device_error() == 0
    kv, vv = _values(shape, ko, vo)
    ref = orc.prefill_attn(inp.q, inp.cu_chunk_lens, kv, vv, inp.U_k, inp.W_v, c.block_table,
                           inp.seq_lens_after, 16)
    assert_close(out.cpu().numpy(), ref, what="int4 prefill")
    # the pages themselves are untouched by the widening pass
    assert np.array_equal(cache.k_pages.cpu().numpy(), ko)
    assert np.array_equal(cache.v_pages.cpu().numpy(), vo)


def test_int4_prefill_after_its_own_append():
    """Chunk appended by the GPU with pair-sum factors on narrow inputs (bytes exact on both
    sides), then the prefill."""
    import torch
    inp = wl.make_prefill_inputs(MAIN, [500, 64, 0], [100, 33, 16], seed=190, fill=np.nan)
    c = inp.cache
    rng = np.random.default_rng(290)
    U, W = wl.pair_sum_factors(rng, 32, 128, 64, 1024)
    k = wl.fp16_narrow(rng, inp.k.shape, emin=-6, emax=-1)
    v = wl.fp16_narrow(rng, inp.v.shape, emin=-6, emax=-1)
    kb, vb = _bytes(MAIN, c.k_pages, c.v_pages)
    cache = _int4_cache(MAIN, U, W, kb, vb)
    cache.append_kv(t(k), t(v), t(inp.slot_mapping))
    out = cache.prefill_attn(t(inp.q), t(inp.cu_chunk_lens), t(c.block_table),
                             t(inp.seq_lens_after))
    torch.cuda.synchronize()
    assert cache.read_device_error() == 0
    ko, vo = orc.append_kv_int4(kb, vb, U, W, k, v, inp.slot_mapping, 16)
    assert np.array_equal(cache.k_pages.cpu().numpy(), ko)
    assert np.array_equal(cache.v_pages.cpu().numpy(), vo)
    kv, vv = _values(MAIN, ko, vo)
    ref = orc.prefill_attn(inp.q, inp.cu_chunk_lens, kv, vv, U, W, c.block_table,
                           inp.seq_lens_after, 16)
    assert_close(out.cpu().numpy(), ref, what="int4 prefill after append")


@pytest.mark.parametrize("shape_name", ["tiny", "mha32"])
def test_int4_append_bad_slot_sets_error_and_writes_nothing(shape_name):
    """A slot past the pool's capacity flags RCP_DEVERR_BAD_SLOT and leaves every byte of
    the pages as it was (the other token of the call is written)."""
    import torch
    from rank_compressed_paged_gb300 import _lib
    shape = wl.SHAPES[shape_name]
    H, d, rk, R = _dims(shape)
    rng = np.random.default_rng(195)
    U, W = wl.make_factors(rng, H, d, rk, R)
    k = wl.fp16(rng.standard_normal((2, H, d)))
    v = wl.fp16(rng.standard_normal((2, H, d)))
    slots = np.array([2 * 16 + 3, 5], np.int64)        # 2 blocks: slot 35 is past the end
    kbytes, vbytes = orc.int4_page_bytes(H, rk, R)
    kb = rng.integers(0, 256, size=(2, kbytes), dtype=np.uint8)
    vb = rng.integers(0, 256, size=(2, vbytes), dtype=np.uint8)
    cache = _int4_cache(shape, U, W, kb, vb)
    cache.append_kv(t(k), t(v), t(slots))
    torch.cuda.synchronize()
    assert cache.read_device_error() & _lib.RCP_DEVERR_BAD_SLOT
    kg, vg = cache.k_pages.cpu().numpy(), cache.v_pages.cpu().numpy()
    # only slot 5 (block 0, offset 5) may differ from the input pages: its codes and scales
    got = orc.int4_unpack_pages(kg, vg, H, rk, R)
    was = orc.int4_unpack_pages(kb, vb, H, rk, R)
    keep = np.arange(16) != 5
    kc_g, ks_g, vc_g, vs_g = got
    kc_i, ks_i, vc_i, vs_i = was
    assert np.array_equal(kc_g[1], kc_i[1]) and np.array_equal(vc_g[1], vc_i[1])
    assert np.array_equal(ks_g[1].view(np.uint16), ks_i[1].view(np.uint16))
    assert np.array_equal(vs_g[1].view(np.uint16), vs_i[1].view(np.uint16))
    assert np.array_equal(kc_g[0][:, keep], kc_i[0][:, keep])
    assert np.array_equal(ks_g[0][:, keep].view(np.uint16), ks_i[0][:, keep].view(np.uint16))
    assert np.array_equal(vc_g[0][keep], vc_i[0][keep])
    assert np.array_equal(vs_g[0][keep].view(np.uint16), vs_i[0][keep].view(np.uint16))
    assert not np.array_equal(vc_g[0][5], vc_i[0][5]) or not np.array_equal(
        vs_g[0][5].view(np.uint16), vs_i[0][5].view(np.uint16))   # slot 5 was written
