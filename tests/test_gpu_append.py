"""GPU append (project + scatter) vs the oracle, through the C ABI (needs a GB300).

Indices are checked bit-exactly (every slot not written keeps its sentinel bits);
coefficient values agree with the oracle's fp64 -> fp16 rounding to within one fp16 ulp
plus the fp32 accumulation error bound (nearly all within one ulp), and exactly when the
factors are coordinate selections (projection is then a copy).
"""
import numpy as np
import pytest

import workloads as wl
from oracle import rcp_oracle as orc
from tests.gpu_util import fp16_ulp_diff, make_cache, t

pytestmark = pytest.mark.gpu

TINY = wl.SHAPES["tiny"]
MAIN = wl.SHAPES["mha32"]
SENTINEL = np.float16(np.nan)     # 0x7E00


def _append(shape, U, W, kp, vp, k, v, slots):
    import torch
    cache = make_cache(shape, U, W, kp, vp)
    cache.append_kv(t(k), t(v), t(np.asarray(slots, np.int64)))
    torch.cuda.synchronize()
    return cache.k_pages.cpu().numpy(), cache.v_pages.cpu().numpy(), cache


def _gamma(n):
    u = 2.0 ** -24                      # fp32 unit roundoff
    return n * u / (1 - n * u)


def _check(shape, U, W, nb, T, slots, seed, exact=False):
    """Written coefficients: |gpu - oracle| <= one fp16 ulp + the fp32 dot-product error
    bound gamma_n * sum_i |a_i b_i| (n = d for keys, H*d for values); exact when the
    factors are coordinate selections (a single nonzero product per output)."""
    H, d, rk, R = shape["num_heads"], shape["head_dim"], shape["rank_k"], shape["rank_v"]
    rng = np.random.default_rng(seed)
    kp = np.full((nb, H, 16, rk), SENTINEL, np.float16)
    vp = np.full((nb, 16, R), SENTINEL, np.float16)
    k = wl.fp16(rng.standard_normal((T, H, d)))
    v = wl.fp16(rng.standard_normal((T, H, d)))
    gk, gv, cache = _append(shape, U, W, kp, vp, k, v, slots)
    assert cache.read_device_error() == 0
    ok_, ov = orc.append_kv(kp, vp, U, W, k, v, slots, 16)
    # untouched slots: identical bits (NaN sentinel compared as integers)
    kn = np.isnan(ok_)
    vn = np.isnan(ov)
    assert np.array_equal(np.isnan(gk), kn) and np.array_equal(np.isnan(gv), vn)
    assert np.array_equal(gk.view(np.uint16)[kn], ok_.view(np.uint16)[kn])
    assert np.array_equal(gv.view(np.uint16)[vn], ov.view(np.uint16)[vn])
    Ua = np.abs(U.astype(np.float64))
    Wa = np.abs(W.astype(np.float64))
    for i, s in enumerate(slots):
        if s < 0:
            continue
        blk, off = s // 16, s % 16
        g_k, r_k = gk[blk, :, off, :], ok_[blk, :, off, :]
        g_v, r_v = gv[blk, off, :], ov[blk, off, :]
        if exact:
            assert np.array_equal(g_k.view(np.uint16), r_k.view(np.uint16))
            assert np.array_equal(g_v.view(np.uint16), r_v.view(np.uint16))
            continue
        sk = np.einsum("hkd,hd->hk", Ua, np.abs(k[i].astype(np.float64)))
        sv = Wa @ np.abs(v[i].astype(np.float64)).reshape(-1)
        tol_k = np.spacing(np.abs(r_k)).astype(np.float64) + _gamma(d) * sk
        tol_v = np.spacing(np.abs(r_v)).astype(np.float64) + _gamma(H * d) * sv
        assert np.all(np.abs(g_k.astype(np.float64) - r_k) <= tol_k), i
        assert np.all(np.abs(g_v.astype(np.float64) - r_v) <= tol_v), i
        # and almost everywhere within one ulp
        assert np.mean(fp16_ulp_diff(g_v, r_v) <= 1) > 0.99


def test_append_tiny_random_factors():
    rng = np.random.default_rng(31)
    U, W = wl.make_factors(rng, 4, 64, 16, 64)
    slots = [5, 17, -1, 100, 63, 64, 0, 127, -1, 33]
    _check(TINY, U, W, 8, len(slots), slots, seed=32)


def test_append_tiny_selection_factors_bit_exact():
    rng = np.random.default_rng(33)
    U, W = wl.selection_factors(rng, 4, 64, 16, 64)
    slots = list(rng.permutation(96)[:40])
    _check(TINY, U, W, 6, len(slots), slots, seed=34, exact=True)


def test_append_main_decode_step_shape():
    """One token per sequence for 64 sequences (the batch-64 decode step's append)."""
    rng = np.random.default_rng(35)
    U, W = wl.make_factors(rng, 32, 128, 64, 1024)
    slots = list(rng.permutation(80 * 16)[:64])
    _check(MAIN, U, W, 80, 64, slots, seed=36)


def test_append_main_chunk_with_skips():
    rng = np.random.default_rng(37)
    U, W = wl.selection_factors(rng, 32, 128, 64, 1024)
    slots = [int(s) if i % 7 else -1 for i, s in enumerate(rng.permutation(40 * 16)[:300])]
    _check(MAIN, U, W, 40, 300, slots, seed=38, exact=True)


def test_append_bad_slot_sets_error_and_writes_nothing():
    import torch
    from rank_compressed_paged_gb300 import _lib
    rng = np.random.default_rng(39)
    U, W = wl.make_factors(rng, 4, 64, 16, 64)
    kp = np.full((2, 4, 16, 16), SENTINEL, np.float16)
    vp = np.full((2, 16, 64), SENTINEL, np.float16)
    k = wl.fp16(rng.standard_normal((1, 4, 64)))
    gk, gv, cache = _append(TINY, U, W, kp, vp, k, k, [32])     # 2 blocks -> slots 0..31
    torch.cuda.synchronize()
    assert cache.read_device_error() & _lib.RCP_DEVERR_BAD_SLOT
    assert np.all(np.isnan(gk)) and np.all(np.isnan(gv))


def test_append_then_decode_round_trip():
    """Prefilled cache + appended last token (the batch-64 step, small): decode parity."""
    import torch
    from tests.gpu_util import assert_close
    inp = wl.make_decode_inputs(MAIN, [300, 17, 1024], seed=40, append=True, fill=np.nan)
    c = inp.cache
    cache = make_cache(inp.shape, inp.U_k, inp.W_v, c.k_pages, c.v_pages)
    cache.append_kv(t(inp.new_k), t(inp.new_v), t(inp.slot_mapping))
    out = cache.decode_attn(t(inp.q), t(c.block_table), t(c.seq_lens))
    torch.cuda.synchronize()
    kp, vp = orc.append_kv(c.k_pages, c.v_pages, inp.U_k, inp.W_v, inp.new_k, inp.new_v,
                           inp.slot_mapping, 16)
    ref = orc.decode_attn(inp.q, kp, vp, inp.U_k, inp.W_v, c.block_table, c.seq_lens, 16)
    assert_close(out.cpu().numpy(), ref, what="append+decode")


def test_decode_step_equals_append_then_decode():
    """The fused step queues the same work: outputs and pages are bitwise identical."""
    import torch
    inp = wl.make_decode_inputs(MAIN, [300, 17, 1024, 0], seed=41, append=True, fill=np.nan)
    c = inp.cache
    a = make_cache(inp.shape, inp.U_k, inp.W_v, c.k_pages, c.v_pages)
    a.append_kv(t(inp.new_k), t(inp.new_v), t(inp.slot_mapping))
    oa = a.decode_attn(t(inp.q), t(c.block_table), t(c.seq_lens))
    b = make_cache(inp.shape, inp.U_k, inp.W_v, c.k_pages, c.v_pages)
    ob = b.decode_step(t(inp.new_k), t(inp.new_v), t(inp.slot_mapping), t(inp.q),
                       t(c.block_table), t(c.seq_lens))
    torch.cuda.synchronize()
    assert a.read_device_error() == 0 and b.read_device_error() == 0
    assert np.array_equal(oa.cpu().numpy().view(np.uint16), ob.cpu().numpy().view(np.uint16))
    assert np.array_equal(a.k_pages.cpu().numpy().view(np.uint16),
                          b.k_pages.cpu().numpy().view(np.uint16))
    assert np.array_equal(a.v_pages.cpu().numpy().view(np.uint16),
                          b.v_pages.cpu().numpy().view(np.uint16))
