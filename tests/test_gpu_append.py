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


def _check(shape, U, W, nb, T, slots, seed, exact=False, narrow=False):
    """Written coefficients: |gpu - oracle| <= one fp16 ulp + the fp32 dot-product error
    bound gamma_n * sum_i |a_i b_i| (n = d for keys, H*d for values); exact when every
    fp32 sum the kernel forms is exact, so that its fp32 -> fp16 conversion is the only
    rounding (coordinate-selection factors; or pair-sum factors with ``narrow`` inputs)."""
    H, d, rk, R = shape["num_heads"], shape["head_dim"], shape["rank_k"], shape["rank_v"]
    rng = np.random.default_rng(seed)
    kp = np.full((nb, H, 16, rk), SENTINEL, np.float16)
    vp = np.full((nb, 16, R), SENTINEL, np.float16)
    if narrow:
        k = wl.fp16_narrow(rng, (T, H, d))
        v = wl.fp16_narrow(rng, (T, H, d))
    else:
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


def _rounding_counts(U, W, k, v):
    """How many exact projections fp16 cannot hold, and how many of those are ties."""
    ex = np.concatenate([np.einsum("hkd,thd->thk", U.astype(np.float64),
                                   k.astype(np.float64)).ravel(),
                         (v.astype(np.float64).reshape(len(v), -1) @
                          W.astype(np.float64).T).ravel()])
    lo = ex.astype(np.float16)
    inexact = lo.astype(np.float64) != ex
    up = np.nextafter(lo, np.where(lo.astype(np.float64) < ex, np.float16(np.inf),
                                   np.float16(-np.inf)))
    tie = inexact & (np.abs(up.astype(np.float64) - ex) == np.abs(lo.astype(np.float64) - ex))
    return int(inexact.sum()), int(tie.sum())


@pytest.mark.parametrize("shape_name,T,nb", [("tiny", 40, 6), ("mha32", 64, 80),
                                             ("mha32", 300, 40)])
def test_append_pair_sum_factors_round_to_nearest_even_bit_exact(shape_name, T, nb):
    """Every coefficient is the sum of two fp16 inputs whose exact sum fits in fp32, so the
    kernel's fp32 accumulation (tensor-core partial sums, the cluster's split-K reduction)
    is exact and its fp32 -> fp16 conversion is the only rounding: the pages must equal
    the oracle's fp64 -> fp16 round-to-nearest-even bit for bit, ties included.  T = 64
    takes the split-K cluster path, T = 300 the 256-token tiles."""
    shape = wl.SHAPES[shape_name]
    H, d, rk, R = shape["num_heads"], shape["head_dim"], shape["rank_k"], shape["rank_v"]
    rng = np.random.default_rng(41 + T)
    U, W = wl.pair_sum_factors(rng, H, d, rk, R)
    slots = [int(s) if i % 9 else -1 for i, s in enumerate(rng.permutation(nb * 16)[:T])]
    seed = 42 + T
    r2 = np.random.default_rng(seed)
    inexact, ties = _rounding_counts(U, W, wl.fp16_narrow(r2, (T, H, d)),
                                     wl.fp16_narrow(r2, (T, H, d)))
    assert inexact > T * (H * rk + R) // 3 and ties > 20, (inexact, ties)   # rounding happens
    _check(shape, U, W, nb, T, slots, seed=seed, exact=True, narrow=True)


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
