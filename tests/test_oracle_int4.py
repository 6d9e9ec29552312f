"""Pins for the oracle's 4-bit coefficient pages and coefficient rotation (no GPU).

Each ties the functions to a fact outside them: values on the code grid round-trip
exactly; every code is the nearest grid point (found by enumeration, ties to even); the
error is at most half a step and no code saturates; a hand-packed byte fixes the nibble
order; a hand case fixes the upward fp16 rounding of the scale; and rotating the
coefficients while folding the rotation into the factors leaves decode unchanged.  (Whether
a rotation lowers the 4-bit error depends on the data: with one dominant channel the plain
max-scaled code errs only on the small channels, so that is not a pin.)
"""
import numpy as np

import workloads as wl
from oracle import rcp_oracle as orc

TINY = wl.SHAPES["tiny"]


def test_grid_values_round_trip_exactly():
    rng = np.random.default_rng(1)
    s = np.float16(0.3125)                              # exact in fp16
    k = rng.integers(-7, 8, size=(5, 16))
    k[:, 0] = 7                                         # the group max sets the scale
    x = k * np.float64(s)
    c, sc = orc.int4_encode(x, 16)
    assert np.all(sc == s)
    np.testing.assert_array_equal(c, k)
    np.testing.assert_array_equal(orc.int4_decode(c, sc, 16), x)


def test_codes_are_the_nearest_grid_points_by_enumeration():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((40, 8)) * rng.uniform(0.01, 10, size=(40, 1))
    x[3] = 0.0                                           # a zero group
    x[5, :] = [0.5, -0.5, 1.5, 2.5, -2.5, 3.5, 7.0, 0.0]  # exact ties at scale 1
    c, s = orc.int4_encode(x, 8)
    grid = np.arange(-7, 8)
    for g in range(40):
        sg = float(s[g, 0])
        for i in range(8):
            if sg == 0:
                assert c[g, i] == 0
                continue
            d = np.abs(x[g, i] - grid * sg)
            best = grid[d == d.min()]
            want = best[0] if len(best) == 1 else best[best % 2 == 0][0]   # ties to even
            assert c[g, i] == want, (g, i, x[g, i], sg, c[g, i], want)
    assert list(c[5]) == [0, 0, 2, 2, -2, 4, 7, 0]


def test_error_is_at_most_half_a_step_and_codes_never_saturate():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((200, 64)) * np.exp(rng.uniform(-6, 6, size=(200, 1)))
    c, s = orc.int4_encode(x, 64)
    assert np.abs(c).max() <= 7
    s64 = s.astype(np.float64)
    assert np.all(s64 * 7 >= np.abs(x).max(axis=1, keepdims=True))   # no saturation
    err = np.abs(orc.int4_decode(c, s, 64) - x)
    assert np.all(err <= s64 / 2 * (1 + 1e-12))


def test_scale_is_the_fp16_at_or_above_max_over_7():
    x = np.array([[1.0, 0.0, 0.0, 0.0]])                 # 1/7 is not an fp16 value
    c, s = orc.int4_encode(x, 4)
    s0 = float(s[0, 0])
    assert s0 * 7 >= 1.0
    below = float(np.nextafter(np.float16(s0), np.float16(0)))
    assert below * 7 < 1.0                               # the smallest such fp16
    assert c[0, 0] == 7


def test_pack_nibble_order_and_round_trip():
    assert orc.pack_int4(np.array([1, -2], np.int8))[0] == 0xE1   # low nibble first
    assert orc.pack_int4(np.array([-7, 7], np.int8))[0] == 0x79
    a = np.array([[i, j] for i in range(-7, 8) for j in range(-7, 8)], np.int8).reshape(1, -1)
    np.testing.assert_array_equal(orc.unpack_int4(orc.pack_int4(a)), a)


def _rotations(rng, H, rk, R):
    qk = np.stack([np.linalg.qr(rng.standard_normal((rk, rk)))[0] for _ in range(H)])
    qv = np.linalg.qr(rng.standard_normal((R, R)))[0]
    return qk, qv


def test_rotation_folds_into_the_factors():
    inp = wl.make_decode_inputs(TINY, [50, 33], seed=4)
    c = inp.cache
    qk, qv = _rotations(np.random.default_rng(5), TINY["num_heads"], TINY["rank_k"],
                        TINY["rank_v"])
    U, W = orc.rotate_factors(inp.U_k, inp.W_v, qk, qv)
    kp = np.einsum("hij,bhtj->bhti", qk, c.k_pages.astype(np.float64))
    vp = np.einsum("ij,btj->bti", qv, c.v_pages.astype(np.float64))
    ref = orc.decode_attn(inp.q, c.k_pages, c.v_pages, inp.U_k, inp.W_v, c.block_table,
                          c.seq_lens)
    got = orc.decode_attn(inp.q, kp, vp, U, W, c.block_table, c.seq_lens)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)



def test_pages_on_their_grids_round_trip_and_decode_unchanged():
    """K groups are single (block, head, slot) rows, V groups 16 joint coefficients here:
    pages built from integer codes times a per-group power of two come back exactly."""
    rng = np.random.default_rng(8)
    inp = wl.make_decode_inputs(TINY, [40, 17], seed=9)
    c = inp.cache
    nb, H, bs, rk = c.k_pages.shape
    R = c.v_pages.shape[-1]
    kc = rng.integers(-7, 8, size=(nb, H, bs, rk))
    kc[..., 0] = 7
    kp = kc * 2.0 ** rng.integers(-6, 3, size=(nb, H, bs, 1))
    vc = rng.integers(-7, 8, size=(nb, bs, R))
    vc[..., ::16] = -7
    vp = vc * np.repeat(2.0 ** rng.integers(-6, 3, size=(nb, bs, R // 16)), 16, axis=-1)
    k4, ks, v4, vs = orc.int4_pages(kp, vp, v_group=16)
    assert ks.shape == (nb, H, bs) and vs.shape == (nb, bs, R // 16)
    kv, vv = orc.int4_page_values(k4, ks, v4, vs, v_group=16)
    np.testing.assert_array_equal(kv, kp)
    np.testing.assert_array_equal(vv, vp)
    a = orc.decode_attn(inp.q, kp, vp, inp.U_k, inp.W_v, c.block_table, c.seq_lens)
    b = orc.decode_attn(inp.q, kv, vv, inp.U_k, inp.W_v, c.block_table, c.seq_lens)
    np.testing.assert_array_equal(a, b)
