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


# ---------------------------------------------------------------------- 4-bit byte pages
def _golden_page():
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "int4_page.json")) as f:
        return json.load(f)


def test_golden_int4_page_layout():
    g = _golden_page()
    s = g["shape"]
    H, rk, R = s["num_heads"], s["rank_k"], s["rank_v"]
    assert orc.int4_page_bytes(H, rk, R) == (g["k_page_bytes"], g["v_page_bytes"])
    kc = np.zeros((1, H, 16, rk), np.int8)
    ks = np.zeros((1, H, 16), np.float16)
    vc = np.zeros((1, 16, R), np.int8)
    vs = np.zeros((1, 16, R // 64), np.float16)
    for e in g["k_codes"]:
        kc[0, e["head"], e["token"]] = e["codes"]
        ks[0, e["head"], e["token"]] = np.array([int(e["scale_hex"], 16)], np.uint16).view(np.float16)[0]
    for e in g["v_codes"]:
        for r, c in e["codes_at"].items():
            vc[0, e["token"], int(r)] = c
        vs[0, e["token"], 0] = np.array([int(e["scale_hex"], 16)], np.uint16).view(np.float16)[0]
    kb, vb = orc.int4_pack_pages(kc, ks, vc, vs)
    assert kb.shape == (1, g["k_page_bytes"]) and vb.shape == (1, g["v_page_bytes"])
    want_k = np.zeros(g["k_page_bytes"], np.uint8)
    for i, b in g["expected_k_bytes"].items():
        want_k[int(i)] = int(b, 16)
    want_v = np.zeros(g["v_page_bytes"], np.uint8)
    for i, b in g["expected_v_bytes"].items():
        want_v[int(i)] = int(b, 16)
    np.testing.assert_array_equal(kb[0], want_k)
    np.testing.assert_array_equal(vb[0], want_v)
    kv, vv = orc.int4_page_coefficients(kb, vb, H, rk, R)
    ek, ev = g["expected_k_values"], g["expected_v_values"]
    np.testing.assert_array_equal(kv[0, ek["head"], ek["token"]], ek["values"])
    np.testing.assert_array_equal(vv[0, ev["token"], ev["ranks"]], ev["values"])
    assert np.count_nonzero(kv) == 4 and np.count_nonzero(vv) == 4


def test_int4_pages_pack_unpack_round_trip():
    rng = np.random.default_rng(5)
    H, rk, R = 4, 16, 128
    kc = rng.integers(-7, 8, size=(3, H, 16, rk)).astype(np.int8)
    ks = rng.uniform(0, 4, size=(3, H, 16)).astype(np.float16)
    vc = rng.integers(-7, 8, size=(3, 16, R)).astype(np.int8)
    vs = rng.uniform(0, 4, size=(3, 16, R // 64)).astype(np.float16)
    kb, vb = orc.int4_pack_pages(kc, ks, vc, vs)
    kc2, ks2, vc2, vs2 = orc.int4_unpack_pages(kb, vb, H, rk, R)
    np.testing.assert_array_equal(kc2, kc)
    np.testing.assert_array_equal(ks2.view(np.uint16), ks.view(np.uint16))
    np.testing.assert_array_equal(vc2, vc)
    np.testing.assert_array_equal(vs2.view(np.uint16), vs.view(np.uint16))


def _smallest_scale(amax: float) -> float:
    """Smallest fp16 s with 7 s >= amax, by walking fp16 values (enumeration)."""
    if amax == 0:
        return 0.0
    s = np.float16(amax / 7.0)
    while float(s) * 7 < amax:
        s = np.nextafter(s, np.float16(np.inf))
    while float(np.nextafter(s, np.float16(0))) * 7 >= amax:
        s = np.nextafter(s, np.float16(0))
    return float(s)


def test_int4_append_groups_rederived_by_enumeration():
    """Every group an append writes: its scale is the smallest fp16 with 7 s >= max|x| of
    the exact projection, and each code is the nearest point of the grid s*[-7..7] (ties to
    even); untouched slots keep their bytes."""
    H, d, rk, R = TINY["num_heads"], TINY["head_dim"], TINY["rank_k"], TINY["rank_v"]
    rng = np.random.default_rng(6)
    U, W = wl.make_factors(rng, H, d, rk, R)
    kbytes = rng.integers(0, 256, size=(4, orc.int4_page_bytes(H, rk, R)[0])).astype(np.uint8)
    vbytes = rng.integers(0, 256, size=(4, orc.int4_page_bytes(H, rk, R)[1])).astype(np.uint8)
    # valid fp16 scales in the untouched slots (random bytes could spell NaN)
    kc0, _, vc0, _ = orc.int4_unpack_pages(kbytes, vbytes, H, rk, R)
    kbytes, vbytes = orc.int4_pack_pages(kc0, np.full((4, H, 16), 0.25, np.float16), vc0,
                                         np.full((4, 16, R // 64), 0.5, np.float16))
    k = wl.fp16(rng.standard_normal((5, H, d)))
    v = wl.fp16(rng.standard_normal((5, H, d)))
    slots = np.array([7, -1, 16, 63, 33], np.int64)
    kb2, vb2 = orc.append_kv_int4(kbytes, vbytes, U, W, k, v, slots)
    kc, ks, vc, vs = orc.int4_unpack_pages(kb2, vb2, H, rk, R)
    grid = np.arange(-7, 8)

    def check(x, codes, scale):
        sc = _smallest_scale(float(np.abs(x).max()))
        assert float(scale) == sc
        for xi, ci in zip(x, codes):
            if sc == 0:
                assert ci == 0
                continue
            dd = np.abs(xi - grid * sc)
            best = grid[dd == dd.min()]
            want = best[0] if len(best) == 1 else best[best % 2 == 0][0]
            assert ci == want

    for i, s in enumerate(slots):
        if s < 0:
            continue
        blk, off = s // 16, s % 16
        for h in range(H):
            check(U[h].astype(np.float64) @ k[i, h].astype(np.float64), kc[blk, h, off],
                  ks[blk, h, off])
        cv = W.astype(np.float64) @ v[i].astype(np.float64).reshape(-1)
        for gi in range(R // 64):
            check(cv[64 * gi:64 * (gi + 1)], vc[blk, off, 64 * gi:64 * (gi + 1)], vs[blk, off, gi])
    written = {int(s) for s in slots if s >= 0}
    kc1, ks1, vc1, vs1 = orc.int4_unpack_pages(kbytes, vbytes, H, rk, R)
    for blk in range(4):
        for off in range(16):
            if blk * 16 + off not in written:
                np.testing.assert_array_equal(kc[blk, :, off], kc1[blk, :, off])
                np.testing.assert_array_equal(vc[blk, off], vc1[blk, off])
                np.testing.assert_array_equal(ks[blk, :, off], ks1[blk, :, off])
