"""Pins for the fp64 oracle against facts fixed outside it (no GPU).

Each test ties the oracle to something other than its own formula: a hand-derived closed
form, a library attention routine on explicitly reconstructed dense K/V, an invariant
(block relabelling, weights summing to one, exact power-of-two scaling), or a special
case that reduces to plain attention.  A dropped term, a wrong sign or index, a transposed
factor or a wrong softmax scale breaks at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import workloads as wl
from oracle import rcp_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TINY = wl.SHAPES["tiny"]


def _sdpa(q, k, v, causal=False):
    """Library multi-head attention in fp64: q [H][Lq][d], k/v [H][Lk][d]."""
    return F.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None],
        is_causal=causal).numpy()[0]


def _golden():
    with open(os.path.join(GOLDEN, "two_token_decode.json")) as f:
        return json.load(f)


def _golden_cache(g):
    s = g["shape"]
    kp = np.full((s["num_blocks"], s["num_heads"], s["block_size"], s["rank_k"]), np.nan,
                 np.float16)
    vp = np.full((s["num_blocks"], s["block_size"], s["rank_v"]), np.nan, np.float16)
    blk = g["block_table"][0][0]
    for t, (ck, cv) in enumerate(zip(g["tokens_ck"], g["tokens_cv"])):
        kp[blk, :, t, :] = ck
        vp[blk, t, :] = cv
    return kp, vp


def test_golden_two_token_decode_closed_form():
    g = _golden()
    kp, vp = _golden_cache(g)
    out = orc.decode_attn(np.array(g["q"], np.float16), kp, vp,
                          np.array(g["U_k"], np.float16), np.array(g["W_v"], np.float16),
                          np.array(g["block_table"]), np.array(g["seq_lens"]), 16)
    exp = np.array([[[eval(x, {"e": math.e}) for x in row] for row in req]
                    for req in g["expected_out"]])
    np.testing.assert_allclose(out, exp, rtol=0, atol=1e-14)


def test_golden_append_hand_derived():
    g = _golden()
    s = g["shape"]
    a = g["append"]
    kp = np.full((s["num_blocks"], s["num_heads"], 16, s["rank_k"]), -7.0, np.float16)
    vp = np.full((s["num_blocks"], 16, s["rank_v"]), -7.0, np.float16)
    kp2, vp2 = orc.append_kv(kp, vp, np.array(g["U_k"], np.float16),
                             np.array(g["W_v"], np.float16), np.array(a["k"], np.float16),
                             np.array(a["v"], np.float16), np.array(a["slot_mapping"]), 16)
    ek, ev = a["expected_k_page"], a["expected_v_page"]
    assert np.array_equal(kp2[ek["block"], :, ek["offset"], :],
                          np.array(ek["values"], np.float16))
    assert np.array_equal(vp2[ev["block"], ev["offset"], :], np.array(ev["values"], np.float16))
    mask = np.ones(kp.shape[:3], bool)
    mask[ek["block"], :, ek["offset"]] = False
    assert np.all(kp2[mask] == -7.0)
    vmask = np.ones(vp.shape[:2], bool)
    vmask[ev["block"], ev["offset"]] = False
    assert np.all(vp2[vmask] == -7.0)


def test_identity_factors_reduce_to_dense_mha():
    """r_k = d, U = I, R = H*d, W_v = I: coefficients are the dense K/V themselves."""
    H, d = 4, 64
    rng = np.random.default_rng(11)
    U, W = wl.identity_factors(H, d)
    cache = wl.make_paged_cache(rng, H, d, H * d, [256, 77], spare_blocks=3, fill=np.nan)
    q = wl.fp16(rng.standard_normal((2, H, d)))
    out = orc.decode_attn(q, cache.k_pages, cache.v_pages, U, W, cache.block_table,
                          cache.seq_lens, 16)
    for b in range(2):
        K = cache.ck[b].astype(np.float64).transpose(1, 0, 2)                 # [H][L][d]
        V = cache.cv[b].astype(np.float64).reshape(-1, H, d).transpose(1, 0, 2)
        ref = _sdpa(q[b].astype(np.float64)[:, None, :], K, V)[:, 0, :]
        np.testing.assert_allclose(out[b], ref, rtol=0, atol=1e-12)


def test_reconstruction_matches_dense_attention():
    """Dense K = C_k U_k and V = C_v W_v built explicitly, then library attention."""
    H, d, rk, R = TINY["num_heads"], TINY["head_dim"], TINY["rank_k"], TINY["rank_v"]
    inp = wl.make_decode_inputs(TINY, [256, 200], seed=1000, fill=np.nan)
    U = inp.U_k.astype(np.float64)
    W = inp.W_v.astype(np.float64)
    out = orc.decode_attn(inp.q, inp.cache.k_pages, inp.cache.v_pages, inp.U_k, inp.W_v,
                          inp.cache.block_table, inp.cache.seq_lens, 16)
    for b in range(2):
        ck = inp.cache.ck[b].astype(np.float64)       # logical order, from the generator
        cv = inp.cache.cv[b].astype(np.float64)
        K = np.einsum("thk,hkd->htd", ck, U)          # k_hat_{t,h} = U_k,h^T c_k[t,h]
        V = (cv @ W).reshape(-1, H, d).transpose(1, 0, 2)
        ref = _sdpa(inp.q[b].astype(np.float64)[:, None, :], K, V)[:, 0, :]
        np.testing.assert_allclose(out[b], ref, rtol=0, atol=1e-12)
    assert rk != d and R != H * d


def test_block_permutation_is_bitwise_invariant():
    inp = wl.make_decode_inputs(TINY, [256, 131, 16], seed=5, spare_blocks=7, fill=np.nan)
    out1 = orc.decode_attn(inp.q, inp.cache.k_pages, inp.cache.v_pages, inp.U_k, inp.W_v,
                           inp.cache.block_table, inp.cache.seq_lens, 16)
    c2 = wl.permute_physical_blocks(inp.cache, np.random.default_rng(9))
    assert not np.array_equal(c2.block_table, inp.cache.block_table)
    out2 = orc.decode_attn(inp.q, c2.k_pages, c2.v_pages, inp.U_k, inp.W_v, c2.block_table,
                           c2.seq_lens, 16)
    assert np.array_equal(out1, out2)


def test_softmax_weights_sum_to_one():
    inp = wl.make_decode_inputs(TINY, [256, 1, 33], seed=6)
    _, ws = orc.decode_attn(inp.q, inp.cache.k_pages, inp.cache.v_pages, inp.U_k, inp.W_v,
                            inp.cache.block_table, inp.cache.seq_lens, 16,
                            return_weights=True)
    for p in ws:
        assert np.all(p >= 0)
        assert np.max(np.abs(p.sum(axis=1) - 1.0)) <= 1e-12


def test_single_token_gives_up_projected_value():
    inp = wl.make_decode_inputs(TINY, [1], seed=7)
    out = orc.decode_attn(inp.q, inp.cache.k_pages, inp.cache.v_pages, inp.U_k, inp.W_v,
                          inp.cache.block_table, inp.cache.seq_lens, 16)
    H, d = TINY["num_heads"], TINY["head_dim"]
    v_hat = (inp.W_v.astype(np.float64).T @ inp.cache.cv[0][0].astype(np.float64))
    np.testing.assert_allclose(out[0], v_hat.reshape(H, d), rtol=0, atol=1e-15)


def test_equal_keys_give_mean_reconstructed_value():
    inp = wl.make_decode_inputs(TINY, [48], seed=8)
    c = inp.cache
    row = c.block_table[0]
    kp = c.k_pages.copy()
    for t in range(48):                               # every token: same K coefficients
        kp[row[t // 16], :, t % 16, :] = c.ck[0][0]
    out = orc.decode_attn(inp.q, kp, c.v_pages, inp.U_k, inp.W_v, c.block_table, c.seq_lens, 16)
    H, d = TINY["num_heads"], TINY["head_dim"]
    mean_v = c.cv[0].astype(np.float64).mean(axis=0) @ inp.W_v.astype(np.float64)
    np.testing.assert_allclose(out[0], mean_v.reshape(H, d), rtol=0, atol=1e-14)


def test_doubling_value_coefficients_doubles_output_exactly():
    inp = wl.make_decode_inputs(TINY, [256, 70], seed=9)
    c = inp.cache
    o1 = orc.decode_attn(inp.q, c.k_pages, c.v_pages, inp.U_k, inp.W_v, c.block_table,
                         c.seq_lens, 16)
    o2 = orc.decode_attn(inp.q, c.k_pages, (c.v_pages.astype(np.float32) * 2).astype(np.float16),
                         inp.U_k, inp.W_v, c.block_table, c.seq_lens, 16)
    assert np.array_equal(o2, 2 * o1)


def test_scores_use_head_dim_scale_not_rank():
    """Two tokens whose score gap is known: weight ratio must be exp(gap / sqrt(d))."""
    H, d, rk, R = 1, 64, 16, 8
    U = np.zeros((1, rk, d), np.float16)
    U[0, np.arange(rk), np.arange(rk)] = 1
    W = np.zeros((R, d), np.float16)
    W[np.arange(R), np.arange(R)] = 1
    kp = np.zeros((1, 1, 16, rk), np.float16)
    kp[0, 0, 1, 0] = 4.0                               # token 1 score = q0 * 4 / 8
    vp = np.zeros((1, 16, R), np.float16)
    vp[0, 0, 0] = 1.0
    vp[0, 1, 1] = 1.0
    q = np.zeros((1, 1, d), np.float16)
    q[0, 0, 0] = 2.0                                   # gap = 2 * 4 / sqrt(64) = 1
    out = orc.decode_attn(q, kp, vp, U, W, np.array([[0]]), np.array([2]), 16)
    np.testing.assert_allclose(out[0, 0, :2], [1 / (1 + math.e), math.e / (1 + math.e)],
                               rtol=0, atol=1e-15)


def test_empty_sequence_gives_zero():
    inp = wl.make_decode_inputs(TINY, [0, 40], seed=10)
    out = orc.decode_attn(inp.q, inp.cache.k_pages, inp.cache.v_pages, inp.U_k, inp.W_v,
                          inp.cache.block_table, inp.cache.seq_lens, 16)
    assert np.all(out[0] == 0)
    assert np.all(np.isfinite(out))


def test_prefill_with_no_prior_is_causal_attention():
    H, d = TINY["num_heads"], TINY["head_dim"]
    inp = wl.make_prefill_inputs(TINY, [0], [40], seed=12, fill=np.nan)
    kp, vp = orc.append_kv(inp.cache.k_pages, inp.cache.v_pages, inp.U_k, inp.W_v, inp.k,
                           inp.v, inp.slot_mapping, 16)
    out = orc.prefill_attn(inp.q, inp.cu_chunk_lens, kp, vp, inp.U_k, inp.W_v,
                           inp.cache.block_table, inp.seq_lens_after, 16)
    # dense reference from the appended coefficients read back by physical position
    ck, cv = orc.gather_request(kp, vp, inp.cache.block_table[0], 40, 16)
    K = np.einsum("thk,hkd->htd", ck, inp.U_k.astype(np.float64))
    V = (cv @ inp.W_v.astype(np.float64)).reshape(-1, H, d).transpose(1, 0, 2)
    ref = _sdpa(inp.q.astype(np.float64).transpose(1, 0, 2), K, V, causal=True)
    np.testing.assert_allclose(out, ref.transpose(1, 0, 2), rtol=0, atol=1e-12)


def test_prefill_rows_equal_decode_at_their_positions():
    inp = wl.make_prefill_inputs(TINY, [37, 64], [21, 16], seed=13, fill=np.nan)
    kp, vp = orc.append_kv(inp.cache.k_pages, inp.cache.v_pages, inp.U_k, inp.W_v, inp.k,
                           inp.v, inp.slot_mapping, 16)
    out = orc.prefill_attn(inp.q, inp.cu_chunk_lens, kp, vp, inp.U_k, inp.W_v,
                           inp.cache.block_table, inp.seq_lens_after, 16)
    for b in range(2):
        for i in range(int(inp.chunk_lens[b])):
            row = inp.cu_chunk_lens[b] + i
            L = int(inp.prior_lens[b]) + i + 1
            dec = orc.decode_attn(inp.q[row][None], kp, vp, inp.U_k, inp.W_v,
                                  inp.cache.block_table[b][None], np.array([L]), 16)
            assert np.array_equal(out[row], dec[0])


def test_append_with_selection_factors_copies_exactly():
    H, d, rk, R = 4, 64, 16, 64
    rng = np.random.default_rng(14)
    U, W = wl.selection_factors(rng, H, d, rk, R)
    kp = np.full((6, H, 16, rk), np.nan, np.float16)
    vp = np.full((6, 16, R), np.nan, np.float16)
    k = wl.fp16(rng.standard_normal((5, H, d)))
    v = wl.fp16(rng.standard_normal((5, H, d)))
    slots = np.array([17, -1, 95, 0, 40], np.int64)
    kp2, vp2 = orc.append_kv(kp, vp, U, W, k, v, slots, 16)
    for i, s in enumerate(slots):
        if s < 0:
            continue
        for h in range(H):
            cols = np.argmax(U[h] != 0, axis=1)
            assert np.array_equal(kp2[s // 16, h, s % 16], k[i, h, cols])
        colsv = np.argmax(W != 0, axis=1)
        assert np.array_equal(vp2[s // 16, s % 16], v[i].reshape(-1)[colsv])
    written = {(int(s) // 16, int(s) % 16) for s in slots if s >= 0}
    for blk in range(6):
        for off in range(16):
            if (blk, off) not in written:
                assert np.all(np.isnan(kp2[blk, :, off])) and np.all(np.isnan(vp2[blk, off]))


def test_golden_append_rounds_to_nearest_even():
    """Hand-derived fp16 bit patterns of projections that fp16 cannot hold exactly: ties
    in both directions, a tie that an intermediate binary32 rounding would create, a
    subnormal tie, the top of the range and the overflow to infinity
    (tests/golden/append_rounding.json)."""
    with open(os.path.join(GOLDEN, "append_rounding.json")) as f:
        g = json.load(f)
    s = g["shape"]

    def hexf(a):
        return np.vectorize(float.fromhex, otypes=[np.float64])(np.array(a, dtype=object))

    U, W = hexf(g["U_k"]), hexf(g["W_v"])
    # every factor and input entry is a binary16 value, so nothing rounds on the way in
    toks = g["tokens"]
    k = np.stack([hexf(tk["k"]) for tk in toks])
    v = np.stack([hexf(tk["v"]) for tk in toks])
    for a in (U, W, k, v):
        assert np.array_equal(a.astype(np.float16).astype(np.float64), a)
    slots = np.array([tk["slot"] for tk in toks], np.int64)
    kp = np.full((s["num_blocks"], s["num_heads"], 16, s["rank_k"]), -7.0, np.float16)
    vp = np.full((s["num_blocks"], 16, s["rank_v"]), -7.0, np.float16)
    kp2, vp2 = orc.append_kv(kp, vp, U.astype(np.float16), W.astype(np.float16),
                             k.astype(np.float16), v.astype(np.float16), slots, 16)
    for e in g["expected"]:
        kb = np.array([[int(x, 16) for x in row] for row in e["k_bits"]], np.uint16)
        vb = np.array([int(x, 16) for x in e["v_bits"]], np.uint16)
        assert np.array_equal(kp2[e["block"], :, e["offset"], :].view(np.uint16), kb), e
        assert np.array_equal(vp2[e["block"], e["offset"], :].view(np.uint16), vb), e
    untouched = np.ones(kp.shape[:3], bool)
    for e in g["expected"]:
        untouched[e["block"], :, e["offset"]] = False
    assert np.all(kp2[untouched] == -7.0)


def _fp16_nearest_even(x: float) -> int:
    """Bit pattern of the binary16 value nearest to x (ties: even fraction), by search
    over all finite binary16 values and the two infinities (IEEE 754 rounds to infinity
    at or beyond 65520)."""
    if x >= 65520.0:
        return 0x7C00
    if x <= -65520.0:
        return 0xFC00
    bits = np.arange(0x10000, dtype=np.uint32).astype(np.uint16)
    vals = bits.view(np.float16).astype(np.float64)
    ok = np.isfinite(vals)
    d = np.abs(vals - x)
    d[~ok] = np.inf
    best = np.nonzero(d == d.min())[0]
    if len(best) > 1:
        even = [b for b in best if (b & 1) == 0]
        best = even if even else best
        if x == 0.0:
            best = [0x8000 if math.copysign(1.0, x) < 0 else 0x0000]
    return int(best[0])


def test_append_with_pair_sum_factors_matches_brute_force_rounding():
    """Two-unit-entry factors sum two fp16 inputs per coefficient; the oracle's fp16 result
    must be the nearest-even binary16 of that exact sum, found by enumeration."""
    H, d, rk, R = 4, 64, 16, 64
    rng = np.random.default_rng(16)
    U, W = wl.pair_sum_factors(rng, H, d, rk, R)
    k = wl.fp16_narrow(rng, (3, H, d))
    v = wl.fp16_narrow(rng, (3, H, d))
    slots = np.array([3, 40, 77], np.int64)
    kp = np.zeros((6, H, 16, rk), np.float16)
    vp = np.zeros((6, 16, R), np.float16)
    kp2, vp2 = orc.append_kv(kp, vp, U, W, k, v, slots, 16)
    ties = inexact = 0
    for i, s in enumerate(slots):
        exact_k = np.einsum("hkd,hd->hk", U.astype(np.float64), k[i].astype(np.float64))
        exact_v = W.astype(np.float64) @ v[i].astype(np.float64).reshape(-1)
        got_k = kp2[s // 16, :, s % 16, :].view(np.uint16)
        got_v = vp2[s // 16, s % 16, :].view(np.uint16)
        for x, gbits in zip(list(exact_k.ravel()) + list(exact_v), list(got_k.ravel()) +
                            list(got_v)):
            assert int(gbits) == _fp16_nearest_even(float(x)), x
            lo = np.float16(x)
            inexact += float(lo) != x
            # halfway cases: the exact sum sits midway between two binary16 neighbours
            nb = np.nextafter(lo, np.float16(np.inf if float(lo) < x else -np.inf))
            ties += float(lo) != x and abs(float(nb) - x) == abs(float(lo) - x)
    assert inexact > 100 and ties > 5, (inexact, ties)


def test_append_then_gather_round_trip():
    """Scatter through slots, gather back through the block table: the projections."""
    inp = wl.make_prefill_inputs(TINY, [5, 30], [12, 9], seed=15, fill=np.nan)
    kp, vp = orc.append_kv(inp.cache.k_pages, inp.cache.v_pages, inp.U_k, inp.W_v, inp.k,
                           inp.v, inp.slot_mapping, 16)
    H, d = TINY["num_heads"], TINY["head_dim"]
    for b in range(2):
        ck, cv = orc.gather_request(kp, vp, inp.cache.block_table[b], inp.seq_lens_after[b], 16)
        P = int(inp.prior_lens[b])
        np.testing.assert_array_equal(ck[:P], inp.cache.ck[b])
        for i in range(int(inp.chunk_lens[b])):
            row = inp.cu_chunk_lens[b] + i
            kk = inp.k[row].astype(np.float64)
            vv = inp.v[row].astype(np.float64).reshape(H * d)
            # projection onto the (nearly orthonormal) factor rows, within fp16 rounding
            np.testing.assert_allclose(
                ck[P + i], np.einsum("hkd,hd->hk", inp.U_k.astype(np.float64), kk),
                rtol=0, atol=4e-3)
            np.testing.assert_allclose(cv[P + i], inp.W_v.astype(np.float64) @ vv,
                                       rtol=0, atol=8e-3)


def test_workload_generator_is_seeded():
    a = wl.make_decode_inputs(TINY, [40, 17], seed=3)
    b = wl.make_decode_inputs(TINY, [40, 17], seed=3)
    assert np.array_equal(a.cache.k_pages, b.cache.k_pages)
    assert np.array_equal(a.q, b.q)
    U = a.U_k.astype(np.float64)
    for h in range(U.shape[0]):
        np.testing.assert_allclose(U[h] @ U[h].T, np.eye(U.shape[1]), atol=3e-3)


# ------------------------------------------------------------------------- E4M3 pages
# Values fixed by the E4M3 format definition (OCP 8-bit floating point, "E4M3"): bias 7,
# three mantissa bits, subnormals m * 2^-9, S.1111.111 = NaN, max finite 448.
E4M3_TABLE = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
              0x30: 0.5, 0x38: 1.0, 0x39: 1.125, 0x3F: 1.875, 0x40: 2.0, 0x77: 240.0,
              0x7E: 448.0, 0x80: -0.0, 0xB8: -1.0, 0xFE: -448.0}


def test_e4m3_decode_matches_the_format_definition():
    for code, val in E4M3_TABLE.items():
        got = orc.e4m3_decode(np.array([code], np.uint8))[0]
        assert got == val and np.signbit(got) == np.signbit(val), (hex(code), got, val)
    assert np.isnan(orc.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))).all()


def test_e4m3_encode_round_trips_every_finite_code():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    np.testing.assert_array_equal(orc.e4m3_encode(orc.e4m3_decode(codes)), codes)


def test_e4m3_encode_rounds_to_nearest_even_and_saturates():
    cases = {1.0625: 0x38,          # halfway 1.0 / 1.125 -> even mantissa (1.0)
             1.1875: 0x3A,          # halfway 1.125 / 1.25 -> even mantissa (1.25)
             1.07: 0x39, 2.0 ** -10: 0x00, 3 * 2.0 ** -10: 0x02,
             448.0: 0x7E, 470.0: 0x7E, 1e9: 0x7E, -1e9: 0xFE, -1.0625: 0xB8}
    for x, code in cases.items():
        assert orc.e4m3_encode(np.array([x]))[0] == code, (x, hex(code))
    assert orc.e4m3_encode(np.array([np.nan]))[0] == 0x7F


def test_e4m3_encode_is_the_nearest_finite_code_brute_force():
    rng = np.random.default_rng(8)
    x = rng.standard_normal(3000) * np.exp(rng.uniform(-10, 6, 3000))
    finite = orc.e4m3_decode(np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8))
    got = orc.e4m3_decode(orc.e4m3_encode(x))
    best = np.min(np.abs(np.clip(x, -448, 448)[:, None] - finite[None, :]), axis=1)
    np.testing.assert_array_equal(np.abs(np.clip(x, -448, 448) - got), best)


def test_e4m3_encode_agrees_with_torch_float8_in_range():
    rng = np.random.default_rng(9)
    x = rng.standard_normal(20000) * np.exp(rng.uniform(-12, 5, 20000))
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(orc.e4m3_encode(x), ref)


def test_fp8_append_with_selection_factors_stores_the_inputs_rounded():
    """Coordinate-selection factors make the fp8 append a rounding of the inputs."""
    H, d, rk, R = 4, 64, 16, 64
    rng = np.random.default_rng(16)
    U, W = wl.selection_factors(rng, H, d, rk, R)
    k = wl.fp16(rng.standard_normal((5, H, d)) * 200)   # some values past 448 saturate
    v = wl.fp16(rng.standard_normal((5, H, d)))
    slots = np.array([17, -1, 95, 0, 40], np.int64)
    kp, vp = orc.append_kv_fp8(np.full((6, H, 16, rk), 0x55, np.uint8),
                               np.full((6, 16, R), 0x55, np.uint8), U, W, k, v, slots, 16)
    assert kp.dtype == np.uint8 and vp.dtype == np.uint8
    for i, s in enumerate(slots):
        if s < 0:
            continue
        for h in range(H):
            cols = np.argmax(U[h] != 0, axis=1)
            np.testing.assert_array_equal(kp[s // 16, h, s % 16],
                                          orc.e4m3_encode(k[i, h, cols].astype(np.float64)))
        colsv = np.argmax(W != 0, axis=1)
        np.testing.assert_array_equal(vp[s // 16, s % 16],
                                      orc.e4m3_encode(v[i].reshape(-1)[colsv].astype(np.float64)))
    assert (kp == 0x7E).any() or (kp == 0xFE).any()      # saturation was exercised
    written = {(int(s) // 16, int(s) % 16) for s in slots if s >= 0}
    for blk in range(6):
        for off in range(16):
            if (blk, off) not in written:
                assert (kp[blk, :, off] == 0x55).all() and (vp[blk, off] == 0x55).all()


def test_fp8_decode_is_decode_on_the_decoded_pages():
    """An fp8 cache holding E4M3 roundings of fp16 pages: the oracle's answer moves by at
    most what E4M3 rounding allows (each coefficient within 2^-4 relative)."""
    inp = wl.make_decode_inputs(wl.SHAPES["mha32"], [300, 77], seed=17)
    c = inp.cache
    k8 = orc.e4m3_decode(orc.e4m3_encode(c.k_pages.astype(np.float64)))
    v8 = orc.e4m3_decode(orc.e4m3_encode(c.v_pages.astype(np.float64)))
    rel_k = np.abs(k8 - c.k_pages) / np.maximum(np.abs(c.k_pages.astype(np.float64)), 2.0 ** -6)
    assert rel_k.max() <= 2.0 ** -4 + 1e-12
    o16 = orc.decode_attn(inp.q, c.k_pages, c.v_pages, inp.U_k, inp.W_v, c.block_table,
                          c.seq_lens, 16)
    o8 = orc.decode_attn(inp.q, k8, v8, inp.U_k, inp.W_v, c.block_table, c.seq_lens, 16)
    rel = np.linalg.norm(o8 - o16) / np.linalg.norm(o16)
    assert 1e-3 < rel < 0.1
