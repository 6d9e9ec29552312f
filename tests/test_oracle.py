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
