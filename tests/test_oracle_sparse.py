"""Pins for the oracle's block-sparse decode pieces (no GPU).

Page skipping: a page is dropped when every head's largest weight in it falls below a
threshold times that head's largest weight; dropped pages leave both the numerator and the
denominator of the softmax.  The pins tie the three oracle functions to facts outside
them: attention over a subset of pages equals plain attention over a compacted block
table (the subset's tokens in order) and a textbook loop over the kept tokens; the
skippable set matches a hand-built score pattern; a sequential single pass with a running
maximum drops a subset of it; and the output change stays within the stated bound.
"""
import math

import numpy as np

import workloads as wl
from oracle import rcp_oracle as orc

TINY = wl.SHAPES["tiny"]


def _compact(cache, kept):
    """Block table holding only the kept pages of each request, with the new lengths."""
    B = len(cache.seq_lens)
    table = np.full_like(cache.block_table, -1)
    lens = np.zeros(B, np.int32)
    for b in range(B):
        L = int(cache.seq_lens[b])
        n = wl.blocks_needed(L)
        cols = [j for j in range(n) if kept[b][j]]
        table[b, :len(cols)] = cache.block_table[b, cols]
        # every kept page is full except possibly the request's last page
        lens[b] = sum(min(16, L - 16 * j) for j in cols)
        # a partial page can only sit last in the compacted row
        assert all(min(16, L - 16 * j) == 16 for j in cols[:-1])
    return table, lens


def _random_kept(rng, cache, keep_last):
    kept = []
    for L in cache.seq_lens:
        n = wl.blocks_needed(int(L))
        m = rng.random(n) < 0.6
        if n:
            m[-1] = keep_last
            m[0] = True
        kept.append(m)
    return kept


def test_kept_attention_equals_attention_over_compacted_table():
    inp = wl.make_decode_inputs(TINY, [100, 57, 16, 33], seed=41, fill=np.nan)
    c = inp.cache
    rng = np.random.default_rng(5)
    for keep_last in (True, False):
        kept = _random_kept(rng, c, keep_last)
        table, lens = _compact(c, kept)
        got = orc.decode_attn_kept(inp.q, c.k_pages, c.v_pages, inp.U_k, inp.W_v,
                                   c.block_table, c.seq_lens, kept)
        ref = orc.decode_attn(inp.q, c.k_pages, c.v_pages, inp.U_k, inp.W_v, table, lens)
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-13)


def test_kept_attention_textbook_loop():
    """Scalar softmax over the explicitly listed kept tokens, one (request, head) at a time."""
    inp = wl.make_decode_inputs(TINY, [40, 20], seed=42)
    c = inp.cache
    kept = [np.array([True, False, True]), np.array([False, True])]
    got = orc.decode_attn_kept(inp.q, c.k_pages, c.v_pages, inp.U_k, inp.W_v, c.block_table,
                               c.seq_lens, kept)
    H, d, rk, R = TINY["num_heads"], TINY["head_dim"], TINY["rank_k"], TINY["rank_v"]
    U = inp.U_k.astype(np.float64)
    W = inp.W_v.astype(np.float64)
    for b in range(2):
        toks = [t for t in range(int(c.seq_lens[b])) if kept[b][t // 16]]
        for h in range(H):
            qt = [sum(float(U[h, k, i]) * float(inp.q[b, h, i]) for i in range(d)) for k in range(rk)]
            s = [sum(qt[k] * float(c.ck[b][t][h][k]) for k in range(rk)) / math.sqrt(d) for t in toks]
            m = max(s)
            w = [math.exp(x - m) for x in s]
            tot = sum(w)
            z = [sum(w[i] * float(c.cv[b][t][r]) for i, t in enumerate(toks)) / tot for r in range(R)]
            o = [sum(W[r, h * d + j] * z[r] for r in range(R)) for j in range(d)]
            np.testing.assert_allclose(got[b, h], o, rtol=0, atol=1e-12)


def test_kept_attention_with_no_kept_page_is_zero_and_all_kept_is_decode():
    inp = wl.make_decode_inputs(TINY, [40, 20], seed=43)
    c = inp.cache
    got = orc.decode_attn_kept(inp.q, c.k_pages, c.v_pages, inp.U_k, inp.W_v, c.block_table,
                               c.seq_lens, [np.zeros(3, bool), np.ones(2, bool)])
    assert np.all(got[0] == 0)
    ref = orc.decode_attn(inp.q, c.k_pages, c.v_pages, inp.U_k, inp.W_v, c.block_table, c.seq_lens)
    np.testing.assert_array_equal(got[1], ref[1])


def _pattern_case():
    """Identity factors (r_k = d, R = H d), q = sqrt(d) e_0 for each head, and every key of
    page j of head h equal to x[h][j] e_0 (padding keys far below): the score of every
    token of page j for head h is exactly x[h][j]."""
    H, d = 2, 16                                     # sqrt(d) = 4 is exact in fp16
    x = np.array([[5.0, 0.0, 4.0, -3.0, 5.0],
                  [0.0, 5.0, 0.0, 0.0, 0.0]])
    n = x.shape[1]
    L = 16 * n - 3                                   # last page partial
    kp = np.zeros((n, H, 16, d), np.float16)
    for j in range(n):
        for h in range(H):
            kp[j, h, :, 0] = x[h, j]
    vp = np.zeros((n, 16, H * d), np.float16)
    U = np.stack([np.eye(d, dtype=np.float16)] * H)
    q = np.zeros((1, H, d), np.float16)
    q[0, :, 0] = math.sqrt(d)
    table = np.arange(n, dtype=np.int32)[None]
    return q, kp, vp, U, table, np.array([L], np.int32), x


def test_skippable_pages_hand_built_scores():
    q, kp, vp, U, table, lens, x = _pattern_case()
    assert np.allclose(orc.page_max_scores(q[0], kp, U, table[0], int(lens[0])), x.T)
    # threshold e^-2: head 0 (max 5) drops pages 1 (0-5) and 3 (-3-5); head 1 (max 5)
    # drops every page but 1; a page goes only if both heads drop it
    got = orc.skippable_pages(q, kp, U, table, lens, math.exp(-2.0))[0]
    np.testing.assert_array_equal(got, [False, False, False, True, False])
    # threshold e^-0.5: head 0 also drops page 2 (4-5 = -1); head 1 still needs page 1
    got = orc.skippable_pages(q, kp, U, table, lens, math.exp(-0.5))[0]
    np.testing.assert_array_equal(got, [False, False, True, True, False])
    # threshold e^-9: nothing is that far below (-8 is the lowest)
    assert not orc.skippable_pages(q, kp, U, table, lens, math.exp(-9.0))[0].any()
    # threshold 0 drops nothing
    assert not orc.skippable_pages(q, kp, U, table, lens, 0.0)[0].any()


def _single_pass_dropped(pm, threshold):
    """Pages a sequential pass drops: running maximum over the kept pages seen so far."""
    H = pm.shape[1]
    run = np.full(H, -np.inf)
    out = np.zeros(pm.shape[0], bool)
    for j in range(pm.shape[0]):
        if np.all(pm[j] - run < math.log(threshold)):
            out[j] = True
        else:
            run = np.maximum(run, pm[j])
    return out


def test_single_pass_drops_a_subset_of_the_skippable_pages_and_error_is_bounded():
    inp = wl.make_decode_inputs(TINY, [400, 260, 16, 97], seed=44, peaked=wl.PEAKED)
    c = inp.cache
    thr = 2.0 ** -6
    skippable = orc.skippable_pages(inp.q, c.k_pages, inp.U_k, c.block_table, c.seq_lens, thr)
    dropped = []
    for b in range(len(c.seq_lens)):
        pm = orc.page_max_scores(inp.q[b], c.k_pages, inp.U_k, c.block_table[b], int(c.seq_lens[b]))
        d = _single_pass_dropped(pm, thr)
        assert not np.any(d & ~skippable[b])
        dropped.append(d)
    # the workload is built so that skipping has something to do
    assert sum(int(d.sum()) for d in dropped) >= 10
    kept = [~d for d in dropped]
    full = orc.decode_attn(inp.q, c.k_pages, c.v_pages, inp.U_k, inp.W_v, c.block_table, c.seq_lens)
    part = orc.decode_attn_kept(inp.q, c.k_pages, c.v_pages, inp.U_k, inp.W_v, c.block_table,
                                c.seq_lens, kept)
    bound = orc.skip_error_bound(inp.q, c.k_pages, c.v_pages, inp.U_k, inp.W_v, c.block_table,
                                 c.seq_lens, dropped)
    assert np.all(np.abs(part - full) <= bound[:, :, None] * (1 + 1e-9) + 1e-15)
    # skipping changed the result, by no more than the bound allows
    assert np.abs(part - full).max() > 0


def test_error_bound_holds_when_heavy_pages_are_dropped():
    """Dropping pages with real weight: the bound must still hold (and is not vacuous)."""
    inp = wl.make_decode_inputs(TINY, [160, 96], seed=45)
    c = inp.cache
    rng = np.random.default_rng(9)
    dropped = [rng.random(wl.blocks_needed(int(L))) < 0.5 for L in c.seq_lens]
    for m in dropped:
        m[0] = False
    full = orc.decode_attn(inp.q, c.k_pages, c.v_pages, inp.U_k, inp.W_v, c.block_table, c.seq_lens)
    part = orc.decode_attn_kept(inp.q, c.k_pages, c.v_pages, inp.U_k, inp.W_v, c.block_table,
                                c.seq_lens, [~m for m in dropped])
    bound = orc.skip_error_bound(inp.q, c.k_pages, c.v_pages, inp.U_k, inp.W_v, c.block_table,
                                 c.seq_lens, dropped)
    diff = np.abs(part - full).max(axis=2)
    assert np.all(diff <= bound * (1 + 1e-9))
    assert np.all(diff > 0) and bound.max() < 10 * np.abs(full).max()


def test_peaked_workload_background_pages_are_skippable():
    """The peaked recipe's background pages are the ones the rule finds (almost all)."""
    inp = wl.make_decode_inputs(TINY, [800, 512], seed=46, peaked=wl.PEAKED)
    c = inp.cache
    sk = orc.skippable_pages(inp.q, c.k_pages, inp.U_k, c.block_table, c.seq_lens, 2.0 ** -6)
    for b in range(2):
        bg = inp.background[b]
        assert bg.sum() > 0
        assert (sk[b] & bg).sum() >= 0.9 * bg.sum()
        assert not sk[b][0] and not sk[b][-1]
