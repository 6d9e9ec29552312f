"""Block-sparse decode on the GPU vs the oracle, through the C ABI (needs a GB300).

Which pages a pass leaves out depends on the order it meets them in (one running maximum
per work partition, each partition starting with a kept page), so several results are
valid.  What is checked: every page the kernel left out satisfies the skipping rule
against the maximum over the whole sequence (the most a running maximum can reach); the
first page of every request is read; the output equals the oracle's attention over
exactly the pages the kernel read (the usual fp16 tolerance); it differs from full
attention by no more than the oracle's bound for the pages left out; and a threshold of
zero gives the dense decode bit for bit.
"""
import math

import numpy as np
import pytest

import workloads as wl
from oracle import rcp_oracle as orc
from tests.gpu_util import MAX_ABS, assert_close, make_cache, t

pytestmark = pytest.mark.gpu

TINY = wl.SHAPES["tiny"]
MAIN = wl.SHAPES["mha32"]
UNTOUCHED = 7        # page_kept entries the kernel must not write
MARGIN = 1e-2        # natural-log units: fp32 scores on the GPU against fp64 in the oracle


def _run(inp, thr, with_kept=True):
    import torch
    c = inp.cache
    cache = make_cache(inp.shape, inp.U_k, inp.W_v, c.k_pages, c.v_pages)
    kept = None
    if with_kept:
        kept = torch.full(c.block_table.shape, UNTOUCHED, dtype=torch.uint8, device="cuda")
    out = cache.decode_attn_sparse(t(inp.q), t(c.block_table), t(c.seq_lens), thr,
                                   page_kept=kept)
    torch.cuda.synchronize()
    assert cache.read_device_error() == 0
    return out.cpu().numpy(), (kept.cpu().numpy() if with_kept else None), cache


def _masks(kept, seq_lens):
    masks = []
    for b, L in enumerate(seq_lens):
        n = wl.blocks_needed(int(L))
        row = kept[b]
        assert np.all(row[n:] == UNTOUCHED), f"request {b}: entries past the sequence written"
        assert set(np.unique(row[:n]).tolist()) <= {0, 1}
        m = row[:n].astype(bool)
        if n:
            assert m[0], f"request {b}: first page left out"
        masks.append(m)
    return masks


def _check_valid(q, k_pages, U, table, seq_lens, masks, thr):
    for b, m in enumerate(masks):
        if (~m).any():
            pm = orc.page_max_scores(q[b], k_pages, U, table[b], int(seq_lens[b]))
            M = pm.max(axis=0)
            assert np.all(pm[~m] - M < math.log(thr) + MARGIN), f"request {b}: invalid skip"


def _check(inp, thr, out, kept, what):
    c = inp.cache
    masks = _masks(kept, c.seq_lens)
    _check_valid(inp.q, c.k_pages, inp.U_k, c.block_table, c.seq_lens, masks, thr)
    ref = orc.decode_attn_kept(inp.q, c.k_pages, c.v_pages, inp.U_k, inp.W_v, c.block_table,
                               c.seq_lens, masks)
    assert_close(out, ref, what=what)
    full = orc.decode_attn(inp.q, c.k_pages, c.v_pages, inp.U_k, inp.W_v, c.block_table,
                           c.seq_lens)
    bound = orc.skip_error_bound(inp.q, c.k_pages, c.v_pages, inp.U_k, inp.W_v,
                                 c.block_table, c.seq_lens, [~m for m in masks])
    assert np.all(np.abs(out - full) <= bound[:, :, None] + MAX_ABS), what
    return sum(int((~m).sum()) for m in masks), sum(len(m) for m in masks)


def test_threshold_zero_is_the_dense_decode_bit_for_bit():
    import torch
    lens = [700, 1, 16, 17, 0, 333, 1024, 40]
    inp = wl.make_decode_inputs(MAIN, lens, seed=61, fill=np.nan, peaked=wl.PEAKED)
    out, kept, cache = _run(inp, 0.0)
    c = inp.cache
    dense = cache.decode_attn(t(inp.q), t(c.block_table), t(c.seq_lens))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out, dense.cpu().numpy())
    assert all(m.all() for m in _masks(kept, c.seq_lens))


# Each work partition (one per SM) restarts its running maximum with a kept page, so the
# batches below hold enough pages for every partition to see several (a single-pass
# simulation of the partitioning drops 25-28 % of their pages).

def test_tiny_sparse_peaked_matches_oracle_on_kept_pages():
    inp = wl.make_decode_inputs(TINY, [20000, 9000, 16, 97, 0, 33, 1], seed=62, fill=np.nan,
                                peaked=wl.PEAKED)
    out, kept, _ = _run(inp, 2.0 ** -6)
    dropped, total = _check(inp, 2.0 ** -6, out, kept, "tiny sparse")
    assert dropped >= 0.15 * total, (dropped, total)


@pytest.mark.parametrize("thr", [2.0 ** -8, 2.0 ** -4])
def test_main_sparse_peaked_matches_oracle_on_kept_pages(thr):
    lens = [20000, 15000, 700, 16, 333, 0, 17, 10240, 4096, 64]
    inp = wl.make_decode_inputs(MAIN, lens, seed=63, fill=np.nan, peaked=wl.PEAKED)
    out, kept, _ = _run(inp, thr)
    dropped, total = _check(inp, thr, out, kept, f"main sparse thr={thr}")
    assert dropped >= 0.15 * total, (dropped, total)


def test_main_sparse_one_long_request_over_many_partitions():
    """One request split across every SM: each partition restarts its running maximum."""
    inp = wl.make_decode_inputs(MAIN, [40000, 3], seed=64, fill=np.nan, peaked=wl.PEAKED)
    out, kept, _ = _run(inp, 2.0 ** -8)
    dropped, total = _check(inp, 2.0 ** -8, out, kept, "long sparse")
    assert dropped >= 0.15 * total, (dropped, total)


def test_sparse_on_flat_attention_drops_nothing_unsafe():
    """N(0,1) scores: hardly any page is negligible for all 32 heads."""
    inp = wl.make_decode_inputs(MAIN, [1024, 513, 77], seed=65, fill=np.nan)
    out, kept, _ = _run(inp, 2.0 ** -8)
    _check(inp, 2.0 ** -8, out, kept, "flat sparse")


def test_sparse_is_deterministic_and_page_kept_is_optional():
    inp = wl.make_decode_inputs(MAIN, [3000, 900, 15], seed=66, fill=np.nan, peaked=wl.PEAKED)
    a, ka, _ = _run(inp, 2.0 ** -8)
    b, kb, _ = _run(inp, 2.0 ** -8)
    c, _, _ = _run(inp, 2.0 ** -8, with_kept=False)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(ka, kb)
    np.testing.assert_array_equal(a, c)


def test_sparse_rejects_bad_thresholds():
    from rank_compressed_paged_gb300 import RcpError
    inp = wl.make_decode_inputs(MAIN, [64], seed=67)
    c = inp.cache
    cache = make_cache(inp.shape, inp.U_k, inp.W_v, c.k_pages, c.v_pages)
    for bad in (1.0, -1.0, float("nan")):
        with pytest.raises(RcpError):
            cache.decode_attn_sparse(t(inp.q), t(c.block_table), t(c.seq_lens), bad)


def test_sparse_b64_l8192_peaked_sampled():
    """The benchmark's sparse workload at full size, sampled requests checked."""
    import torch
    from rank_compressed_paged_gb300 import PagedCoeffCache
    lens = np.full(64, 8192, np.int32)
    seed = 1002
    kp, vp, table, lens = wl.make_paged_cache_device(lens, MAIN, seed, device="cuda",
                                                     peaked=wl.PEAKED)
    rng = np.random.default_rng(seed)
    U, W = wl.make_factors(rng, 32, 128, 64, 1024)
    q = wl.fp16(rng.standard_normal((64, 32, 128)) * wl.PEAKED["q_scale"])
    cache = PagedCoeffCache(32, 128, 64, 1024, kp.shape[0], t(U), t(W), k_pages=kp, v_pages=vp)
    kept_t = torch.full(table.shape, UNTOUCHED, dtype=torch.uint8, device="cuda")
    out = cache.decode_attn_sparse(t(q), t(table), t(lens), 2.0 ** -8, page_kept=kept_t)
    torch.cuda.synchronize()
    assert cache.read_device_error() == 0
    out = out.cpu().numpy()
    masks = _masks(kept_t.cpu().numpy(), lens)
    frac = sum(int((~m).sum()) for m in masks) / sum(len(m) for m in masks)
    assert frac >= 0.3, frac        # about 0.41 in a single-pass simulation
    for b in (0, 37, 63):
        n = wl.blocks_needed(int(lens[b]))
        ids = torch.from_numpy(table[b, :n].astype(np.int64)).cuda()
        hk = kp.index_select(0, ids).cpu().numpy()
        hv = vp.index_select(0, ids).cpu().numpy()
        tab = np.arange(n, dtype=np.int32)[None]
        _check_valid(q[b:b + 1], hk, U, tab, lens[b:b + 1], masks[b:b + 1], 2.0 ** -8)
        ref = orc.decode_attn_kept(q[b:b + 1], hk, hv, U, W, tab, lens[b:b + 1], masks[b:b + 1])
        assert_close(out[b:b + 1], ref, what=f"sparse request {b}")


def test_sparse_is_block_relabelling_invariant():
    """Decisions depend on scores and page order only, not on physical block ids."""
    inp = wl.make_decode_inputs(MAIN, [9000, 5000, 33], seed=68, spare_blocks=9,
                                peaked=wl.PEAKED)
    a, ka, _ = _run(inp, 2.0 ** -8)
    c2 = wl.permute_physical_blocks(inp.cache, np.random.default_rng(4))
    inp2 = wl.DecodeInputs(inp.shape, inp.U_k, inp.W_v, c2, inp.q)
    b, kb, _ = _run(inp2, 2.0 ** -8)
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
    np.testing.assert_array_equal(ka, kb)
    assert (ka[:, :1] == 1).all() and (ka == 0).any()


def test_sparse_rejects_bad_block_ids_on_device():
    """A bad id sets the error bit and its page contributes nothing; others unaffected."""
    import torch
    from rank_compressed_paged_gb300 import _lib
    inp = wl.make_decode_inputs(MAIN, [3000, 3000], seed=69, peaked=wl.PEAKED)
    c = inp.cache
    table = c.block_table.copy()
    table[1, 5] = c.k_pages.shape[0] + 7            # out-of-range physical id
    cache = make_cache(inp.shape, inp.U_k, inp.W_v, c.k_pages, c.v_pages)
    kept = torch.full(table.shape, UNTOUCHED, dtype=torch.uint8, device="cuda")
    out = cache.decode_attn_sparse(t(inp.q), t(table), t(c.seq_lens), 2.0 ** -8,
                                   page_kept=kept)
    torch.cuda.synchronize()
    assert cache.read_device_error() & _lib.RCP_DEVERR_BAD_BLOCK
    o = out.cpu().numpy()
    assert np.all(np.isfinite(o))
    masks = _masks(kept.cpu().numpy(), c.seq_lens)
    ref0 = orc.decode_attn_kept(inp.q[:1], c.k_pages, c.v_pages, inp.U_k, inp.W_v, table[:1],
                                c.seq_lens[:1], masks[:1])
    assert_close(o[:1], ref0, what="unaffected request")


def test_sparse_decode_replays_from_a_cuda_graph():
    import torch
    inp = wl.make_decode_inputs(MAIN, [9000, 33, 4000, 0], seed=70, peaked=wl.PEAKED)
    c = inp.cache
    cache = make_cache(inp.shape, inp.U_k, inp.W_v, c.k_pages, c.v_pages)
    q, table, lens = t(inp.q), t(c.block_table), t(c.seq_lens)
    ws = cache.workspace(q.shape[0])
    kept = torch.zeros(c.block_table.shape, dtype=torch.uint8, device="cuda")
    eager = cache.decode_attn_sparse(q, table, lens, 2.0 ** -8, page_kept=kept,
                                     workspace=ws).clone()
    eager_kept = kept.clone()
    out = torch.empty_like(q)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):   # warm the capture stream
        cache.decode_attn_sparse(q, table, lens, 2.0 ** -8, page_kept=kept, out=out,
                                 workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    out.fill_(float("nan"))
    kept.fill_(9)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cache.decode_attn_sparse(q, table, lens, 2.0 ** -8, page_kept=kept, out=out,
                                 workspace=ws)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert cache.read_device_error() == 0
    assert np.array_equal(eager.cpu().numpy().view(np.uint16), out.cpu().numpy().view(np.uint16))
    n = [wl.blocks_needed(int(x)) for x in c.seq_lens]
    for b in range(len(n)):
        assert np.array_equal(eager_kept[b, :n[b]].cpu().numpy(), kept[b, :n[b]].cpu().numpy())
