"""GPU decode attention vs the fp64 oracle, through the C ABI (needs a GB300)."""
import numpy as np
import pytest

import workloads as wl
from oracle import rcp_oracle as orc
from tests.gpu_util import assert_close, make_cache, t

pytestmark = pytest.mark.gpu

TINY = wl.SHAPES["tiny"]
MAIN = wl.SHAPES["mha32"]


def _run_decode(inp, q=None):
    import torch
    c = inp.cache
    cache = make_cache(inp.shape, inp.U_k, inp.W_v, c.k_pages, c.v_pages)
    out = cache.decode_attn(t(inp.q if q is None else q), t(c.block_table), t(c.seq_lens))
    torch.cuda.synchronize()
    assert cache.read_device_error() == 0
    return out.cpu().numpy(), cache


def _oracle(inp, q=None):
    c = inp.cache
    return orc.decode_attn(inp.q if q is None else q, c.k_pages, c.v_pages, inp.U_k, inp.W_v,
                           c.block_table, c.seq_lens, 16)


def test_tiny_decode_matches_oracle():
    inp = wl.make_decode_inputs(TINY, [256, 256], seed=1000, fill=np.nan)
    out, _ = _run_decode(inp)
    assert_close(out, _oracle(inp), what="tiny B2 L256")


def test_tiny_decode_ragged_and_edge_lengths():
    lens = [0, 1, 15, 16, 17, 31, 33, 255, 256, 100, 2, 64]
    inp = wl.make_decode_inputs(TINY, lens, seed=21, fill=np.nan, spare_blocks=5)
    out, _ = _run_decode(inp)
    ref = _oracle(inp)
    assert np.all(out[0] == 0)                      # empty sequence -> zeros
    assert_close(out, ref, what="tiny ragged")


def test_main_decode_b16_l1024_matches_oracle():
    inp = wl.make_decode_inputs(MAIN, [1024] * 16, seed=1001, fill=np.nan)
    out, _ = _run_decode(inp)
    assert_close(out, _oracle(inp), what="B16 L1024")


def test_main_decode_ragged_small():
    rng = np.random.default_rng(5)
    lens = list(rng.integers(1, 700, size=9)) + [0, 16, 17]
    inp = wl.make_decode_inputs(MAIN, lens, seed=22, fill=np.nan)
    out, _ = _run_decode(inp)
    assert_close(out, _oracle(inp), what="main ragged")


def test_decode_is_deterministic_and_block_relabelling_invariant():
    inp = wl.make_decode_inputs(MAIN, [700, 1024, 33], seed=23, spare_blocks=9)
    o1, cache = _run_decode(inp)
    o2, _ = _run_decode(inp)
    assert np.array_equal(o1.view(np.uint16), o2.view(np.uint16))
    c2 = wl.permute_physical_blocks(inp.cache, np.random.default_rng(3))
    inp2 = wl.DecodeInputs(inp.shape, inp.U_k, inp.W_v, c2, inp.q)
    o3, _ = _run_decode(inp2)
    assert np.array_equal(o1.view(np.uint16), o3.view(np.uint16))


def test_decode_large_score_range_exercises_rescaling():
    """Scores spanning tens of units force the running max to move mid-sequence."""
    inp = wl.make_decode_inputs(MAIN, [900, 400], seed=24)
    c = inp.cache
    kp = c.k_pages.astype(np.float32)
    # grow key coefficients along the sequence so later blocks dominate
    for b, L in enumerate(c.seq_lens):
        for tkn in range(int(L)):
            blk = c.block_table[b, tkn // 16]
            kp[blk, :, tkn % 16, :] *= 1.0 + 6.0 * tkn / L
    c.k_pages = kp.astype(np.float16)
    q = (inp.q.astype(np.float32) * 3).astype(np.float16)
    out, _ = _run_decode(inp, q)
    assert_close(out, _oracle(inp, q), what="rescale")


def test_decode_rejects_bad_block_ids_on_device():
    import torch
    from rank_compressed_paged_gb300 import _lib
    inp = wl.make_decode_inputs(TINY, [40, 40], seed=25)
    c = inp.cache
    table = c.block_table.copy()
    table[1, 1] = c.k_pages.shape[0] + 7            # out of range physical id
    cache = make_cache(inp.shape, inp.U_k, inp.W_v, c.k_pages, c.v_pages)
    out = cache.decode_attn(t(inp.q), t(table), t(c.seq_lens))
    torch.cuda.synchronize()
    assert cache.read_device_error() & _lib.RCP_DEVERR_BAD_BLOCK
    o = out.cpu().numpy()
    assert np.all(np.isfinite(o))
    ref0 = orc.decode_attn(inp.q[:1], c.k_pages, c.v_pages, inp.U_k, inp.W_v, table[:1],
                           c.seq_lens[:1], 16)
    assert_close(o[:1], ref0, what="unaffected request")


def test_main_decode_one_long_request_spans_every_partition():
    """A single long sequence is split over all CTAs: many partial records to merge."""
    inp = wl.make_decode_inputs(MAIN, [0, 12000, 0], seed=26, fill=np.nan)
    out, _ = _run_decode(inp)
    assert np.all(out[0] == 0) and np.all(out[2] == 0)
    assert_close(out, _oracle(inp), what="one long request")


def test_decode_empty_request_after_a_full_one_gives_zeros():
    """The same workspace first holds a merged z for request 0, then request 0 is empty."""
    import torch
    inp = wl.make_decode_inputs(MAIN, [500, 300], seed=27)
    c = inp.cache
    cache = make_cache(inp.shape, inp.U_k, inp.W_v, c.k_pages, c.v_pages)
    ws = cache.workspace(2)
    o1 = cache.decode_attn(t(inp.q), t(c.block_table), t(c.seq_lens), workspace=ws)
    lens2 = c.seq_lens.copy()
    lens2[0] = 0
    o2 = cache.decode_attn(t(inp.q), t(c.block_table), t(lens2), workspace=ws)
    torch.cuda.synchronize()
    assert cache.read_device_error() == 0
    o1, o2 = o1.cpu().numpy(), o2.cpu().numpy()
    assert np.any(o1[0] != 0) and np.all(o2[0] == 0)
    ref = orc.decode_attn(inp.q, c.k_pages, c.v_pages, inp.U_k, inp.W_v, c.block_table, lens2, 16)
    assert_close(o2, ref, what="empty after full")


def test_decode_with_shared_prefix_blocks():
    """Prefix caching: several requests' tables point at the same physical blocks."""
    inp = wl.make_decode_inputs(MAIN, [320, 300, 170, 16], seed=28, fill=np.nan)
    c = inp.cache
    table = c.block_table.copy()
    table[1, :10] = table[0, :10]     # request 1 shares request 0's first 160 tokens
    table[2, :5] = table[0, :5]       # request 2 shares the first 80
    table[3, 0] = table[0, 0]         # request 3 is one shared block
    inp2 = wl.DecodeInputs(inp.shape, inp.U_k, inp.W_v, c, inp.q)
    inp2.cache.block_table = table
    out, _ = _run_decode(inp2)
    assert_close(out, _oracle(inp2), what="shared prefix blocks")


def test_decode_ignores_table_entries_past_each_sequence():
    """Entries beyond ceil(L/16) are never read, so garbage there raises no error."""
    import torch
    inp = wl.make_decode_inputs(MAIN, [40, 200, 0], seed=29, fill=np.nan)
    c = inp.cache
    need = (c.seq_lens + 15) // 16
    table = np.full((3, 40), 1 << 30, np.int32)
    for b in range(3):
        table[b, :need[b]] = c.block_table[b, :need[b]]
    cache = make_cache(inp.shape, inp.U_k, inp.W_v, c.k_pages, c.v_pages)
    out = cache.decode_attn(t(inp.q), t(table), t(c.seq_lens))
    torch.cuda.synchronize()
    assert cache.read_device_error() == 0
    ref = orc.decode_attn(inp.q, c.k_pages, c.v_pages, inp.U_k, inp.W_v, table, c.seq_lens, 16)
    assert_close(out.cpu().numpy(), ref, what="padded table")
