"""Batches with many more requests than work partitions (one per SM), against the oracle.

A partition then covers pages of many requests, so segments start and end inside it,
records outnumber requests only slightly, the plan's per-thread ranges hold several
requests each, and the combine runs one CTA row per request.
"""
import math

import numpy as np
import pytest

import workloads as wl
from oracle import rcp_oracle as orc
from tests.gpu_util import assert_close, make_cache, t

pytestmark = pytest.mark.gpu

MAIN = wl.SHAPES["mha32"]


def test_decode_640_short_requests():
    import torch
    rng = np.random.default_rng(101)
    lens = rng.integers(0, 65, size=640)
    inp = wl.make_decode_inputs(MAIN, lens, seed=101, fill=np.nan)
    c = inp.cache
    cache = make_cache(inp.shape, inp.U_k, inp.W_v, c.k_pages, c.v_pages)
    out = cache.decode_attn(t(inp.q), t(c.block_table), t(c.seq_lens))
    torch.cuda.synchronize()
    assert cache.read_device_error() == 0
    out = out.cpu().numpy()
    assert np.all(out[lens == 0] == 0)
    ref = orc.decode_attn(inp.q, c.k_pages, c.v_pages, inp.U_k, inp.W_v, c.block_table,
                          c.seq_lens, 16)
    assert_close(out, ref, what="640 short requests")


@pytest.mark.parametrize("variant", ["rank", "reconstruct"])
def test_prefill_160_requests_small_chunks(variant):
    import torch
    rng = np.random.default_rng(102)
    prior = rng.integers(0, 200, size=160)
    chunk = rng.integers(0, 25, size=160)
    inp = wl.make_prefill_inputs(MAIN, prior, chunk, seed=102, fill=np.nan)
    c = inp.cache
    cache = make_cache(inp.shape, inp.U_k, inp.W_v, c.k_pages, c.v_pages)
    cache.append_kv(t(inp.k), t(inp.v), t(inp.slot_mapping))
    out = cache.prefill_attn(t(inp.q), t(inp.cu_chunk_lens), t(c.block_table),
                             t(inp.seq_lens_after), variant=variant)
    torch.cuda.synchronize()
    assert cache.read_device_error() == 0
    kp, vp = orc.append_kv(c.k_pages, c.v_pages, inp.U_k, inp.W_v, inp.k, inp.v,
                           inp.slot_mapping, 16)
    ref = orc.prefill_attn(inp.q, inp.cu_chunk_lens, kp, vp, inp.U_k, inp.W_v, c.block_table,
                           inp.seq_lens_after, 16)
    assert_close(out.cpu().numpy(), ref, what=f"160-request prefill ({variant})")


def test_sparse_decode_400_short_requests():
    """Every request restarts the running maximum: skips are rare but must be valid."""
    import torch
    rng = np.random.default_rng(103)
    lens = rng.integers(1, 200, size=400)
    inp = wl.make_decode_inputs(MAIN, lens, seed=103, fill=np.nan, peaked=wl.PEAKED)
    c = inp.cache
    cache = make_cache(inp.shape, inp.U_k, inp.W_v, c.k_pages, c.v_pages)
    kept = torch.full(c.block_table.shape, 7, dtype=torch.uint8, device="cuda")
    out = cache.decode_attn_sparse(t(inp.q), t(c.block_table), t(c.seq_lens), 2.0 ** -8,
                                   page_kept=kept)
    torch.cuda.synchronize()
    assert cache.read_device_error() == 0
    kept = kept.cpu().numpy()
    masks = []
    for b, L in enumerate(c.seq_lens):
        n = wl.blocks_needed(int(L))
        assert np.all(kept[b, n:] == 7) and kept[b, 0] == 1
        masks.append(kept[b, :n].astype(bool))
        if (~masks[-1]).any():
            pm = orc.page_max_scores(inp.q[b], c.k_pages, inp.U_k, c.block_table[b], int(L))
            assert np.all(pm[~masks[-1]] - pm.max(axis=0) < math.log(2.0 ** -8) + 1e-2)
    ref = orc.decode_attn_kept(inp.q, c.k_pages, c.v_pages, inp.U_k, inp.W_v, c.block_table,
                               c.seq_lens, masks)
    assert_close(out.cpu().numpy(), ref, what="400-request sparse decode")
