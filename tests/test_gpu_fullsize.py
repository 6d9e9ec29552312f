"""Full-size workloads on the GPU, checked on sampled requests against the oracle.

The GPU runs every request at the sizes and launch configuration the benchmark uses
(one CTA per SM split-K); the oracle recomputes a few sampled requests from host copies
of their *input* pages (taken before any append, which the oracle redoes itself).
"""
import numpy as np
import pytest

import workloads as wl
from oracle import rcp_oracle as orc
from tests.gpu_util import assert_close, t

pytestmark = pytest.mark.gpu

MAIN = wl.SHAPES["mha32"]


def _device_cache(seq_lens, seed, spare=16):
    import torch
    from rank_compressed_paged_gb300 import PagedCoeffCache
    kp, vp, table, lens = wl.make_paged_cache_device(seq_lens, MAIN, seed, device="cuda",
                                                     spare_blocks=spare)
    rng = np.random.default_rng(seed)
    U, W = wl.make_factors(rng, 32, 128, 64, 1024)
    cache = PagedCoeffCache(32, 128, 64, 1024, kp.shape[0], t(U), t(W), k_pages=kp, v_pages=vp)
    torch.cuda.synchronize()
    return cache, table, lens, U, W, rng


def _host_request(cache, table, b, n_blocks):
    """Host copy of request b's pages, re-addressed as blocks 0..n-1."""
    import torch
    ids = torch.from_numpy(table[b, :n_blocks].astype(np.int64)).cuda()
    kp = cache.k_pages.index_select(0, ids).cpu().numpy()
    vp = cache.v_pages.index_select(0, ids).cpu().numpy()
    return kp, vp, np.arange(n_blocks, dtype=np.int32)[None]


def _decode_sampled(seq_lens, seed, sample, append):
    import torch
    cache, table, lens, U, W, rng = _device_cache(seq_lens, seed)
    B = len(lens)
    q = wl.fp16(rng.standard_normal((B, 32, 128)))
    hosts = {b: _host_request(cache, table, b, wl.blocks_needed(lens[b])) for b in sample}
    if append:
        nk = wl.fp16(rng.standard_normal((B, 32, 128)))
        nv = wl.fp16(rng.standard_normal((B, 32, 128)))
        slots = np.array([wl.slot_for(table, b, int(lens[b]) - 1) for b in range(B)], np.int64)
        cache.append_kv(t(nk), t(nv), t(slots))
    out = cache.decode_attn(t(q), t(table), t(lens)).cpu().numpy()
    torch.cuda.synchronize()
    assert cache.read_device_error() == 0
    for b in sample:
        kp, vp, tab = hosts[b]
        if append:
            L = int(lens[b])
            kp, vp = orc.append_kv(kp, vp, U, W, nk[b:b + 1], nv[b:b + 1],
                                   np.array([(L - 1)], np.int64), 16)
        ref = orc.decode_attn(q[b:b + 1], kp, vp, U, W, tab, lens[b:b + 1], 16)
        assert_close(out[b:b + 1], ref, what=f"request {b} (L={lens[b]})")


def test_decode_b64_l8192_with_append_sampled():
    _decode_sampled(np.full(64, 8192, np.int32), 1002, [0, 37, 63], append=True)


def test_decode_b20_l32768_sampled():
    _decode_sampled(np.full(20, 32768, np.int32), 1003, [0, 19], append=False)


def test_decode_ragged64_sampled():
    lens = wl.ragged_lengths(np.random.default_rng(1003), 64, 128, 16384)
    order = np.argsort(lens)
    sample = sorted({int(order[0]), int(order[-1]), 5, 40})
    _decode_sampled(lens, 1013, sample, append=False)


@pytest.mark.parametrize("variant", ["rank", "reconstruct"])
def test_prefill_b16_p4096_c256_sampled(variant):
    import torch
    B, prior, chunk = 16, 4096, 256
    after = np.full(B, prior + chunk, np.int32)
    cache, table, lens, U, W, rng = _device_cache(after, 1004)
    T = B * chunk
    q = wl.fp16(rng.standard_normal((T, 32, 128)))
    k = wl.fp16(rng.standard_normal((T, 32, 128)))
    v = wl.fp16(rng.standard_normal((T, 32, 128)))
    slots = np.array([wl.slot_for(table, b, prior + i) for b in range(B) for i in range(chunk)],
                     np.int64)
    cu = (np.arange(B + 1) * chunk).astype(np.int32)
    sample = [0, 11]
    hosts = {b: _host_request(cache, table, b, wl.blocks_needed(after[b])) for b in sample}
    cache.append_kv(t(k), t(v), t(slots))
    out = cache.prefill_attn(t(q), t(cu), t(table), t(lens), variant=variant).cpu().numpy()
    torch.cuda.synchronize()
    assert cache.read_device_error() == 0
    for b in sample:
        kp, vp, tab = hosts[b]
        rows = slice(b * chunk, (b + 1) * chunk)
        loc = np.arange(prior, prior + chunk, dtype=np.int64)     # re-addressed slots
        kp, vp = orc.append_kv(kp, vp, U, W, k[rows], v[rows], loc, 16)
        ref = orc.prefill_attn(q[rows], np.array([0, chunk], np.int32), kp, vp, U, W, tab,
                               after[b:b + 1], 16)
        assert_close(out[rows], ref, what=f"prefill request {b} ({variant})")
