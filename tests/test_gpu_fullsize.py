"""Full-size workloads on the GPU, every request checked against the oracle.

The GPU runs each batch at the sizes and in the launch configuration the benchmark uses
(one CTA per SM, split-K over equal slices of the global block list); partitions cut
requests at arbitrary blocks, so every request is compared, not a sample.  The oracle
recomputes each request from host copies of its *input* pages (taken before any append,
which the oracle redoes itself), in a spawn process pool.
"""
import numpy as np
import pytest

import workloads as wl
from tests.gpu_util import assert_close, t
from tests.oracle_jobs import decode_request, decode_request_quantized, prefill_request, run_pool

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
    return kp, vp


def _decode_every_request(seq_lens, seed, append):
    import torch
    cache, table, lens, U, W, rng = _device_cache(seq_lens, seed)
    B = len(lens)
    q = wl.fp16(rng.standard_normal((B, 32, 128)))
    hosts = [_host_request(cache, table, b, wl.blocks_needed(lens[b])) for b in range(B)]
    if append:
        nk = wl.fp16(rng.standard_normal((B, 32, 128)))
        nv = wl.fp16(rng.standard_normal((B, 32, 128)))
        slots = np.array([wl.slot_for(table, b, int(lens[b]) - 1) for b in range(B)], np.int64)
        cache.append_kv(t(nk), t(nv), t(slots))
    out = cache.decode_attn(t(q), t(table), t(lens)).cpu().numpy()
    torch.cuda.synchronize()
    assert cache.read_device_error() == 0
    del cache
    torch.cuda.empty_cache()
    jobs = [(q[b:b + 1], hosts[b][0], hosts[b][1], U, W, int(lens[b]),
             (nk[b:b + 1], nv[b:b + 1]) if append else None) for b in range(B)]
    hosts.clear()
    refs = run_pool(decode_request, jobs)
    for b, ref in enumerate(refs):
        assert_close(out[b:b + 1], ref, what=f"request {b} (L={lens[b]})")
    # and the batch as a whole
    assert_close(out, np.concatenate(refs), what="whole batch")


def test_decode_b64_l8192_with_append_every_request():
    _decode_every_request(np.full(64, 8192, np.int32), 1002, append=True)


def test_decode_b20_l32768_every_request():
    _decode_every_request(np.full(20, 32768, np.int32), 1003, append=False)


def test_decode_ragged64_every_request():
    lens = wl.ragged_lengths(np.random.default_rng(1003), 64, 128, 16384)
    _decode_every_request(lens, 1013, append=False)


@pytest.mark.parametrize("pages", ["fp8_e4m3", "int4"])
def test_quantized_decode_b64_l8192_every_request(pages):
    """E4M3 and 4-bit pages at the batch-64 x 8192 size: the seeded fp16 pages are encoded
    by torch casts (E4M3) or the benchmark's torch encoder (4-bit), the GPU decodes them in
    the benchmark's launch configuration, and the oracle decodes every request from host
    copies of the same bytes."""
    import torch
    import bench
    from rank_compressed_paged_gb300 import PagedCoeffCache
    lens = np.full(64, 8192, np.int32)
    kp, vp, table, lens = wl.make_paged_cache_device(lens, MAIN, 1102, device="cuda",
                                                     spare_blocks=16)
    if pages == "fp8_e4m3":
        kq = kp.to(torch.float8_e4m3fn).view(torch.uint8)
        vq = vp.to(torch.float8_e4m3fn).view(torch.uint8)
    else:
        kq, vq = bench.int4_pages_torch(kp, vp)
    del kp, vp
    torch.cuda.empty_cache()
    rng = np.random.default_rng(1102)
    U, W = wl.make_factors(rng, 32, 128, 64, 1024)
    cache = PagedCoeffCache(32, 128, 64, 1024, kq.shape[0], t(U), t(W), k_pages=kq,
                            v_pages=vq, page_format=pages)
    B = len(lens)
    q = wl.fp16(rng.standard_normal((B, 32, 128)))
    out = cache.decode_attn(t(q), t(table), t(lens)).cpu().numpy()
    torch.cuda.synchronize()
    assert cache.read_device_error() == 0
    jobs = []
    for b in range(B):
        ids = torch.from_numpy(table[b, :wl.blocks_needed(lens[b])].astype(np.int64)).cuda()
        jobs.append((q[b:b + 1], cache.k_pages.index_select(0, ids).cpu().numpy(),
                     cache.v_pages.index_select(0, ids).cpu().numpy(), U, W, int(lens[b]), pages))
    del cache, kq, vq
    torch.cuda.empty_cache()
    refs = run_pool(decode_request_quantized, jobs)
    for b, ref in enumerate(refs):
        assert_close(out[b:b + 1], ref, what=f"{pages} request {b}")


def test_prefill_b16_p4096_c256_every_request_both_variants():
    """Every request of the benchmark's prefill workload, both variants and the one-call step,
    against the oracle."""
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
    hosts = [_host_request(cache, table, b, wl.blocks_needed(after[b])) for b in range(B)]
    # the step the benchmark times (append + reconstructing prefill in one call) appends the
    # chunk; both prefill calls then attend the same pages
    outs = {"reconstruct, one step": cache.prefill_step(
        t(k), t(v), t(slots), t(q), t(cu), t(table), t(lens), variant="reconstruct").cpu().numpy()}
    for variant in ("rank", "reconstruct"):
        outs[variant] = cache.prefill_attn(t(q), t(cu), t(table), t(lens),
                                           variant=variant).cpu().numpy()
    torch.cuda.synchronize()
    assert cache.read_device_error() == 0
    del cache
    torch.cuda.empty_cache()
    jobs = []
    for b in range(B):
        rows = slice(b * chunk, (b + 1) * chunk)
        jobs.append((q[rows], k[rows], v[rows], hosts[b][0], hosts[b][1], U, W, prior, chunk))
    hosts.clear()
    refs = run_pool(prefill_request, jobs)
    for variant, out in outs.items():
        for b, ref in enumerate(refs):
            rows = slice(b * chunk, (b + 1) * chunk)
            assert_close(out[rows], ref, what=f"prefill request {b} ({variant})")
