"""Block-sparse decode on E4M3 and 4-bit pages vs the oracle, through the C ABI (needs a GB300).

The pages hold the oracle's own encoding of the seeded coefficients (E4M3 codes; 4-bit codes
with fp16 scales) and the oracle reads them back as the values they stand for, so every
check of the fp16 sparse tests applies unchanged to those values: each page the kernel left
out satisfies the skipping rule against the maximum over the whole sequence; the first page
of every request is read; the output equals the oracle's attention over exactly the pages
the kernel read; and it differs from full attention by no more than the oracle's bound for
the pages left out.
"""
import math

import numpy as np
import pytest

import workloads as wl
from oracle import rcp_oracle as orc
from tests.gpu_util import MAX_ABS, assert_close, t

pytestmark = pytest.mark.gpu

TINY = wl.SHAPES["tiny"]
MAIN = wl.SHAPES["mha32"]
FORMATS = ["fp8_e4m3", "int4"]
UNTOUCHED = 7        # page_kept entries the kernel must not write
MARGIN = 1e-2        # natural-log units: fp32 scores on the GPU against fp64 in the oracle


def _dims(shape):
    return shape["num_heads"], shape["head_dim"], shape["rank_k"], shape["rank_v"]


def _encode(fmt, shape, k_pages, v_pages):
    """Page bytes in the format and the coefficient values the oracle reads from them (a
    NaN-filled slot keeps a NaN value, so reading it would poison the output)."""
    H, _, rk, R = _dims(shape)
    if fmt == "fp8_e4m3":
        kb = orc.e4m3_encode(np.asarray(k_pages, np.float64))
        vb = orc.e4m3_encode(np.asarray(v_pages, np.float64))
        return kb, vb, orc.e4m3_decode(kb), orc.e4m3_decode(vb)
    with np.errstate(invalid="ignore"):
        kc, ks, vc, vs = orc.int4_pages(k_pages, v_pages)
    kb, vb = orc.int4_pack_pages(kc, ks, vc, vs)
    kv, vv = orc.int4_page_coefficients(kb, vb, H, rk, R)
    return kb, vb, kv, vv


class _Case:
    def __init__(self, fmt, shape, lens, seed, **kw):
        from rank_compressed_paged_gb300 import PagedCoeffCache
        self.inp = wl.make_decode_inputs(shape, lens, seed=seed, fill=np.nan, **kw)
        c = self.inp.cache
        kb, vb, self.kv, self.vv = _encode(fmt, shape, c.k_pages, c.v_pages)
        H, d, rk, R = _dims(shape)
        self.cache = PagedCoeffCache(H, d, rk, R, kb.shape[0], t(self.inp.U_k), t(self.inp.W_v),
                                     k_pages=t(kb), v_pages=t(vb), page_format=fmt)

    def sparse(self, thr, with_kept=True):
        import torch
        c = self.inp.cache
        kept = None
        if with_kept:
            kept = torch.full(c.block_table.shape, UNTOUCHED, dtype=torch.uint8, device="cuda")
        out = self.cache.decode_attn_sparse(t(self.inp.q), t(c.block_table), t(c.seq_lens), thr,
                                            page_kept=kept)
        torch.cuda.synchronize()
        assert self.cache.read_device_error() == 0
        return out.cpu().numpy(), (kept.cpu().numpy() if with_kept else None)

    def dense(self):
        import torch
        c = self.inp.cache
        out = self.cache.decode_attn(t(self.inp.q), t(c.block_table), t(c.seq_lens))
        torch.cuda.synchronize()
        assert self.cache.read_device_error() == 0
        return out.cpu().numpy()

    def masks(self, kept):
        masks = []
        for b, L in enumerate(self.inp.cache.seq_lens):
            n = wl.blocks_needed(int(L))
            row = kept[b]
            assert np.all(row[n:] == UNTOUCHED), f"request {b}: entries past the sequence written"
            assert set(np.unique(row[:n]).tolist()) <= {0, 1}
            m = row[:n].astype(bool)
            if n:
                assert m[0], f"request {b}: first page left out"
            masks.append(m)
        return masks

    def check(self, thr, out, kept, what):
        inp, c = self.inp, self.inp.cache
        masks = self.masks(kept)
        for b, m in enumerate(masks):
            if (~m).any():
                pm = orc.page_max_scores(inp.q[b], self.kv, inp.U_k, c.block_table[b],
                                         int(c.seq_lens[b]))
                assert np.all(pm[~m] - pm.max(axis=0) < math.log(thr) + MARGIN), \
                    f"{what}: request {b}: invalid skip"
        ref = orc.decode_attn_kept(inp.q, self.kv, self.vv, inp.U_k, inp.W_v, c.block_table,
                                   c.seq_lens, masks)
        assert_close(out, ref, what=what)
        full = orc.decode_attn(inp.q, self.kv, self.vv, inp.U_k, inp.W_v, c.block_table,
                               c.seq_lens)
        bound = orc.skip_error_bound(inp.q, self.kv, self.vv, inp.U_k, inp.W_v, c.block_table,
                                     c.seq_lens, [~m for m in masks])
        assert np.all(np.abs(out - full) <= bound[:, :, None] + MAX_ABS), what
        return sum(int((~m).sum()) for m in masks), sum(len(m) for m in masks)


@pytest.mark.parametrize("fmt", FORMATS)
def test_quantized_sparse_tiny_peaked_matches_oracle_on_kept_pages(fmt):
    case = _Case(fmt, TINY, [20000, 9000, 16, 97, 0, 33, 1], 262, peaked=wl.PEAKED)
    out, kept = case.sparse(2.0 ** -6)
    dropped, total = case.check(2.0 ** -6, out, kept, f"{fmt} tiny sparse")
    assert np.all(out[4] == 0)
    assert dropped >= 0.15 * total, (dropped, total)


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("thr", [2.0 ** -8, 2.0 ** -4])
def test_quantized_sparse_main_peaked_matches_oracle_on_kept_pages(fmt, thr):
    lens = [20000, 15000, 700, 16, 333, 0, 17, 10240, 4096, 64]
    case = _Case(fmt, MAIN, lens, 263, peaked=wl.PEAKED)
    out, kept = case.sparse(thr)
    dropped, total = case.check(thr, out, kept, f"{fmt} main sparse thr={thr}")
    assert dropped >= 0.15 * total, (dropped, total)


@pytest.mark.parametrize("fmt", FORMATS)
def test_quantized_sparse_one_long_request_over_many_partitions(fmt):
    case = _Case(fmt, MAIN, [40000, 3], 264, peaked=wl.PEAKED)
    out, kept = case.sparse(2.0 ** -8)
    dropped, total = case.check(2.0 ** -8, out, kept, f"{fmt} long sparse")
    assert dropped >= 0.15 * total, (dropped, total)


@pytest.mark.parametrize("fmt", FORMATS)
def test_quantized_sparse_flat_attention_ragged(fmt):
    """N(0,1) scores and ragged lengths (partial last pages, an empty request)."""
    case = _Case(fmt, MAIN, [1024, 513, 77, 0, 15, 1], 265)
    out, kept = case.sparse(2.0 ** -8)
    case.check(2.0 ** -8, out, kept, f"{fmt} flat sparse")


@pytest.mark.parametrize("fmt", FORMATS)
def test_quantized_sparse_threshold_zero_keeps_every_page(fmt):
    """Threshold 0: every page read; the tiny shape scores keys on the CUDA cores in the
    dense decode too, so the two agree bit for bit there; on the main shape the dense decode
    scores on the tensor cores and both are held to the oracle."""
    tiny = _Case(fmt, TINY, [700, 1, 16, 17, 0, 333], 266, peaked=wl.PEAKED)
    out, kept = tiny.sparse(0.0)
    assert all(m.all() for m in tiny.masks(kept))
    np.testing.assert_array_equal(out, tiny.dense())
    main = _Case(fmt, MAIN, [700, 1, 16, 17, 0, 333, 1024, 40], 267, peaked=wl.PEAKED)
    out, kept = main.sparse(0.0)
    assert all(m.all() for m in main.masks(kept))
    c = main.inp.cache
    ref = orc.decode_attn(main.inp.q, main.kv, main.vv, main.inp.U_k, main.inp.W_v,
                          c.block_table, c.seq_lens)
    assert_close(out, ref, what=f"{fmt} threshold 0")
    assert_close(main.dense(), ref, what=f"{fmt} dense")


@pytest.mark.parametrize("fmt", FORMATS)
def test_quantized_sparse_is_deterministic_and_page_kept_is_optional(fmt):
    case = _Case(fmt, MAIN, [3000, 900, 15], 268, peaked=wl.PEAKED)
    a, ka = case.sparse(2.0 ** -8)
    b, kb = case.sparse(2.0 ** -8)
    c, _ = case.sparse(2.0 ** -8, with_kept=False)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(ka, kb)
    np.testing.assert_array_equal(a, c)
