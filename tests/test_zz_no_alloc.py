"""The decode entry point that allocates nothing (needs a GB300).

Some callers cannot allocate device memory at all: a host runtime that owns every byte of
device memory and gives its plugins no workspace, or a serving loop that must not call
cudaMalloc once it runs.  rcp_decode_attn_noalloc serves them with a fixed scratch array
inside the library.  This file checks, through the C ABI, that two calls in a row (the
second on different inputs, over the scratch the first one left behind) agree with the
workspace-taking rcp_decode_attn within the parity tolerance, and that a batch beyond the
scratch limit is refused without a launch.  It is collected last so that a run stopping
at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import workloads as wl
from oracle import rcp_oracle as orc
from tests.gpu_util import assert_close, make_cache, t

pytestmark = pytest.mark.gpu

MAIN = wl.SHAPES["mha32"]


def _noalloc(cache, q, table, lens, out):
    import torch
    from rank_compressed_paged_gb300 import _lib
    lib = _lib.load()
    return lib.rcp_decode_attn_noalloc(cache._h, q.data_ptr(), table.data_ptr(),
                                       int(table.shape[1]), lens.data_ptr(), int(q.shape[0]),
                                       out.data_ptr(), torch.cuda.current_stream().cuda_stream)


def test_noalloc_decode_matches_workspace_decode_on_two_calls():
    import torch
    from rank_compressed_paged_gb300 import _lib
    inp = wl.make_decode_inputs(MAIN, [1024] * 16, seed=1001, fill=np.nan)
    c = inp.cache
    cache = make_cache(inp.shape, inp.U_k, inp.W_v, c.k_pages, c.v_pages)
    table = t(c.block_table)
    rng = np.random.default_rng(77)
    q2 = wl.fp16(rng.standard_normal(inp.q.shape))
    lens2 = rng.integers(0, 1025, size=16).astype(np.int32)
    cases = [(inp.q, c.seq_lens), (q2, lens2)]
    for qh, lh in cases:
        q, lens = t(qh), t(lh)
        ref = cache.decode_attn(q, table, lens)
        out = torch.full_like(q, float("nan"))
        assert _noalloc(cache, q, table, lens, out) == _lib.RCP_OK
        torch.cuda.synchronize()
        assert cache.read_device_error() == 0
        got = out.cpu().numpy()
        assert_close(got, ref.cpu().numpy().astype(np.float64), what="noalloc vs workspace")
        # and against the fp64 oracle on the same inputs
        oref = orc.decode_attn(qh, c.k_pages, c.v_pages, inp.U_k, inp.W_v, c.block_table, lh, 16)
        assert_close(got, oref, what="noalloc vs oracle")


def test_noalloc_limit_is_batch_157_at_the_main_shape():
    """The header's limit for (H, d, r_k, R) = (32, 128, 64, 1024): batch 157 runs, batch
    158 is refused without a launch."""
    import torch
    from rank_compressed_paged_gb300 import _lib
    inp = wl.make_decode_inputs(MAIN, [16], seed=5)
    c = inp.cache
    cache = make_cache(inp.shape, inp.U_k, inp.W_v, c.k_pages, c.v_pages)
    assert cache.workspace_bytes(157) <= _lib.RCP_NOALLOC_SCRATCH_BYTES
    assert cache.workspace_bytes(158) > _lib.RCP_NOALLOC_SCRATCH_BYTES
    for big, want in ((157, _lib.RCP_OK), (158, _lib.RCP_ERR_WORKSPACE)):
        q = torch.zeros((big, 32, 128), dtype=torch.float16, device="cuda")
        lens = torch.zeros(big, dtype=torch.int32, device="cuda")        # empty sequences
        table = torch.zeros((big, 1), dtype=torch.int32, device="cuda")
        out = torch.full_like(q, float("nan"))
        assert _noalloc(cache, q, table, lens, out) == want
        torch.cuda.synchronize()
        if want == _lib.RCP_OK:
            assert cache.read_device_error() == 0
            assert torch.all(out == 0)                 # L = 0 gives zeros
