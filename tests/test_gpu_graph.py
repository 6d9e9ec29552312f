"""The step entry points enqueue only kernels on the caller's stream (no host sync, no
allocation), so a CUDA graph can capture them; replays match eager calls bitwise."""
import numpy as np
import pytest

import workloads as wl
from tests.gpu_util import make_cache, t

pytestmark = pytest.mark.gpu

MAIN = wl.SHAPES["mha32"]


def test_decode_step_replays_from_a_cuda_graph():
    import torch
    inp = wl.make_decode_inputs(MAIN, [700, 33, 1024, 0, 160], seed=61, append=True)
    c = inp.cache
    cache = make_cache(inp.shape, inp.U_k, inp.W_v, c.k_pages, c.v_pages)
    k, v, sl, q = t(inp.new_k), t(inp.new_v), t(inp.slot_mapping), t(inp.q)
    table, lens = t(c.block_table), t(c.seq_lens)
    ws = cache.workspace(q.shape[0])
    eager = cache.decode_step(k, v, sl, q, table, lens, workspace=ws).clone()
    out = torch.empty_like(q)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):   # warm the capture stream
        cache.decode_step(k, v, sl, q, table, lens, out=out, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    out.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cache.decode_step(k, v, sl, q, table, lens, out=out, workspace=ws)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert cache.read_device_error() == 0
    assert np.array_equal(eager.cpu().numpy().view(np.uint16), out.cpu().numpy().view(np.uint16))


@pytest.mark.parametrize("variant", ["rank", "reconstruct"])
def test_prefill_replays_from_a_cuda_graph(variant):
    import torch
    inp = wl.make_prefill_inputs(MAIN, [300, 40], [130, 200], seed=62)
    c = inp.cache
    cache = make_cache(inp.shape, inp.U_k, inp.W_v, c.k_pages, c.v_pages)
    cache.append_kv(t(inp.k), t(inp.v), t(inp.slot_mapping))
    q, cu, table, lens = t(inp.q), t(inp.cu_chunk_lens), t(c.block_table), t(inp.seq_lens_after)
    ws_bytes = (cache.workspace_bytes(q.shape[0]) if variant == "rank" else
                cache.reconstruct_workspace_bytes(q.shape[0], lens.shape[0], table.shape[1]))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    eager = cache.prefill_attn(q, cu, table, lens, workspace=ws, variant=variant).clone()
    out = torch.empty_like(q)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        cache.prefill_attn(q, cu, table, lens, out=out, workspace=ws, variant=variant)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    out.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cache.prefill_attn(q, cu, table, lens, out=out, workspace=ws, variant=variant)
    g.replay()
    torch.cuda.synchronize()
    assert cache.read_device_error() == 0
    assert np.array_equal(eager.cpu().numpy().view(np.uint16), out.cpu().numpy().view(np.uint16))


@pytest.mark.parametrize("pages", ["fp8_e4m3", "int4"])
def test_quantized_decode_step_replays_from_a_cuda_graph(pages):
    """E4M3 and 4-bit pages (the oracle's encoding of the seeded coefficients): the step's
    three launches replay from a graph bit for bit as eager calls."""
    import torch
    from oracle import rcp_oracle as orc
    from rank_compressed_paged_gb300 import PagedCoeffCache
    inp = wl.make_decode_inputs(MAIN, [700, 33, 1024, 0, 160], seed=63, append=True)
    c = inp.cache
    if pages == "fp8_e4m3":
        kb = orc.e4m3_encode(c.k_pages.astype(np.float64))
        vb = orc.e4m3_encode(c.v_pages.astype(np.float64))
    else:
        kb, vb = orc.int4_pack_pages(*orc.int4_pages(c.k_pages, c.v_pages))
    cache = PagedCoeffCache(32, 128, 64, 1024, kb.shape[0], t(inp.U_k), t(inp.W_v),
                            k_pages=t(kb), v_pages=t(vb), page_format=pages)
    k, v, sl, q = t(inp.new_k), t(inp.new_v), t(inp.slot_mapping), t(inp.q)
    table, lens = t(c.block_table), t(c.seq_lens)
    ws = cache.workspace(q.shape[0])
    eager = cache.decode_step(k, v, sl, q, table, lens, workspace=ws).clone()
    out = torch.empty_like(q)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        cache.decode_step(k, v, sl, q, table, lens, out=out, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    out.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cache.decode_step(k, v, sl, q, table, lens, out=out, workspace=ws)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert cache.read_device_error() == 0
    assert np.array_equal(eager.cpu().numpy().view(np.uint16), out.cpu().numpy().view(np.uint16))
