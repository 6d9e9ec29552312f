"""The seeded workload generators (no GPU): the peaked-attention recipe of the block-sparse
benchmark scales exactly the background key pages and nothing else."""
import numpy as np
import torch

import workloads as wl

TINY = wl.SHAPES["tiny"]


def test_device_generator_peaked_scales_only_background_key_pages():
    lens = np.array([300, 17, 160, 1], np.int32)
    kp0, vp0, table0, _ = wl.make_paged_cache_device(lens, TINY, 11, device="cpu")
    kp1, vp1, table1, _ = wl.make_paged_cache_device(lens, TINY, 11, device="cpu",
                                                     peaked=wl.PEAKED)
    np.testing.assert_array_equal(table0, table1)
    assert torch.equal(vp0, vp1)                          # values untouched
    # the generator draws the table permutation first: replay both draws in order
    rng = np.random.default_rng(11)
    wl._assign_blocks(rng, lens, 0, wl.BLOCK_SIZE)
    bg = wl.background_pages(rng, lens, wl.PEAKED["background_frac"])
    scaled = set()
    for b, m in enumerate(bg):
        n = wl.blocks_needed(int(lens[b]))
        assert len(m) == n and (n == 0 or (not m[0] and not m[-1]))
        scaled |= {int(table0[b, j]) for j in np.nonzero(m)[0]}
    assert scaled, "the recipe should mark some background pages"
    for blk in range(kp0.shape[0]):
        a, c = kp0[blk].float(), kp1[blk].float()
        if blk in scaled:
            assert torch.equal((a * wl.PEAKED["background_scale"]).half().float(), c)
        else:
            assert torch.equal(a, c)


def test_host_generator_peaked_matches_its_logical_sequences():
    inp = wl.make_decode_inputs(TINY, [100, 40, 0, 16], seed=3, peaked=wl.PEAKED)
    c = inp.cache
    for b, L in enumerate(c.seq_lens):
        for t in range(int(L)):
            assert np.array_equal(c.k_pages[c.block_table[b, t // 16], :, t % 16, :], c.ck[b][t])
    assert np.abs(inp.q).max() > 5          # queries scaled up
