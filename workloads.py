"""Seeded synthetic inputs for rank-compressed paged attention.

This module only draws random numbers and lays them out in the paged format; it holds
none of the attention arithmetic (no projection into rank space, no score, softmax or
contraction).  The oracle-side tests, the GPU tests, ``bench.py`` and the smoke run all
take their inputs from here, so both sides of every parity check see identical bytes.

Workloads mirror the decode / prefill shapes of the Proxima page ("Per-decode-step
attention": 32-head MHA, head size 128, key rank 64, fp16, block size 16), with a joint
value rank of 1024.  Coefficients are N(0,1) rounded to fp16; factors have orthonormal
rows taken from a Householder QR of an N(0,1) matrix (fp64), rounded to fp16.

Two generation routes exist:

* ``make_paged_cache`` (numpy, host): draws *logical* per-request coefficient sequences
  first, then scatters them into physical blocks through a seeded permutation.  Tests use
  the logical sequences as an independent view of the cache.
* ``make_paged_cache_device`` (torch on a CUDA device): fills every physical page
  directly with seeded normal draws; used for the multi-GB workloads where host
  generation would take minutes.  Parity at that size copies the sampled requests' pages
  back to the host for the oracle.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BLOCK_SIZE = 16

# Model shapes: (num_heads H, head_dim d, key rank r_k, joint value rank R).
SHAPES = {
    "tiny": dict(num_heads=4, head_dim=64, rank_k=16, rank_v=64),
    "mha32": dict(num_heads=32, head_dim=128, rank_k=64, rank_v=1024),
}

# Named workloads.  ``seed`` = 1000 + position in the list of configurations.
WORKLOADS = {
    "decode_tiny_b2_l256": dict(shape="tiny", kind="decode", batch=2, seq_len=256, seed=1000),
    "decode_b16_l1024": dict(shape="mha32", kind="decode", batch=16, seq_len=1024, seed=1001),
    "decode_b64_l8192_append": dict(shape="mha32", kind="decode", batch=64, seq_len=8192,
                                    append=True, seed=1002),
    "decode_b20_l32768": dict(shape="mha32", kind="decode", batch=20, seq_len=32768, seed=1003),
    "decode_ragged64_l128_16384": dict(shape="mha32", kind="decode", batch=64,
                                       len_range=(128, 16384), seed=1003),
    "prefill_b16_p4096_c256": dict(shape="mha32", kind="prefill", batch=16, prior=4096,
                                   chunk=256, seed=1004),
}


# Peaked attention for the block-sparse decode.  The sparse-decode measurements on the
# "KV-cache LLM serving" page come from a real model whose attention leaves about 42 % of
# KV blocks with negligible weight ("What it measured", item 3, and "What did not work").
# Synthetic stand-in: a random 42 % of each request's pages (never its first page, the
# attention sink, nor its last, the recent tokens) hold background keys whose coefficients
# are scaled down 16x, and queries are scaled up 6x, so that the remaining pages dominate
# every head's softmax.
PEAKED = dict(background_frac=0.42, background_scale=1.0 / 16, q_scale=6.0)


def background_pages(rng: np.random.Generator, seq_lens, frac: float,
                     block_size: int = BLOCK_SIZE) -> list:
    """Per request, a bool array over its pages: True marks a background page.  Each
    page is drawn independently with probability ``frac``; the first and the last page of
    a request are never background."""
    out = []
    for L in seq_lens:
        n = blocks_needed(int(L), block_size)
        m = rng.random(n) < frac
        if n:
            m[0] = False
            m[-1] = False
        out.append(m)
    return out


def fp16(x) -> np.ndarray:
    """Round to fp16 (numpy rounds float64 -> float16 to nearest, ties to even)."""
    return np.asarray(x, dtype=np.float64).astype(np.float16)


def orthonormal_rows(rng: np.random.Generator, rows: int, cols: int) -> np.ndarray:
    """fp64 matrix [rows][cols] with orthonormal rows (rows <= cols).

    The first ``rows`` columns of Q from a Householder QR of a cols x rows N(0,1) matrix,
    transposed.
    """
    assert rows <= cols
    g = rng.standard_normal((cols, rows))
    q, _ = np.linalg.qr(g, mode="reduced")
    return q.T.copy()


def make_factors(rng: np.random.Generator, num_heads: int, head_dim: int, rank_k: int,
                 rank_v: int):
    """U_k [H][r_k][d] and W_v [R][H*d], fp16, orthonormal rows before rounding."""
    U = np.stack([orthonormal_rows(rng, rank_k, head_dim) for _ in range(num_heads)])
    W = orthonormal_rows(rng, rank_v, num_heads * head_dim)
    return fp16(U), fp16(W)


def identity_factors(num_heads: int, head_dim: int):
    """U_k,h = I_d (r_k = d) and W_v = I (R = H*d)."""
    U = np.stack([np.eye(head_dim) for _ in range(num_heads)])
    W = np.eye(num_heads * head_dim)
    return fp16(U), fp16(W)


def selection_factors(rng: np.random.Generator, num_heads: int, head_dim: int, rank_k: int,
                      rank_v: int):
    """Factors whose rows are distinct unit vectors (coordinate selections).

    Projecting with them picks coordinates exactly, so coefficients written by an append
    are exact copies of chosen input entries.
    """
    U = np.zeros((num_heads, rank_k, head_dim))
    for h in range(num_heads):
        cols = rng.permutation(head_dim)[:rank_k]
        U[h, np.arange(rank_k), cols] = 1.0
    W = np.zeros((rank_v, num_heads * head_dim))
    cols = rng.permutation(num_heads * head_dim)[:rank_v]
    W[np.arange(rank_v), cols] = 1.0
    return fp16(U), fp16(W)


def pair_sum_factors(rng: np.random.Generator, num_heads: int, head_dim: int, rank_k: int,
                     rank_v: int):
    """Factors whose rows each hold two unit entries in distinct, seeded columns.

    Projecting with them sums two chosen input entries per output.  With inputs from
    ``fp16_narrow`` every such sum is exact in fp32 (and in fp64), so rounding the sum to
    the page format is the only rounding an append performs.
    """
    U = np.zeros((num_heads, rank_k, head_dim))
    for h in range(num_heads):
        for k in range(rank_k):
            a, b = rng.choice(head_dim, size=2, replace=False)
            U[h, k, a] = U[h, k, b] = 1.0
    W = np.zeros((rank_v, num_heads * head_dim))
    for r in range(rank_v):
        a, b = rng.choice(num_heads * head_dim, size=2, replace=False)
        W[r, a] = W[r, b] = 1.0
    return fp16(U), fp16(W)


def fp16_narrow(rng: np.random.Generator, shape, emin: int = -4, emax: int = 3) -> np.ndarray:
    """fp16 values with a random sign, a binary exponent uniform in [emin, emax] and a
    uniformly random 10-bit fraction.  Two of them differ by at most emax - emin binades,
    so their sum needs at most 11 + (emax - emin) + 1 significant bits: exact in fp32 for
    the default range (19 bits), while most sums carry bits below fp16 precision and some
    sit exactly halfway between two fp16 neighbours."""
    e = rng.integers(emin, emax + 1, size=shape)
    frac = rng.integers(0, 1024, size=shape)
    sign = np.where(rng.random(shape) < 0.5, -1.0, 1.0)
    return fp16(sign * (1.0 + frac / 1024.0) * np.exp2(e))


def blocks_needed(seq_len: int, block_size: int = BLOCK_SIZE) -> int:
    return (int(seq_len) + block_size - 1) // block_size


@dataclass
class PagedCache:
    """A filled paged coefficient cache and the tables that address it."""
    k_pages: np.ndarray          # [num_blocks][H][bs][r_k] fp16
    v_pages: np.ndarray          # [num_blocks][bs][R] fp16
    block_table: np.ndarray      # [B][max_blocks] int32, -1 past a request's blocks
    seq_lens: np.ndarray         # [B] int32
    spare_blocks: np.ndarray     # physical ids not referenced by any request
    ck: list = field(default_factory=list)   # per request [L_b][H][r_k] fp16 (logical order)
    cv: list = field(default_factory=list)   # per request [L_b][R] fp16


def _assign_blocks(rng, seq_lens, spare_blocks, block_size, max_blocks=None):
    nblk = [blocks_needed(L, block_size) for L in seq_lens]
    used = int(sum(nblk))
    num_blocks = used + int(spare_blocks)
    perm = rng.permutation(num_blocks).astype(np.int32)
    mb = max(1, max(nblk) if nblk else 1)
    if max_blocks is not None:
        mb = max(mb, int(max_blocks))
    table = np.full((len(seq_lens), mb), -1, dtype=np.int32)
    cur = 0
    for b, n in enumerate(nblk):
        table[b, :n] = perm[cur:cur + n]
        cur += n
    return num_blocks, table, perm[used:].copy()


def make_paged_cache(rng: np.random.Generator, num_heads: int, rank_k: int, rank_v: int,
                     seq_lens, block_size: int = BLOCK_SIZE, spare_blocks: int = 0,
                     fill: float = 0.0, max_blocks: int | None = None) -> PagedCache:
    """Random logical coefficient sequences scattered into shuffled physical blocks.

    Slots that hold no token keep ``fill`` (tests use NaN to prove those slots are never
    read into a result).
    """
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    num_blocks, table, spare = _assign_blocks(rng, seq_lens, spare_blocks, block_size,
                                              max_blocks)
    kp = np.full((num_blocks, num_heads, block_size, rank_k), fill, dtype=np.float16)
    vp = np.full((num_blocks, block_size, rank_v), fill, dtype=np.float16)
    cks, cvs = [], []
    for b, L in enumerate(seq_lens):
        ck = fp16(rng.standard_normal((int(L), num_heads, rank_k)))
        cv = fp16(rng.standard_normal((int(L), rank_v)))
        for t in range(int(L)):
            blk = table[b, t // block_size]
            off = t % block_size
            kp[blk, :, off, :] = ck[t]
            vp[blk, off, :] = cv[t]
        cks.append(ck)
        cvs.append(cv)
    return PagedCache(kp, vp, table, seq_lens, spare, cks, cvs)


def permute_physical_blocks(cache: PagedCache, rng: np.random.Generator) -> PagedCache:
    """Same logical cache, physical blocks relabelled by a random permutation."""
    nb = cache.k_pages.shape[0]
    perm = rng.permutation(nb)               # new id of old block i is perm[i]
    kp = np.empty_like(cache.k_pages)
    vp = np.empty_like(cache.v_pages)
    kp[perm] = cache.k_pages
    vp[perm] = cache.v_pages
    table = cache.block_table.copy()
    m = table >= 0
    table[m] = perm[table[m]]
    return PagedCache(kp, vp, table, cache.seq_lens.copy(), perm[cache.spare_blocks],
                      cache.ck, cache.cv)


def slot_for(block_table: np.ndarray, b: int, pos: int, block_size: int = BLOCK_SIZE) -> int:
    """vLLM slot convention: physical block * block_size + offset in block."""
    return int(block_table[b, pos // block_size]) * block_size + pos % block_size


def ragged_lengths(rng: np.random.Generator, batch: int, lo: int, hi: int) -> np.ndarray:
    return rng.integers(lo, hi + 1, size=batch).astype(np.int32)


# ----------------------------------------------------------------------------- host workloads

@dataclass
class DecodeInputs:
    shape: dict
    U_k: np.ndarray
    W_v: np.ndarray
    cache: PagedCache
    q: np.ndarray                      # [B][H][d] fp16
    new_k: np.ndarray | None = None    # [B][H][d] fp16 (appended token, position L-1)
    new_v: np.ndarray | None = None
    slot_mapping: np.ndarray | None = None   # [B] int64
    background: list | None = None     # peaked workloads: per request, background pages


def make_decode_inputs(shape: dict, seq_lens, seed: int, append: bool = False,
                       spare_blocks: int = 4, fill: float = 0.0,
                       max_blocks: int | None = None, peaked: dict | None = None) -> DecodeInputs:
    """Host-side decode workload.

    Draw order: factors, K/V coefficient sequences (with the block permutation), q, then
    the appended token's k and v, then (``peaked``, e.g. ``PEAKED``) the background pages,
    whose key coefficients are then scaled by ``background_scale``; q is scaled by
    ``q_scale``.
    """
    rng = np.random.default_rng(seed)
    H, d, rk, R = shape["num_heads"], shape["head_dim"], shape["rank_k"], shape["rank_v"]
    U, W = make_factors(rng, H, d, rk, R)
    cache = make_paged_cache(rng, H, rk, R, seq_lens, spare_blocks=spare_blocks, fill=fill,
                             max_blocks=max_blocks)
    B = len(cache.seq_lens)
    q = fp16(rng.standard_normal((B, H, d)))
    out = DecodeInputs(shape, U, W, cache, q)
    if append:
        out.new_k = fp16(rng.standard_normal((B, H, d)))
        out.new_v = fp16(rng.standard_normal((B, H, d)))
        out.slot_mapping = np.array(
            [slot_for(cache.block_table, b, int(L) - 1) if L > 0 else -1
             for b, L in enumerate(cache.seq_lens)], dtype=np.int64)
    if peaked:
        bg = background_pages(rng, cache.seq_lens, peaked["background_frac"])
        scale = peaked["background_scale"]
        for b, m in enumerate(bg):
            for j in np.nonzero(m)[0]:
                blk = cache.block_table[b, j]
                cache.k_pages[blk] = fp16(cache.k_pages[blk].astype(np.float64) * scale)
                lo, hi = j * BLOCK_SIZE, min(int(cache.seq_lens[b]), (j + 1) * BLOCK_SIZE)
                cache.ck[b][lo:hi] = cache.k_pages[blk][:, :hi - lo, :].transpose(1, 0, 2)
        out.q = fp16(q.astype(np.float64) * peaked["q_scale"])
        out.background = bg
    return out


@dataclass
class PrefillInputs:
    shape: dict
    U_k: np.ndarray
    W_v: np.ndarray
    cache: PagedCache                  # holds prior tokens; chunk slots start as ``fill``
    prior_lens: np.ndarray             # [B]
    chunk_lens: np.ndarray             # [B]
    cu_chunk_lens: np.ndarray          # [B+1] int32
    q: np.ndarray                      # [sum chunk][H][d]
    k: np.ndarray                      # [sum chunk][H][d]
    v: np.ndarray                      # [sum chunk][H][d]
    slot_mapping: np.ndarray           # [sum chunk] int64
    seq_lens_after: np.ndarray         # [B] prior + chunk


def make_prefill_inputs(shape: dict, prior_lens, chunk_lens, seed: int, spare_blocks: int = 4,
                        fill: float = 0.0) -> PrefillInputs:
    """Host-side chunked-prefill workload.

    The cache holds ``prior_lens[b]`` random tokens; the blocks for the chunk are assigned
    up front (their slots hold ``fill`` until the chunk is appended).  Draw order:
    factors, prior coefficients, q, k, v of the chunk.
    """
    rng = np.random.default_rng(seed)
    H, d, rk, R = shape["num_heads"], shape["head_dim"], shape["rank_k"], shape["rank_v"]
    U, W = make_factors(rng, H, d, rk, R)
    prior = np.asarray(prior_lens, dtype=np.int32)
    chunk = np.asarray(chunk_lens, dtype=np.int32)
    after = prior + chunk
    cache = make_paged_cache(rng, H, rk, R, prior, spare_blocks=spare_blocks, fill=fill,
                             max_blocks=max(blocks_needed(x) for x in after) if len(after) else 1)
    # extend each request's block list so that prior+chunk tokens fit
    extra = [blocks_needed(a) - blocks_needed(p) for a, p in zip(after, prior)]
    need = int(sum(extra))
    nb0 = cache.k_pages.shape[0]
    new_ids = (nb0 + rng.permutation(need)).astype(np.int32)
    kp = np.concatenate([cache.k_pages,
                         np.full((need,) + cache.k_pages.shape[1:], fill, np.float16)])
    vp = np.concatenate([cache.v_pages,
                         np.full((need,) + cache.v_pages.shape[1:], fill, np.float16)])
    table = cache.block_table
    cur = 0
    for b in range(len(prior)):
        n0 = blocks_needed(prior[b])
        table[b, n0:n0 + extra[b]] = new_ids[cur:cur + extra[b]]
        cur += extra[b]
    cache = PagedCache(kp, vp, table, after.copy(), cache.spare_blocks, cache.ck, cache.cv)
    T = int(chunk.sum())
    cu = np.zeros(len(chunk) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(chunk)
    q = fp16(rng.standard_normal((T, H, d)))
    k = fp16(rng.standard_normal((T, H, d)))
    v = fp16(rng.standard_normal((T, H, d)))
    slots = np.empty(T, dtype=np.int64)
    for b in range(len(chunk)):
        for i in range(int(chunk[b])):
            slots[cu[b] + i] = slot_for(table, b, int(prior[b]) + i)
    return PrefillInputs(shape, U, W, cache, prior, chunk, cu, q, k, v, slots, after)


# --------------------------------------------------------------------------- device workloads

def make_paged_cache_device(seq_lens, shape: dict, seed: int, device="cuda",
                            spare_blocks: int = 0, block_size: int = BLOCK_SIZE,
                            chunk_blocks: int = 4096, peaked: dict | None = None):
    """Fill every physical page of a (multi-GB) cache with seeded N(0,1) fp16 on the device.

    Returns (k_pages, v_pages, block_table numpy int32, seq_lens numpy int32).  The block
    permutation is drawn on the host (numpy, ``seed``); page values by a torch generator
    seeded with ``seed`` on ``device``, in chunks of ``chunk_blocks`` blocks.  With
    ``peaked`` the background pages are then drawn on the host (same numpy stream) and
    their key coefficients scaled by ``background_scale`` (q scaling is the caller's).
    """
    import torch
    rng = np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    num_blocks, table, _ = _assign_blocks(rng, seq_lens, spare_blocks, block_size)
    H, rk, R = shape["num_heads"], shape["rank_k"], shape["rank_v"]
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    kp = torch.empty((num_blocks, H, block_size, rk), dtype=torch.float16, device=device)
    vp = torch.empty((num_blocks, block_size, R), dtype=torch.float16, device=device)
    for s in range(0, num_blocks, chunk_blocks):
        e = min(num_blocks, s + chunk_blocks)
        kp[s:e] = torch.randn((e - s, H, block_size, rk), generator=g, device=device,
                              dtype=torch.float32).half()
        vp[s:e] = torch.randn((e - s, block_size, R), generator=g, device=device,
                              dtype=torch.float32).half()
    if peaked:
        bg = background_pages(rng, seq_lens, peaked["background_frac"], block_size)
        ids = np.concatenate([table[b, :len(m)][m] for b, m in enumerate(bg)] + [
            np.zeros(0, np.int32)]).astype(np.int64)
        for s in range(0, len(ids), chunk_blocks):
            idx = torch.from_numpy(ids[s:s + chunk_blocks]).to(device)
            kp[idx] = (kp[idx].float() * peaked["background_scale"]).half()
    return kp, vp, table, seq_lens


def key_bytes_per_token(shape: dict, pages: str = "fp16") -> int:
    """Bytes of K pages per cached token: H*r_k coefficients at 2 bytes (fp16) or 1 (E4M3);
    4-bit pages hold half a byte per coefficient plus an fp16 scale per key row of a head."""
    H, rk = shape["num_heads"], shape["rank_k"]
    if pages == "fp16":
        return H * rk * 2
    if pages == "fp8_e4m3":
        return H * rk
    if pages == "int4":
        return H * rk // 2 + 2 * H
    raise ValueError(pages)


def value_bytes_per_token(shape: dict, pages: str = "fp16") -> int:
    """Bytes of V pages per cached token: R coefficients at 2 bytes (fp16) or 1 (E4M3);
    4-bit pages hold half a byte per coefficient plus an fp16 scale per 64 of them."""
    R = shape["rank_v"]
    if pages == "fp16":
        return R * 2
    if pages == "fp8_e4m3":
        return R
    if pages == "int4":
        return R // 2 + 2 * (R // 64)
    raise ValueError(pages)


def page_bytes_per_token(shape: dict, pages: str = "fp16") -> int:
    """Bytes of K and V pages per cached token."""
    return key_bytes_per_token(shape, pages) + value_bytes_per_token(shape, pages)


def algorithmic_bytes_decode(shape: dict, seq_lens, pages: str = "fp16") -> int:
    """Page bytes one decode step reads: page_bytes_per_token per cached token."""
    return int(np.sum(np.asarray(seq_lens, dtype=np.int64))) * page_bytes_per_token(shape, pages)


def factor_bytes(shape: dict) -> int:
    H, d, rk, R = shape["num_heads"], shape["head_dim"], shape["rank_k"], shape["rank_v"]
    return (H * rk * d + R * H * d) * 2

