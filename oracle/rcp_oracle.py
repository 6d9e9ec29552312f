"""Oracle for rank-compressed paged attention: a plain, slow fp64 CPU restatement.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links this
module; only the tests, the package smoke check and the benchmark's CPU-baseline leg do.
It shares no code with the CUDA library.

What it computes follows the Proxima page (STAR-KV plugin for vLLM), intro paragraph:
keys use a head-wise low-rank decomposition and values a joint one, kept in a compressed
paged format; its "Per-decode-step attention" and "Per-prefill-chunk attention" sections
name the two attention steps, and its "Kernel profiling breakdown" names the cache-write
step (low-rank projection of each new token).  The page prints no equations; the exact
definitions used here are:

* append:   c_k[t,h] = fp16(U_k,h k_{t,h}),   c_v[t] = fp16(W_v v_t)
            (v_t is the head-major concatenation of the H head vectors), written to
            K page [s // bs][h][s % bs][:] and V page [s // bs][s % bs][:] for slot s;
            slot -1 writes nothing.
* decode:   q~_h = U_k,h q_h;  s_{h,t} = q~_h . c_k[t,h] / sqrt(d) for t < L;
            p_h = softmax(s_h) (max subtracted first);  z_h = sum_t p_{h,t} c_v[t];
            o_h = W_v[:, h*d:(h+1)*d]^T z_h.
            Token t of request b lives in block block_table[b][t // bs] at offset t % bs.
            L = 0 gives o = 0.
* prefill:  the chunk is appended first; chunk query i of request b sits at absolute
            position P_b + i with P_b = seq_len_b - chunk_len_b and attends keys
            t <= P_b + i, read back from the pages (i.e. after fp16 rounding).

All arithmetic is fp64 on the stored fp16 values; results are fp64 (fp16 only where the
definition stores fp16: the coefficients an append writes).

fp8 pages (E4M3 codes, see e4m3_encode) hold the same coefficients rounded to E4M3 instead
of fp16; decode over them is the decode above on the decoded values.

Pins (see tests/test_oracle.py): identity factors reduce decode to textbook multi-head
attention computed by a library routine; explicit reconstruction K = C_k U_k, V = C_v W_v
followed by library attention agrees to 1e-12; physical block permutation leaves outputs
bitwise unchanged; softmax weights sum to 1; single-token, equal-key, power-of-two
scaling, causal-prefill and hand-derived closed-form cases; coordinate-selection factors
make appends exact copies.  Block-sparse skipping (tests/test_oracle_sparse.py): attention
over a page subset equals attention over a compacted block table and a scalar textbook
loop; the skippable set matches a hand-built score pattern; a sequential running-maximum
pass drops a subset of it; the output change stays within the derived bound.  4-bit
pages and rotation (tests/test_oracle_int4.py): grid values round-trip exactly, codes are
the nearest grid points by enumeration, errors stay within half a step without saturation,
a hand-packed byte fixes the nibble order, a hand-packed page (tests/golden/int4_page.json)
fixes the page layout, every group an append writes is re-derived by enumeration, and a
rotation folded into the factors leaves decode unchanged.
"""
from __future__ import annotations

import numpy as np


def _f64(a) -> np.ndarray:
    return np.asarray(a).astype(np.float64)


def gather_request(k_pages, v_pages, block_table_row, seq_len: int, block_size: int):
    """Logical-order coefficients of one request through its block-table row.

    Returns c_k [L][H][r_k] and c_v [L][R] (fp64).  Token t is in physical block
    block_table_row[t // block_size] at offset t % block_size (the paged layout the
    Proxima page's intro calls "compressed paged format", addressed the vLLM way).
    """
    t = np.arange(int(seq_len))
    row = np.asarray(block_table_row, dtype=np.int64)
    blocks = row[t // block_size]
    offs = t % block_size
    ck = _f64(k_pages[blocks, :, offs, :])      # advanced indices first: [L, H, r_k]
    cv = _f64(v_pages[blocks, offs, :])         # [L, R]
    return ck, cv


def attend(q, ck, cv, U_k, W_v, head_dim: int, n_keys=None):
    """Rank-space attention of one query set against one request's coefficients.

    q: [Q][H][d]; ck: [L][H][r_k]; cv: [L][R]; n_keys[i] = number of leading keys query i
    may attend (default: all L).  Returns (o [Q][H][d], p [Q][H][L]) in fp64.
    """
    q = _f64(q)
    U = _f64(U_k)
    W = _f64(W_v)
    nq, H, d = q.shape
    L = ck.shape[0]
    if n_keys is None:
        n_keys = np.full(nq, L)
    o = np.zeros((nq, H, d))
    p_all = np.zeros((nq, H, L))
    for i in range(nq):
        n = int(n_keys[i])
        if n == 0:
            continue
        qt = np.einsum("hkd,hd->hk", U, q[i])                     # q~_h = U_k,h q_h
        s = np.einsum("thk,hk->ht", ck[:n], qt) / np.sqrt(head_dim)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        p = e / e.sum(axis=1, keepdims=True)                       # [H][n]
        z = p @ cv[:n]                                             # [H][R]
        for h in range(H):
            o[i, h] = W[:, h * d:(h + 1) * d].T @ z[h]            # o_h = W_v,h^T z_h
        p_all[i, :, :n] = p
    return o, p_all


def decode_attn(q, k_pages, v_pages, U_k, W_v, block_table, seq_lens, block_size: int = 16,
                requests=None, return_weights: bool = False):
    """Decode attention for a batch: one query per request.

    q [B][H][d]; returns o [B][H][d] fp64 (only rows in ``requests`` if given, else all)
    and, if asked, the list of softmax weight arrays [H][L_b].
    """
    q = np.asarray(q)
    B, H, d = q.shape
    reqs = range(B) if requests is None else list(requests)
    out = np.zeros((len(reqs), H, d))
    weights = []
    for n, b in enumerate(reqs):
        L = int(seq_lens[b])
        ck, cv = gather_request(k_pages, v_pages, block_table[b], L, block_size)
        o, p = attend(q[b:b + 1], ck, cv, U_k, W_v, d)
        out[n] = o[0]
        weights.append(p[0])
    return (out, weights) if return_weights else out


# ------------------------------------------------------------------ block-sparse skipping
# The "KV-cache LLM serving" page's sparse decode (its BLASST kernels, "What it measured",
# item 3) skips blocks whose weights are small, judged with the online softmax.
# Here a block is a page, and the value coefficients of a page are shared by every head
# (joint decomposition), so a page's values can only be left out when no head needs them.
# Readings taken (the page gives no formula): a page is dropped when, for every head, its
# largest weight is below ``threshold`` times that head's largest weight so far; a
# dropped page takes part in neither the numerator nor the denominator of the softmax.
# Which pages a single pass drops depends on the order it meets them in, so the oracle
# provides (a) attention restricted to any given set of pages, (b) the set of pages that
# any order may drop (judged against the maximum over the whole sequence, the largest
# value a running maximum can reach), and (c) the bound on the output change that
# dropping a set of pages can cause.

def page_max_scores(q, k_pages, U_k, block_table_row, seq_len: int, block_size: int = 16):
    """Largest score (natural-log units) of each head in each page of one request.

    q [H][d]; returns [n_pages][H] fp64 with n_pages = ceil(seq_len / block_size).
    """
    q = _f64(q)
    H, d = q.shape
    L = int(seq_len)
    t = np.arange(L)
    blocks = np.asarray(block_table_row, dtype=np.int64)[t // block_size]
    ck = _f64(k_pages[blocks, :, t % block_size, :])                   # [L][H][r_k]
    qt = np.einsum("hkd,hd->hk", _f64(U_k), q)
    s = np.einsum("thk,hk->th", ck, qt) / np.sqrt(d)                # [L][H]
    n_pages = (L + block_size - 1) // block_size
    out = np.full((n_pages, H), -np.inf)
    for j in range(n_pages):
        out[j] = s[j * block_size:min(L, (j + 1) * block_size)].max(axis=0)
    return out


def skippable_pages(q, k_pages, U_k, block_table, seq_lens, threshold: float,
                    block_size: int = 16):
    """Pages that skipping with weight threshold ``threshold`` may drop, per request.

    Page j of request b qualifies when, for every head h, exp(max_t in page s_{h,t} - M_h)
    < threshold, with M_h the largest score of head h over the whole sequence.  Returns a
    list of bool arrays [n_pages_b].  A running maximum never exceeds M_h, so a single pass
    in any page order drops a subset of these.
    """
    q = np.asarray(q)
    res = []
    for b in range(q.shape[0]):
        L = int(seq_lens[b])
        if L == 0:
            res.append(np.zeros(0, bool))
            continue
        pm = page_max_scores(q[b], k_pages, U_k, block_table[b], L, block_size)
        M = pm.max(axis=0)
        res.append(np.all(pm - M < np.log(threshold), axis=1) if threshold > 0
                   else np.zeros(pm.shape[0], bool))
    return res


def decode_attn_kept(q, k_pages, v_pages, U_k, W_v, block_table, seq_lens, kept,
                     block_size: int = 16):
    """Decode attention over the kept pages only: token t of request b takes part iff
    kept[b][t // block_size].  A request with no kept token gives zeros."""
    q = np.asarray(q)
    B, H, d = q.shape
    out = np.zeros((B, H, d))
    for b in range(B):
        L = int(seq_lens[b])
        ck, cv = gather_request(k_pages, v_pages, block_table[b], L, block_size)
        sel = np.array([bool(kept[b][t // block_size]) for t in range(L)], dtype=bool)
        if sel.any():
            out[b] = attend(q[b:b + 1], ck[sel], cv[sel], U_k, W_v, d)[0][0]
    return out


def skip_error_bound(q, k_pages, v_pages, U_k, W_v, block_table, seq_lens, dropped,
                     block_size: int = 16):
    """Largest change, per (request, head), that leaving out the dropped pages can make to
    the decode output.

    With A the kept set and S the dropped one, weights w_t = exp(s_t - max),
    o_all = (sum_A w v + sum_S w v) / (sum_A w + sum_S w) and o_A = sum_A w v / sum_A w, so
    o_A - o_all = (w_S / w_all) (o_A - sum_S w v / w_S) and every component is at most
    (w_S / w_all) * 2 max_t |v_t| in size, v_t = W_v,h^T c_v[t] the value of token t.
    Returns [B][H] fp64.
    """
    q = np.asarray(q)
    B, H, d = q.shape
    W = _f64(W_v)
    bound = np.zeros((B, H))
    for b in range(B):
        L = int(seq_lens[b])
        if L == 0:
            continue
        ck, cv = gather_request(k_pages, v_pages, block_table[b], L, block_size)
        qt = np.einsum("hkd,hd->hk", _f64(U_k), _f64(q[b]))
        s = np.einsum("thk,hk->ht", ck, qt) / np.sqrt(d)              # [H][L]
        w = np.exp(s - s.max(axis=1, keepdims=True))
        drop = np.array([bool(dropped[b][t // block_size]) for t in range(L)], dtype=bool)
        for h in range(H):
            vmax = np.abs(cv @ W[:, h * d:(h + 1) * d]).max()
            bound[b, h] = w[h, drop].sum() / w[h].sum() * 2.0 * vmax
    return bound


def append_kv(k_pages, v_pages, U_k, W_v, k, v, slot_mapping, block_size: int = 16):
    """Project new tokens to coefficients and write them at their slots (returns copies).

    k, v: [T][H][d]; slot_mapping: [T]; slot -1 is skipped.  Coefficients are rounded
    from fp64 to fp16 (nearest, ties to even).
    """
    kp = np.array(k_pages, copy=True)
    vp = np.array(v_pages, copy=True)
    U = _f64(U_k)
    W = _f64(W_v)
    k = _f64(k)
    v = _f64(v)
    T, H, d = k.shape
    for i in range(T):
        s = int(slot_mapping[i])
        if s < 0:
            continue
        blk, off = s // block_size, s % block_size
        for h in range(H):
            kp[blk, h, off, :] = (U[h] @ k[i, h]).astype(np.float16)
        vp[blk, off, :] = (W @ v[i].reshape(H * d)).astype(np.float16)
    return kp, vp


# ---------------------------------------------------------------------------------------
# fp8 coefficient pages.  E4M3 as defined by the OCP 8-bit floating point format (the
# "E4M3" encoding, also NVIDIA's e4m3): sign bit, 4 exponent bits with bias 7, 3 mantissa
# bits; exponent field 0 holds subnormals m * 2^-9; no infinities; S.1111.111 is NaN, so
# the largest finite magnitude is S.1111.110 = 1.75 * 2^8 = 448.

def e4m3_decode(codes) -> np.ndarray:
    """fp64 values of E4M3 codes (uint8 array)."""
    c = np.asarray(codes).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * 2.0 ** (e - 7))
    mag = np.where((e == 0xF) & (m == 0x7), np.nan, mag)
    return sign * mag


_E4M3_POS = e4m3_decode(np.arange(0x7F))        # codes 0x00 .. 0x7E, ascending, 0 .. 448


def e4m3_encode(x) -> np.ndarray:
    """Nearest E4M3 code to each value (ties to the even code), magnitudes above 448
    saturating to 448 (the "satfinite" conversion), NaN to 0x7F; the sign of zero kept."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    hi = np.clip(np.searchsorted(_E4M3_POS, a, side="left"), 1, 0x7E)
    lo = hi - 1
    d_lo = a - _E4M3_POS[lo]
    d_hi = _E4M3_POS[hi] - a
    code = np.where(d_lo < d_hi, lo, np.where(d_hi < d_lo, hi, np.where(lo % 2 == 0, lo, hi)))
    code = np.where(a >= 448.0, 0x7E, code)
    code = np.where(a == 0.0, 0, code)
    code = code | np.where(np.signbit(x), 0x80, 0)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def append_kv_fp8(k_pages, v_pages, U_k, W_v, k, v, slot_mapping, block_size: int = 16):
    """append_kv for E4M3 pages: the same projections, rounded from fp64 to E4M3 codes
    (uint8 pages, same layout).  Read the pages back with e4m3_decode."""
    kp = np.array(k_pages, copy=True)
    vp = np.array(v_pages, copy=True)
    U = _f64(U_k)
    W = _f64(W_v)
    k = _f64(k)
    v = _f64(v)
    T, H, d = k.shape
    for i in range(T):
        s = int(slot_mapping[i])
        if s < 0:
            continue
        blk, off = s // block_size, s % block_size
        for h in range(H):
            kp[blk, h, off, :] = e4m3_encode(U[h] @ k[i, h])
        vp[blk, off, :] = e4m3_encode(W @ v[i].reshape(H * d))
    return kp, vp


# ------------------------------------------------------ 4-bit coefficient pages, rotation
# The "KV-cache LLM serving" page's TurboQuant pages rotate before they quantize to 4 bits,
# which keeps accuracy ("What it measured", item 1).  The page gives no format; readings
# taken here:
#   * codes are symmetric 4-bit integers in [-7, 7], one fp16 scale per group: a group is
#     one (token, head) key row (r_k values) or 64 consecutive joint value coefficients;
#   * the scale is max|x| / 7 of the group, rounded up to the next fp16 so that no code
#     saturates; code = round-half-even(x / scale); a group of zeros has scale 0, codes 0;
#   * two codes per byte, even index in the low nibble, two's complement;
#   * the rotation is an orthogonal matrix applied to the coefficients before they are
#     quantized.  It folds into the factors (U_k,h -> Q_h U_k,h, W_v -> Q W_v): every score
#     and output is unchanged, so it needs no step of its own at decode time.

def int4_encode(x, group: int):
    """Codes (int8 in [-7, 7], same shape as x) and fp16 scales ([..., n / group]) of x,
    grouped along its last axis."""
    x = _f64(x)
    n = x.shape[-1]
    assert n % group == 0
    g = x.reshape(x.shape[:-1] + (n // group, group))
    amax = np.abs(g).max(axis=-1)
    s = (amax / 7.0).astype(np.float16)
    low = s.astype(np.float64) * 7.0 < amax                 # fp16 rounding went down
    s[low] = np.nextafter(s[low], np.float16(np.inf))
    s64 = s.astype(np.float64)[..., None]
    q = np.where(s64 > 0, g / np.where(s64 > 0, s64, 1.0), 0.0)
    codes = np.clip(np.round(q), -7, 7).astype(np.int8)     # np.round: half to even
    return codes.reshape(x.shape), s


def int4_decode(codes, scales, group: int) -> np.ndarray:
    """fp64 values code * scale of its group."""
    c = np.asarray(codes, np.float64)
    n = c.shape[-1]
    g = c.reshape(c.shape[:-1] + (n // group, group))
    return (g * np.asarray(scales, np.float64)[..., None]).reshape(c.shape)


def pack_int4(codes) -> np.ndarray:
    """Two codes per byte along the last axis: even index in the low nibble."""
    c = np.asarray(codes, np.int16) & 0xF
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_int4(packed) -> np.ndarray:
    """Inverse of pack_int4 (int8 codes, sign-extended nibbles)."""
    p = np.asarray(packed, np.int16)
    lo, hi = p & 0xF, (p >> 4) & 0xF
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), np.int16)
    out[..., 0::2], out[..., 1::2] = lo, hi
    return np.where(out >= 8, out - 16, out).astype(np.int8)


def rotate_factors(U_k, W_v, Q_k, Q_v):
    """Factors with the coefficient rotation folded in: U_k,h -> Q_k[h] U_k,h (Q_k [H][r_k]
    [r_k] orthogonal) and W_v -> Q_v W_v (Q_v [R][R] orthogonal), in fp64."""
    U = np.einsum("hij,hjd->hid", _f64(Q_k), _f64(U_k))
    W = _f64(Q_v) @ _f64(W_v)
    return U, W


def int4_pages(k_pages, v_pages, v_group: int = 64):
    """Quantize coefficient pages (fp64 values) to 4 bits: K groups are the r_k values of one
    (block, head, slot) row, V groups v_group consecutive joint coefficients.  Returns
    (k_codes, k_scales, v_codes, v_scales) with codes unpacked (int8)."""
    kc, ks = int4_encode(k_pages, _f64(k_pages).shape[-1])
    vc, vs = int4_encode(v_pages, v_group)
    return kc, ks[..., 0], vc, vs


def int4_page_values(kc, ks, vc, vs, v_group: int = 64):
    """The coefficient values 4-bit pages hold (fp64), for the decode definition above."""
    kv = int4_decode(kc, ks[..., None], kc.shape[-1])
    vv = int4_decode(vc, vs, v_group)
    return kv, vv


# The 4-bit page format (bytes per physical block; reading taken for the page layout, the
# page gives none): a K page holds the codes of its [H][bs][r_k] coefficients packed two
# per byte (pack_int4 along r_k), then the fp16 scales [H][bs] of its key rows; a V page
# holds the codes of its [bs][R] coefficients packed along R, then the fp16 scales
# [bs][R / 64] of its 64-coefficient groups.  Little-endian fp16.

def int4_page_bytes(num_heads: int, rank_k: int, rank_v: int, block_size: int = 16):
    """(bytes of a K page, bytes of a V page) in the 4-bit format."""
    kb = num_heads * block_size * rank_k // 2 + num_heads * block_size * 2
    vb = block_size * rank_v // 2 + block_size * (rank_v // 64) * 2
    return kb, vb


def int4_pack_pages(kc, ks, vc, vs):
    """Byte pages [nb][K bytes], [nb][V bytes] from codes kc [nb][H][bs][r_k] (int8),
    scales ks [nb][H][bs] (fp16), codes vc [nb][bs][R], scales vs [nb][bs][R / 64]."""
    nb = np.asarray(kc).shape[0]
    kb = np.concatenate([pack_int4(kc).reshape(nb, -1),
                         np.ascontiguousarray(np.asarray(ks, np.float16)).reshape(nb, -1)
                         .view(np.uint8)], axis=1)
    vb = np.concatenate([pack_int4(vc).reshape(nb, -1),
                         np.ascontiguousarray(np.asarray(vs, np.float16)).reshape(nb, -1)
                         .view(np.uint8)], axis=1)
    return kb, vb


def int4_unpack_pages(k_bytes, v_bytes, num_heads: int, rank_k: int, rank_v: int,
                      block_size: int = 16):
    """Inverse of int4_pack_pages: (kc, ks, vc, vs)."""
    kb = np.asarray(k_bytes, np.uint8)
    vb = np.asarray(v_bytes, np.uint8)
    nb = kb.shape[0]
    nk = num_heads * block_size * rank_k // 2
    nv = block_size * rank_v // 2
    kc = unpack_int4(kb[:, :nk].reshape(nb, num_heads, block_size, rank_k // 2))
    ks = np.ascontiguousarray(kb[:, nk:]).view(np.float16).reshape(nb, num_heads, block_size)
    vc = unpack_int4(vb[:, :nv].reshape(nb, block_size, rank_v // 2))
    vs = np.ascontiguousarray(vb[:, nv:]).view(np.float16).reshape(nb, block_size, rank_v // 64)
    return kc, ks, vc, vs


def int4_page_coefficients(k_bytes, v_bytes, num_heads: int, rank_k: int, rank_v: int,
                           block_size: int = 16):
    """The coefficient values (fp64) 4-bit byte pages hold, as K pages [nb][H][bs][r_k] and
    V pages [nb][bs][R] for the decode and prefill definitions above."""
    kc, ks, vc, vs = int4_unpack_pages(k_bytes, v_bytes, num_heads, rank_k, rank_v, block_size)
    return int4_page_values(kc, ks, vc, vs, 64)


def append_kv_int4(k_bytes, v_bytes, U_k, W_v, k, v, slot_mapping, block_size: int = 16):
    """append_kv for 4-bit pages (returns copies): each new token's projections (fp64) are
    quantized per group (int4_encode: a key row of r_k values, 64 value coefficients) and
    written, codes and scales, at its slot; slot -1 writes nothing."""
    U = _f64(U_k)
    W = _f64(W_v)
    k = _f64(k)
    v = _f64(v)
    T, H, d = k.shape
    rk, R = U.shape[1], W.shape[0]
    kc, ks, vc, vs = int4_unpack_pages(k_bytes, v_bytes, H, rk, R, block_size)
    kc, ks, vc, vs = kc.copy(), ks.copy(), vc.copy(), vs.copy()
    for i in range(T):
        s = int(slot_mapping[i])
        if s < 0:
            continue
        blk, off = s // block_size, s % block_size
        for h in range(H):
            c, sc = int4_encode(U[h] @ k[i, h], rk)
            kc[blk, h, off] = c
            ks[blk, h, off] = sc[0]
        c, sc = int4_encode(W @ v[i].reshape(H * d), 64)
        vc[blk, off] = c
        vs[blk, off] = sc
    return int4_pack_pages(kc, ks, vc, vs)


def prefill_attn(q, cu_chunk_lens, k_pages, v_pages, U_k, W_v, block_table, seq_lens,
                 block_size: int = 16, requests=None):
    """Chunked-prefill attention over pages that already hold the chunk.

    q: [sum chunk][H][d]; cu_chunk_lens [B+1]; seq_lens [B] include the chunk.  Returns
    o [sum chunk][H][d] fp64 (rows of requests not in ``requests`` stay zero).
    """
    q = np.asarray(q)
    T, H, d = q.shape
    out = np.zeros((T, H, d))
    B = len(seq_lens)
    reqs = range(B) if requests is None else list(requests)
    for b in reqs:
        c0, c1 = int(cu_chunk_lens[b]), int(cu_chunk_lens[b + 1])
        n = c1 - c0
        if n == 0:
            continue
        L = int(seq_lens[b])
        P = L - n
        ck, cv = gather_request(k_pages, v_pages, block_table[b], L, block_size)
        n_keys = P + 1 + np.arange(n)                  # causal: query i sees t <= P + i
        o, _ = attend(q[c0:c1], ck, cv, U_k, W_v, d, n_keys=n_keys)
        out[c0:c1] = o
    return out
