"""Per-request oracle jobs for the full-size GPU tests, run in a spawn process pool.

Each job takes one request's *input* pages (host copies taken before the GPU ran, and
re-addressed as blocks 0..n-1) plus its query and appended rows, and returns the fp64
oracle output.  The functions only call the oracle; they are top-level so that a spawn
pool can pickle them.
"""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

from oracle import rcp_oracle as orc


def decode_request(job):
    """job: (q [1][H][d], kp, vp, U, W, L, append) with append None or (k [1][H][d],
    v [1][H][d]) written at position L - 1 before the decode."""
    q, kp, vp, U, W, L, append = job
    tab = np.arange(kp.shape[0], dtype=np.int32)[None]
    if append is not None:
        kp, vp = orc.append_kv(kp, vp, U, W, append[0], append[1],
                               np.array([L - 1], np.int64), 16)
    return orc.decode_attn(q, kp, vp, U, W, tab, np.array([L], np.int32), 16)


def decode_request_quantized(job):
    """job: (q [1][H][d], K page bytes, V page bytes, U, W, L, page format): the oracle
    decodes the bytes (E4M3 codes, or 4-bit codes with their scales) and attends them."""
    q, kb, vb, U, W, L, fmt = job
    if fmt == "fp8_e4m3":
        kp, vp = orc.e4m3_decode(kb), orc.e4m3_decode(vb)
    else:
        H, rk, R = U.shape[0], U.shape[1], W.shape[0]
        kp, vp = orc.int4_page_coefficients(kb, vb, H, rk, R)
    tab = np.arange(kp.shape[0], dtype=np.int32)[None]
    return orc.decode_attn(q, kp, vp, U, W, tab, np.array([L], np.int32), 16)


def prefill_request(job):
    """job: (q, k, v rows of the chunk, kp, vp, U, W, prior, chunk): the chunk is appended
    at positions prior .. prior + chunk - 1, then the chunk's rows attend causally."""
    q, k, v, kp, vp, U, W, prior, chunk = job
    tab = np.arange(kp.shape[0], dtype=np.int32)[None]
    slots = np.arange(prior, prior + chunk, dtype=np.int64)
    kp, vp = orc.append_kv(kp, vp, U, W, k, v, slots, 16)
    return orc.prefill_attn(q, np.array([0, chunk], np.int32), kp, vp, U, W, tab,
                            np.array([prior + chunk], np.int32), 16)


def run_pool(fn, jobs, workers: int | None = None):
    """fn over jobs in a spawn pool (a forked child of a process that has used the GPU can
    hang).  BLAS threads per worker are capped so that the workers share the cores."""
    cores = os.cpu_count() or 2
    n = workers or max(1, min(len(jobs), 8, cores // 2))
    keys = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in keys}
    for k in keys:
        os.environ[k] = str(max(1, cores // n))
    try:
        with mp.get_context("spawn").Pool(n) as pool:
            return pool.map(fn, jobs, chunksize=1)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
