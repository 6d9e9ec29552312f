"""Benchmark: one decode step (append 1 token per sequence + decode attention) at
batch 64, 8192 cached tokens per sequence, 32 heads, d=128, r_k=64, R=1024, fp16.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0).  ``value`` is algorithmic GB/s: coefficient bytes one
decode step must read ((H*r_k + R) * 2 bytes per cached token, 3,221,225,472 bytes per
GPU) divided by the device time of the whole step, summed over ranks and divided by the
slowest rank's time.  Under torchrun every rank runs its own batch of 64 independent
sequences (weak scaling, no collective on the data path).

``--impl reference`` times the fp64 CPU oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import contextlib
import datetime
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "decode-attn µs/step & GB/s at B=64,L=8192; fraction of GB300 HBM roofline"
SHAPE = wl.SHAPES["mha32"]
BATCH, SEQ = 64, 8192   # the measured configuration; --batch / --seq-len shrink it for ncu
RAGGED = None           # (lo, hi): per-sequence lengths uniform in [lo, hi] instead of SEQ
PEAKED = False          # peaked-attention pages and queries (workloads.PEAKED)
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "decode_main_b64_l8192.md")
SPARSE_PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "decode_sparse_b64_l8192_peaked.md")
E4M3_PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "decode_main_e4m3_b64_l8192.md")
INT4_PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "decode_main_int4_b64_l8192.md")
KERNEL_SRC = os.path.join(ROOT, "rank_compressed_paged_gb300", "csrc", "decode.cu")


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def rank_seed(rank: int) -> int:
    """Each rank draws its own batch of sequences (weak scaling: work per GPU is fixed)."""
    return 1002 + rank


def reduce_max(values, world: int, device=None):
    """Max over ranks of per-rank timings: the slowest rank bounds the whole job."""
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def job_gbs(bytes_per_rank: int, world: int, max_ms: float) -> float:
    """Whole-job throughput: every rank's bytes over the slowest rank's time."""
    return world * bytes_per_rank / (max_ms * 1e-3) / 1e9


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def measured_tensor_peak():
    """Sustained dense bf16 TFLOP/s (fp16 runs at the same nominal rate on tcgen05)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops_sustained"]), "measured (sustained)"
    return 1700.0, "fallback (sustained)"


def kernel_src_hash() -> str:
    """First 16 hex digits of the sha256 of the decode kernel source with its // comments
    and blank lines removed (a comment edit does not change the kernel's traffic)."""
    lines = []
    with open(KERNEL_SRC) as f:
        for ln in f.read().splitlines():
            code = ln.split("//", 1)[0].rstrip()
            if code:
                lines.append(code)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()[:16]


def ncu_traffic_per_launch(summary=None):
    """DRAM bytes per decode-kernel launch from a committed ncu summary, or None when the
    summary is missing or was taken on a different version of the kernel source."""
    summary = summary or PROFILE_SUMMARY
    if not os.path.exists(summary):
        return None
    txt = open(summary).read()
    h = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]{16})", txt)
    t = re.search(r"dram_bytes_per_launch_full_size:\s*([0-9]+)", txt)
    if not h or not t or h.group(1) != kernel_src_hash():
        return None
    return int(t.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples (every 10 ms, each with its timestamp);
    the summary keeps the samples taken while the timed region ran.  Timed regions can be
    marked (``with clk.region(): ...``); the summary then describes the first one and adds
    the samples of all marked regions of the run."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        self.t0 = self.t1 = None
        self.regions = []

    @contextlib.contextmanager
    def region(self):
        t0 = time.time()
        try:
            yield
        finally:
            self.regions.append((t0, time.time()))

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}",
                 "--query-gpu=timestamp,clocks.sm,clocks.max.sm,power.draw,"
                 "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
                 "clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "10"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        self.t0 = time.time()
        return self

    def __exit__(self, *a):
        self.t1 = time.time()
        if self.proc is not None:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def _rows(self):
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(f[1]), float(f[2]), f[5:9]))
            except ValueError:
                continue
        return rows

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = self._rows()
        os.unlink(self.path)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        regions = self.regions or [(self.t0, self.t1)]
        t0, t1 = regions[0]

        def stats(rs):
            reasons = {n for r in rs for n, v in zip(names, r[3]) if v.lower() == "active"}
            sm = [r[1] for r in rs]
            return sm, reasons

        inside = [r for r in rows if t0 <= r[0] <= t1]
        window = "timed region"
        if not inside:   # a region shorter than the sampling interval: nearest samples
            inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
            window = "timed region +- 50 ms"
        sm, reasons = stats(inside)
        out = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": inside[-1][2] if inside else None,
               "reasons": sorted(reasons), "samples": len(sm), "window": window,
               "region_s": round(t1 - t0, 3)}
        if len(regions) > 1:   # every timed region of the run (device, kernel, end to end)
            allr = [r for r in rows if any(a <= r[0] <= b for a, b in regions)]
            sm2, reasons2 = stats(allr)
            out["all_timed_regions"] = {
                "regions": len(regions), "seconds": round(sum(b - a for a, b in regions), 3),
                "samples": len(sm2), "sm_mhz": statistics.median(sm2) if sm2 else None,
                "sm_min_mhz": min(sm2) if sm2 else None, "reasons": sorted(reasons2)}
        return out


def workload_name():
    tail = "_append" + ("_peaked" if PEAKED else "")
    if RAGGED:
        return f"decode_b{BATCH}_ragged{RAGGED[0]}-{RAGGED[1]}{tail}"
    return f"decode_b{BATCH}_l{SEQ}{tail}"


def make_workload(device, seed, shape=None, batch=None, seq=None, ragged="default",
                  peaked=None):
    """Device-resident cache (pages drawn on the GPU) + the step's host inputs.  Defaults
    are the measured configuration (module globals)."""
    shape = SHAPE if shape is None else shape
    batch = BATCH if batch is None else batch
    seq = SEQ if seq is None else seq
    ragged = RAGGED if ragged == "default" else ragged
    peaked = PEAKED if peaked is None else peaked
    seq_lens = (wl.ragged_lengths(np.random.default_rng(seed + 1), batch, *ragged) if ragged
                else np.full(batch, seq, np.int32))
    kp, vp, table, seq_lens = wl.make_paged_cache_device(seq_lens, shape, seed, device=device,
                                                         spare_blocks=16,
                                                         peaked=wl.PEAKED if peaked else None)
    rng = np.random.default_rng(seed)
    H, d = shape["num_heads"], shape["head_dim"]
    U, W = wl.make_factors(rng, H, d, shape["rank_k"], shape["rank_v"])
    q = wl.fp16(rng.standard_normal((batch, H, d)) * (wl.PEAKED["q_scale"] if peaked else 1.0))
    nk = wl.fp16(rng.standard_normal((batch, H, d)))
    nv = wl.fp16(rng.standard_normal((batch, H, d)))
    slots = np.array([wl.slot_for(table, b, int(seq_lens[b]) - 1) for b in range(batch)],
                     np.int64)
    return dict(kp=kp, vp=vp, table=table, seq_lens=seq_lens, U=U, W=W, q=q, nk=nk, nv=nv,
                slots=slots, shape=shape, batch=batch)


# ------------------------------------------------------------------ CPU baseline (oracle)
def oracle_worker(job):
    """One host process of the CPU baseline: for each of its requests, draw the pages of
    one sequence of the workload (untimed), then time the oracle's append of the step's new
    token and its decode.  Runs single-threaded (the pool caps BLAS at one thread)."""
    from oracle import rcp_oracle as orc
    seed, n_req, budget_s, seq, U, W = job
    H, d, rk, R = SHAPE["num_heads"], SHAPE["head_dim"], SHAPE["rank_k"], SHAPE["rank_v"]
    rng = np.random.default_rng(seed)
    done, busy = 0, 0.0
    while done < n_req and busy < budget_s:
        nb = seq // 16
        kp = wl.fp16(rng.standard_normal((nb, H, 16, rk), dtype=np.float32))
        vp = wl.fp16(rng.standard_normal((nb, 16, R), dtype=np.float32))
        table = rng.permutation(nb).astype(np.int32)[None]
        q = wl.fp16(rng.standard_normal((1, H, d)))
        nk = wl.fp16(rng.standard_normal((1, H, d)))
        slot = np.array([wl.slot_for(table, 0, seq - 1)], np.int64)
        t0 = time.perf_counter()
        kp2, vp2 = orc.append_kv(kp, vp, U, W, nk, nk, slot, 16)
        orc.decode_attn(q, kp2, vp2, U, W, table, np.array([seq], np.int32), 16)
        busy += time.perf_counter() - t0
        done += 1
    return done, busy


def _worker_ready(i):
    return i


class OraclePool:
    """Spawn pool of single-threaded oracle workers, one per host core (a process forked
    from one that has used the GPU can hang, so the pool spawns).  The workers are started
    and idle before the constructor returns, so their start-up never overlaps a GPU timed
    region."""

    def __init__(self, workers=None):
        import multiprocessing as mp
        self.n = workers or os.cpu_count() or 1
        keys = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")
        saved = {k: os.environ.get(k) for k in keys}
        for k in keys:
            os.environ[k] = "1"
        try:
            self.pool = mp.get_context("spawn").Pool(self.n)
            self.pool.map(_worker_ready, range(4 * self.n), chunksize=1)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v

    def run(self, U, W, per_worker, seed, budget_s):
        """Every worker times up to per_worker requests; returns (requests, seconds), the
        seconds being the busiest worker's oracle time (the workers run concurrently)."""
        jobs = [(seed + 7919 * i, per_worker, budget_s, SEQ, U, W) for i in range(self.n)]
        res = self.pool.map(oracle_worker, jobs, chunksize=1)
        return sum(r[0] for r in res), max(r[1] for r in res)

    def close(self):
        self.pool.close()
        self.pool.join()


def oracle_sample(U, W, n_req, seed, budget_s):
    """Time the fp64 oracle on about n_req requests of the workload, spread over every host
    core; returns (requests, seconds, GB/s, processes)."""
    pool = OraclePool()
    try:
        per = max(1, (n_req + pool.n - 1) // pool.n)
        done, busy = pool.run(U, W, per, seed, budget_s)
    finally:
        pool.close()
    return done, busy, done * bytes_per_request() / busy / 1e9, pool.n


def bytes_per_request() -> float:
    """A request's share of the step's bytes: its coefficients plus 1/BATCH of the factors
    (the GPU step reads U_k and W_v once for the whole batch)."""
    return wl.algorithmic_bytes_decode(SHAPE, [SEQ]) + wl.factor_bytes(SHAPE) / BATCH


def blas_threads() -> int:
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(k, "").isdigit():
            return int(os.environ[k])
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    return os.cpu_count() or 1


def run_reference(args, rank, world):
    if rank != 0:
        return
    rng = np.random.default_rng(2002)
    U, W = wl.make_factors(rng, SHAPE["num_heads"], SHAPE["head_dim"], SHAPE["rank_k"],
                           SHAPE["rank_v"])
    pool = OraclePool()
    try:
        for i in range(args.warmup):
            pool.run(U, W, 1, 1 + i, 1e9)
        times, nreq = [], 0
        for s in range(args.steps):
            n, busy = pool.run(U, W, 1, 100 + s, 1e9)
            times.append(busy)
            nreq += n
    finally:
        pool.close()
    value = nreq * bytes_per_request() / sum(times) / 1e9
    sample = (f"{nreq} sequences of {SEQ} tokens in all: each step one sequence (like one of "
              f"the batch's {BATCH}) per host process, {pool.n} single-threaded processes "
              "running concurrently, append + decode, fp64 numpy oracle; a step's time is "
              "the busiest process's oracle time")
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "impl": "reference",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * sum(times) / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_name(), "batch": BATCH,
                   "seq_len": SEQ if not RAGGED else f"uniform {RAGGED[0]}..{RAGGED[1]}",
                   "num_heads": 32,
                   "head_dim": 128, "rank_k": 64, "rank_v": 1024, "block_size": 16},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": pool.n,
                         "host_cores": os.cpu_count(), "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------- GPU timing
L2_BYTES = 129e6


def time_steps(step, steps, stream, flush=None, cache=None):
    """Mean device time (ms) of one step, by CUDA events on ``stream``.  Without ``flush``
    the steps run back to back inside one event pair; with it, ``flush()`` (a write larger
    than L2) runs before each step and each step has its own event pair.  With ``cache``
    the steps are run again with its profile events around the split-K attention kernel,
    whose mean time is returned as well (else None)."""
    import torch

    def ev():
        return torch.cuda.Event(enable_timing=True)

    torch.cuda.synchronize()
    if flush is None:
        a, b = ev(), ev()
        a.record(stream)
        for _ in range(steps):
            step()
        b.record(stream)
        torch.cuda.synchronize()
        step_ms = a.elapsed_time(b) / steps
    else:
        pairs = [(ev(), ev()) for _ in range(steps)]
        for a, b in pairs:
            flush()
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize()
        step_ms = statistics.mean(a.elapsed_time(b) for a, b in pairs)
    kern_ms = None
    if cache is not None:
        pairs = [(ev(), ev()) for _ in range(steps)]
        for a, b in pairs:
            if flush is not None:
                flush()
            cache.set_profile_events(a, b)
            step()
        torch.cuda.synchronize()
        cache.set_profile_events(None, None)
        kern_ms = statistics.mean(a.elapsed_time(b) for a, b in pairs)
    return step_ms, kern_ms


def make_flush(dev):
    """A callable that overwrites a buffer of 4x the L2 size (evicts every cached line)."""
    import torch
    buf = torch.empty(int(4 * L2_BYTES), dtype=torch.uint8, device=dev)
    return lambda: buf.fill_(1)


def int4_pages_torch(kp, vp):
    """The seeded fp16 pages (device tensors [nb][H][16][r_k], [nb][16][R]) in the 4-bit
    byte format: per group (a key row of one head, 64 value coefficients of a token) the
    smallest fp16 scale with 7 * scale >= max |x| and codes x / scale rounded to nearest
    (ties to even), two per byte (the even coefficient in the low nibble), then the
    group scales.  Input preparation only, done once before timing."""
    import torch

    def enc(x, group):
        n = x.shape[-1]
        xf = x.float().reshape(*x.shape[:-1], n // group, group)
        amax = xf.abs().amax(-1)
        s = (amax / 7).half()
        s = torch.where(s.float() * 7 < amax, (s.view(torch.int16) + 1).view(torch.float16), s)
        sf = s.float().unsqueeze(-1)
        c = torch.where(sf > 0, torch.round(xf / torch.where(sf > 0, sf, 1.0)),
                        torch.zeros_like(xf)).clamp(-7, 7).to(torch.int16).reshape(x.shape)
        packed = ((c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)).to(torch.uint8)
        return packed, s

    nb = kp.shape[0]
    out = []
    for x, group in ((kp, kp.shape[-1]), (vp, 64)):
        parts = []
        for b0 in range(0, nb, 4096):   # bounded temporaries
            codes, scales = enc(x[b0:b0 + 4096], group)
            parts.append(torch.cat([codes.reshape(codes.shape[0], -1),
                                    scales.contiguous().view(torch.uint8)
                                    .reshape(codes.shape[0], -1)], dim=1))
        out.append(torch.cat(parts, dim=0))
    return out[0], out[1]


def build_decode(dev, w, pages="fp16"):
    """The library cache and device tensors of a decode workload from make_workload."""
    import torch
    from rank_compressed_paged_gb300 import PagedCoeffCache
    shape = w["shape"]

    def td(x):
        return torch.from_numpy(np.ascontiguousarray(x)).to(dev)

    kp_dev, vp_dev = w["kp"], w["vp"]
    if pages == "fp8_e4m3":
        # the same seeded coefficients stored as E4M3 codes (torch's float8 cast)
        kp_dev = kp_dev.to(torch.float8_e4m3fn).view(torch.uint8)
        vp_dev = vp_dev.to(torch.float8_e4m3fn).view(torch.uint8)
        del w["kp"], w["vp"]
        torch.cuda.empty_cache()
    elif pages == "int4":
        kp_dev, vp_dev = int4_pages_torch(kp_dev, vp_dev)
        del w["kp"], w["vp"]
        torch.cuda.empty_cache()
    cache = PagedCoeffCache(shape["num_heads"], shape["head_dim"], shape["rank_k"],
                            shape["rank_v"], kp_dev.shape[0], td(w["U"]), td(w["W"]),
                            k_pages=kp_dev, v_pages=vp_dev, page_format=pages)
    t = dict(q=td(w["q"]), nk=td(w["nk"]), nv=td(w["nv"]), slots=td(w["slots"]),
             table=td(w["table"]), lens=td(w["seq_lens"]))
    t["out"] = torch.empty_like(t["q"])
    t["ws"] = cache.workspace(w["batch"])
    return cache, t


def measure_decode_config(dev, stream, steps, warmup, shape_name, batch, seq=None,
                          ragged=None, seed=1001, pages="fp16"):
    """One decode configuration (append 1 token per sequence + decode), timed like the
    headline; inputs smaller than twice the L2 size are timed one step at a time with L2
    overwritten before each.  Returns a dict of the figures the bench line reports."""
    import torch
    shape = wl.SHAPES[shape_name]
    w = make_workload(dev, seed, shape=shape, batch=batch, seq=seq, ragged=ragged,
                      peaked=False)
    cache, t = build_decode(dev, w, pages)

    def step():
        cache.decode_step(t["nk"], t["nv"], t["slots"], t["q"], t["table"], t["lens"],
                          out=t["out"], workspace=t["ws"])

    for _ in range(max(warmup, 3)):
        step()
    coeff = wl.algorithmic_bytes_decode(shape, w["seq_lens"], pages)
    step_bytes = coeff + wl.factor_bytes(shape)
    flush = make_flush(dev) if coeff < 2 * L2_BYTES else None
    step_ms, kern_ms = time_steps(step, steps, stream, flush=flush, cache=cache)
    assert cache.read_device_error() == 0, cache.read_device_error()
    peak, kind = measured_peaks()
    res = {"shape": shape_name, "batch": batch,
           "seq_len": seq if ragged is None else f"uniform {ragged[0]}..{ragged[1]}",
           "tokens": int(np.sum(w["seq_lens"])), "pages": pages,
           "step": "append 1 token/seq + decode",
           "l2": "flushed before each timed step" if flush else "inputs larger than L2",
           "us_per_step": round(step_ms * 1e3, 2),
           "step_bytes": step_bytes, "coefficient_bytes": coeff,
           "step_gbs": round(step_bytes / (step_ms * 1e-3) / 1e9, 1),
           "step_frac_of_8TBps": round(step_bytes / (step_ms * 1e-3) / 8e12, 4),
           "kernel": "decode_main_kernel", "kernel_us": round(kern_ms * 1e3, 2),
           "kernel_gbs": round(coeff / (kern_ms * 1e-3) / 1e9, 1),
           "kernel_frac_of_peak": round(coeff / (kern_ms * 1e-3) / 1e9 / peak, 4),
           "peak_gbs": peak, "peak_kind": kind,
           "kernel_frac_of_8TBps": round(coeff / (kern_ms * 1e-3) / 8e12, 4),
           "pv_tflops_kernel": round(decode_step_flops(w["seq_lens"], shape=shape)["pv"] /
                                     (kern_ms * 1e-3) / 1e12, 2)}
    if (shape_name, batch, seq, ragged) == ("mha32", 64, 8192, None) and pages != "fp16":
        # DRAM bytes per launch from the committed ncu summary of this kernel source
        res["traffic"] = ncu_traffic_per_launch(
            E4M3_PROFILE_SUMMARY if pages == "fp8_e4m3" else INT4_PROFILE_SUMMARY)
    del cache, t, w
    torch.cuda.empty_cache()
    return res


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from rank_compressed_paged_gb300 import build as _build

    if rank == 0 or world == 1:
        _build.build()
    if world > 1:
        dist.barrier()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    # the CPU baseline's pool is spawned before the device work starts
    pool = OraclePool() if (world == 1 and not args.no_cpu_baseline) else None
    w = make_workload(dev, seed=rank_seed(rank))
    cache, tt = build_decode(dev, w, args.pages)
    q, nk, nv, slots = tt["q"], tt["nk"], tt["nv"], tt["slots"]
    table, lens, out, ws = tt["table"], tt["lens"], tt["out"], tt["ws"]
    stream = torch.cuda.current_stream()

    def step():
        if args.sparse is None:
            cache.decode_step(nk, nv, slots, q, table, lens, out=out, workspace=ws)
        else:   # the same step with the block-sparse decode
            cache.append_kv(nk, nv, slots)
            cache.decode_attn_sparse(q, table, lens, args.sparse, out=out, workspace=ws)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()

    # ---- device-timed region (inputs resident in HBM; pages 3.2 GB >> L2, no flush needed)
    s_start = torch.cuda.Event(enable_timing=True)
    s_stop = torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clk = ClockSampler(local_rank).__enter__()
    with clk.region():
        s_start.record(stream)
        for _ in range(args.steps):
            step()
        s_stop.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    step_ms = s_start.elapsed_time(s_stop) / args.steps
    # ---- the split-K attention kernel alone: events recorded around it on its stream
    # (the library then launches it in plain stream order so the events bracket it)
    k_starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    k_stops = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with clk.region():
        for i in range(args.steps):
            cache.set_profile_events(k_starts[i], k_stops[i])
            step()
        torch.cuda.synchronize()
    cache.set_profile_events(None, None)
    kern_ms = statistics.mean(a.elapsed_time(b) for a, b in zip(k_starts, k_stops))
    assert cache.read_device_error() == 0, cache.read_device_error()

    # ---- end to end through the public API with host buffers (pinned), copies included.
    # The step's inputs sit in one pinned staging buffer (as a serving loop packs them), so
    # one host->device copy brings all of them; the API gets views into the device copy.
    parts = [("q", w["q"]), ("k", w["nk"]), ("v", w["nv"]), ("s", w["slots"]),
             ("t", w["table"]), ("l", w["seq_lens"])]
    offs, nbytes = {}, 0
    for name, a in parts:
        offs[name] = nbytes
        nbytes += (a.nbytes + 255) // 256 * 256
    hbuf = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    dview = {}
    for name, a in parts:
        hbuf[offs[name]:offs[name] + a.nbytes].numpy()[:] = np.ascontiguousarray(a).view(np.uint8).ravel()
        dtype = {np.float16: torch.float16, np.int64: torch.int64, np.int32: torch.int32}[a.dtype.type]
        dview[name] = dbuf[offs[name]:offs[name] + a.nbytes].view(dtype).view(a.shape)
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = nbytes
    d2h = hout.numel() * hout.element_size()

    def e2e_step():
        dbuf.copy_(hbuf, non_blocking=True)
        if args.sparse is None:
            cache.decode_step(dview["k"], dview["v"], dview["s"], dview["q"], dview["t"],
                              dview["l"], out=out, workspace=ws)
        else:
            cache.append_kv(dview["k"], dview["v"], dview["s"])
            cache.decode_attn_sparse(dview["q"], dview["t"], dview["l"], args.sparse, out=out,
                                     workspace=ws)
        hout.copy_(out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with clk.region():
        e0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
    clk.__exit__(None, None, None)
    e2e_ms = e0.elapsed_time(e1) / args.steps

    # ---- block-sparse decode: which pages the timed configuration reads (deterministic)
    sparse = None
    coeff_bytes = wl.algorithmic_bytes_decode(SHAPE, w["seq_lens"], args.pages)
    read_bytes = coeff_bytes
    kept_tok = None   # block-sparse decode: tokens of the pages it reads
    if args.sparse is not None:
        kept = torch.zeros(w["table"].shape, dtype=torch.uint8, device=dev)
        cache.decode_attn_sparse(q, table, lens, args.sparse, page_kept=kept, out=out,
                                 workspace=ws)
        kept = kept.cpu().numpy()
        L = w["seq_lens"].astype(np.int64)
        kept_tok = sum(int(min(16, L[b] - 16 * j)) for b in range(BATCH)
                       for j in range(wl.blocks_needed(int(L[b]))) if kept[b, j])
        n_pages = sum(wl.blocks_needed(int(x)) for x in L)
        n_kept = sum(int(kept[b, :wl.blocks_needed(int(L[b]))].sum()) for b in range(BATCH))
        # keys of every token + values of the kept pages' tokens
        read_bytes = int(L.sum()) * wl.key_bytes_per_token(SHAPE, args.pages) + \
            kept_tok * wl.value_bytes_per_token(SHAPE, args.pages)
        sparse = {"threshold": args.sparse, "pages": n_pages,
                  "pages_skipped_frac": round(1 - n_kept / n_pages, 4),
                  "bytes_read": read_bytes,
                  "note": "value counts the dense decode's coefficient bytes (comparable with "
                          "the dense line on the same workload); roofline.achieved counts the "
                          "bytes the sparse pass reads (all keys, kept pages' values)"}

    # ---- aggregate over ranks (max time)
    step_ms, e2e_ms, kern_ms = reduce_max([step_ms, e2e_ms, kern_ms], world, dev)
    w_seq_lens, w_U, w_W = w["seq_lens"], w["U"], w["W"]
    del cache, tt, w, dbuf
    torch.cuda.empty_cache()

    # ---- every other configuration (1 GPU runs only; rank 0 of a replica job skips them)
    configs = None
    if world == 1 and not args.no_configs and args.sparse is None and args.pages == "fp16" \
            and not RAGGED and not PEAKED and BATCH == 64 and SEQ == 8192:
        with ClockSampler(local_rank) as cclk:
            configs = measure_configs(dev, stream, args)
        configs["clocks"] = cclk.summary()
    if rank != 0:
        if pool is not None:
            pool.close()
        return
    # the step's bytes: the coefficients plus the factors U_k and W_v, each counted once
    step_bytes = coeff_bytes + wl.factor_bytes(SHAPE)
    value = job_gbs(step_bytes, world, step_ms)
    e2e_value = job_gbs(step_bytes, world, e2e_ms)
    flops = decode_step_flops(w_seq_lens, kept_tok)
    peak, peak_kind = measured_peaks()
    achieved = read_bytes / (kern_ms * 1e-3) / 1e9
    traffic = None
    if args.pages == "fp16" and not RAGGED and BATCH == 64 and SEQ == 8192:
        if args.sparse is None and not PEAKED:
            traffic = ncu_traffic_per_launch()
        elif args.sparse == 2.0 ** -8 and PEAKED:
            traffic = ncu_traffic_per_launch(SPARSE_PROFILE_SUMMARY)
    elif args.pages != "fp16" and not RAGGED and BATCH == 64 and SEQ == 8192 and not PEAKED:
        traffic = ncu_traffic_per_launch(
            E4M3_PROFILE_SUMMARY if args.pages == "fp8_e4m3" else INT4_PROFILE_SUMMARY)
    if configs is not None:
        configs["C2_b64_l8192_append"] = {
            "see": "headline keys (value, us_per_step, roofline)", "us_per_step":
            round(step_ms * 1e3, 2), "kernel_us": round(kern_ms * 1e3, 2),
            "kernel_frac_of_peak": round(achieved / peak, 4)}
    # CPU baseline: the oracle on a bounded sample of the same workload (rank 0, N=1)
    cpu = None
    if pool is not None:
        per = max(1, (args.cpu_requests + pool.n - 1) // pool.n)
        n, busy = pool.run(w_U, w_W, per, 4242, args.cpu_budget_s)
        pool.close()
        cpu = {"value": round(n * bytes_per_request() / busy / 1e9, 4), "unit": "GB/s",
               "cores": pool.n, "host_cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{n} sequences of {SEQ} tokens (append + decode), each like one "
                         f"of the batch's {BATCH}, over {pool.n} single-threaded processes "
                         f"running concurrently; {busy:.1f} s of fp64 numpy oracle in the "
                         "busiest process"}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": round(step_ms, 4),
        "us_per_step": round(step_ms * 1e3, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"fp16": "f16", "fp8_e4m3": "e4m3 pages, f16/f32 arithmetic",
                  "int4": "4-bit pages with f16 scales, f16/f32 arithmetic"}[args.pages],
        "data": "synthetic",
        "config": {"workload": workload_name(), "batch": BATCH,
                   "seq_len": SEQ if not RAGGED else f"uniform {RAGGED[0]}..{RAGGED[1]}",
                   "num_heads": 32,
                   "head_dim": 128, "rank_k": 64, "rank_v": 1024, "block_size": 16,
                   "step": "append 1 token/seq + decode attention" +
                           (f" (block-sparse, threshold {args.sparse})" if args.sparse is not None
                            else ""), "pages": args.pages,
                   "attention": "peaked (42% background pages)" if PEAKED else "N(0,1) scores",
                   "l2": f"inputs larger than L2 ({coeff_bytes / 1e9:.2f} GB of pages per GPU), "
                         "no flush" if coeff_bytes > 2 * L2_BYTES else
                         "pages smaller than 2x L2: later steps may hit L2",
                   "parallelism": f"replicas x{world}, batch-sharded, no collective",
                   "step_bytes": {"coefficients": coeff_bytes, "factors": wl.factor_bytes(SHAPE),
                                  "value": "(coefficients + factors, each read once) / step"}},
        "step_frac_of_8TBps": round(value / world / 8000.0, 4),
        "roofline": {"bound": "hbm", "kernel": "decode_main_kernel" +
                               ("<sparse>" if args.sparse is not None else ""),
                     "achieved": round(achieved, 1), "peak": peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_bytes": read_bytes, "kernel_us": round(kern_ms * 1e3, 1),
                     "frac_of_8TBps": round(achieved / 8000.0, 4)},
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "copies": "inputs packed in one pinned buffer: one H2D copy and one D2H copy "
                          "per step, on the step's stream"},
        "contraction": {"flops_per_step": flops,
                        "tflops_step": round(world * flops["total"] / (step_ms * 1e-3) / 1e12, 2),
                        "pv_tflops_kernel": round(flops["pv"] / (kern_ms * 1e-3) / 1e12, 2),
                        "note": "P*C_v on tcgen05 (fp16 in, fp32 accumulation); scores on " +
                                ("CUDA cores" if args.pages == "fp16" or args.sparse is not None
                                 else "tcgen05 (E4M3 keys x a four-term E4M3 query split)"
                                 if args.pages == "fp8_e4m3"
                                 else "tcgen05 (4-bit codes widened to E4M3 x a four-term E4M3 "
                                      "query split, times the row scale)") +
                                "; query / output projections and the append on tcgen05"},
        "sparse": sparse,
        "gpu_launches": args.steps * LAUNCHES_PER_DECODE_STEP,
        "clocks": clk.summary(),
        "configs": configs,
    }
    print(json.dumps(line), flush=True)


# kernels one decode step launches: the append with the query projection, the split-K
# attention, the combine fused with the up-projection
LAUNCHES_PER_DECODE_STEP = 3


def measure_configs(dev, stream, args):
    """Every other configuration of the workload list, each timed on its own (one GPU):
    decode steps at the tiny shape, batch 16 x 1024, E4M3 and 4-bit pages at batch 64 x 8192,
    batch 20 x 32768, 64 ragged sequences, and the chunked prefill in both variants."""
    steps = max(args.steps, 20)
    out = {}
    out["C0_tiny_b2_l256"] = measure_decode_config(dev, stream, steps, args.warmup, "tiny", 2,
                                                   seq=256, seed=1000)
    out["C1_b16_l1024"] = measure_decode_config(dev, stream, steps, args.warmup, "mha32", 16,
                                                seq=1024, seed=1001)
    out["C2_b64_l8192_append_e4m3"] = measure_decode_config(
        dev, stream, steps, args.warmup, "mha32", 64, seq=8192, seed=1002, pages="fp8_e4m3")
    out["C2_b64_l8192_append_int4"] = measure_decode_config(
        dev, stream, steps, args.warmup, "mha32", 64, seq=8192, seed=1002, pages="int4")
    out["C3_b20_l32768"] = measure_decode_config(dev, stream, steps, args.warmup, "mha32", 20,
                                                 seq=32768, seed=1003)
    out["C3_ragged64_l128_16384"] = measure_decode_config(
        dev, stream, steps, args.warmup, "mha32", 64, ragged=(128, 16384), seed=1013)
    for variant in ("rank", "reconstruct"):
        out[f"C4_prefill_b16_p4096_c256_{variant}"] = measure_prefill(
            dev, stream, 16, 4096, 256, variant, "fp16", steps, args.warmup)
    return out


def decode_step_flops(seq_lens, kept_tokens=None, shape=None) -> dict:
    """Multiply-add work of one decode step (2 FLOPs each): P*C_v (H*R per cached token, or
    per kept token for the block-sparse decode), scores (H*r_k per token), the query and the
    output projections (H*r_k*d and H*R*d per request) and the append of one token per
    request (H*r_k*d + R*H*d)."""
    shape = SHAPE if shape is None else shape
    H, d, rk, R = shape["num_heads"], shape["head_dim"], shape["rank_k"], shape["rank_v"]
    L = int(np.sum(np.asarray(seq_lens, np.int64)))
    B = len(seq_lens)
    f = {"pv": 2 * (L if kept_tokens is None else kept_tokens) * H * R,
         "scores": 2 * L * H * rk,
         "qproj": 2 * B * H * rk * d,
         "upproj": 2 * B * H * R * d,
         "append": 2 * B * (H * rk * d + R * H * d)}
    f["total"] = sum(f.values())
    return f


def prefill_flops(prior, chunk, batch):
    """Algorithmic FLOPs of one chunked-prefill step in rank space (per request: chunk rows,
    row i attends prior + i + 1 keys): scores 2*H*r_k, weighted sum 2*H*R per attended
    key, query projection 2*H*r_k*d and up-projection 2*H*R*d per row, and the append's
    projections 2*(H*r_k*d + R*H*d) per chunk token."""
    H, d, rk, R = SHAPE["num_heads"], SHAPE["head_dim"], SHAPE["rank_k"], SHAPE["rank_v"]
    keys = batch * sum(prior + i + 1 for i in range(chunk))
    rows = batch * chunk
    attn = keys * 2 * H * (rk + R) + rows * 2 * H * (rk * d + R * d)
    append = rows * 2 * (H * rk * d + R * H * d)
    return attn, append


def prefill_recon_flops(prior, chunk, batch):
    """FLOPs the reconstructing variant executes in its attention proper: V^ = C_v W_v for
    every cached key (2*R*H*d per key), then scores 2*H*r_k and O += P V^ 2*H*d per
    attended key."""
    H, d, rk, R = SHAPE["num_heads"], SHAPE["head_dim"], SHAPE["rank_k"], SHAPE["rank_v"]
    keys = batch * sum(prior + i + 1 for i in range(chunk))
    return batch * (prior + chunk) * 2 * R * H * d + keys * 2 * H * (rk + d)


def measure_prefill(dev, stream, B, prior, chunk, variant, pages, steps, warmup):
    """Chunked prefill: append the chunk, then causal chunk attention; returns the figures
    of the prefill line (step time, the attention kernels' time and tensor rate)."""
    import torch
    from rank_compressed_paged_gb300 import PagedCoeffCache
    after = np.full(B, prior + chunk, np.int32)
    kp, vp, table, lens = wl.make_paged_cache_device(after, SHAPE, 1004, device=dev,
                                                     spare_blocks=16)
    rng = np.random.default_rng(1004)
    U, W = wl.make_factors(rng, 32, 128, 64, 1024)
    T = B * chunk

    def td(x):
        return torch.from_numpy(np.ascontiguousarray(x)).to(dev)

    q = td(wl.fp16(rng.standard_normal((T, 32, 128))))
    k = td(wl.fp16(rng.standard_normal((T, 32, 128))))
    v = td(wl.fp16(rng.standard_normal((T, 32, 128))))
    slots = td(np.array([wl.slot_for(table, b, prior + i) for b in range(B) for i in range(chunk)],
                        np.int64))
    cu = td((np.arange(B + 1) * chunk).astype(np.int32))
    if pages == "fp8_e4m3":   # the same seeded coefficients as E4M3 codes
        kp = kp.to(torch.float8_e4m3fn).view(torch.uint8)
        vp = vp.to(torch.float8_e4m3fn).view(torch.uint8)
        torch.cuda.empty_cache()
    cache = PagedCoeffCache(32, 128, 64, 1024, kp.shape[0], td(U), td(W), k_pages=kp, v_pages=vp,
                            page_format=pages)
    tab, ln = td(table), td(lens)
    out = torch.empty_like(q)
    if variant == "auto":
        from rank_compressed_paged_gb300 import RECONSTRUCT_MIN_CHUNK
        variant = "reconstruct" if (chunk >= RECONSTRUCT_MIN_CHUNK or
                                    pages == "fp8_e4m3") else "rank"
    ws = (cache.workspace(T, cache.reconstruct_workspace_bytes(T, B, table.shape[1]))
          if variant == "reconstruct" else cache.workspace(T))

    def step():
        # one call: the chunk's append and its attention (rcp_prefill_step)
        cache.prefill_step(k, v, slots, q, cu, tab, ln, out=out, workspace=ws, variant=variant)

    for _ in range(max(warmup, 3)):
        step()
    step_ms, kern_ms = time_steps(step, steps, stream, cache=cache)
    assert cache.read_device_error() == 0
    attn_f, app_f = prefill_flops(prior, chunk, B)
    kern_f = attn_f if variant == "rank" else prefill_recon_flops(prior, chunk, B)
    peak_tf, kind = measured_tensor_peak()
    res = {"variant": variant, "batch": B, "prior": prior, "chunk": chunk, "pages": pages,
           "step": "append the chunk (T = B*chunk tokens) + chunk attention, one rcp_prefill_step call",
           "ms_per_step": round(step_ms, 4),
           "algorithmic_flops": attn_f + app_f,
           "algorithmic_tflops_step": round((attn_f + app_f) / (step_ms * 1e-3) / 1e12, 2),
           "kernel": "prefill_kernel" if variant == "rank"
           else "recon_kernel + prefill_kernel (reconstructing)",
           "kernel_ms": round(kern_ms, 4), "kernel_flops_executed": kern_f,
           "kernel_tflops": round(kern_f / (kern_ms * 1e-3) / 1e12, 2),
           "kernel_frac_of_peak": round(kern_f / (kern_ms * 1e-3) / 1e12 / peak_tf, 4),
           "peak_tflops": peak_tf, "peak_kind": kind,
           "l2": "inputs larger than L2 (0.43 GB of pages, 0.57 GB of reconstructed values)"}
    del cache, kp, vp, q, k, v, out, ws
    torch.cuda.empty_cache()
    return res


def run_prefill(args):
    """Chunked prefill at batch 16, 4096 cached tokens + a 256-token chunk per request:
    append the chunk, then causal chunk attention.  One JSON line (not the default run)."""
    import torch
    from rank_compressed_paged_gb300 import build as _build
    _build.build()
    B, prior, chunk = args.prefill_batch, args.prefill_prior, args.prefill_chunk
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    with ClockSampler(0) as clk:
        r = measure_prefill(dev, stream, B, prior, chunk, args.prefill_variant, args.pages,
                            args.steps, args.warmup)
    line = {
        "metric": f"chunked-prefill ms/step & algorithmic TFLOP/s at B={B}, prior {prior} + chunk {chunk}",
        "variant": r["variant"],
        "value": r["algorithmic_tflops_step"], "unit": "TFLOP/s",
        "ms_per_step": r["ms_per_step"], "steps": args.steps, "warmup": max(args.warmup, 3),
        "higher_is_better": True, "data": "synthetic",
        "dtype": "f16" if args.pages == "fp16" else "e4m3 pages widened to f16, f16/f32 arithmetic",
        "config": {"workload": f"prefill_b{B}_p{prior}_c{chunk}", "batch": B, "prior": prior,
                   "chunk": chunk, "algorithmic_flops": r["algorithmic_flops"],
                   "step": r["step"], "pages": args.pages,
                   "value_flops": "rank-space work of the method, the same for both variants"},
        "roofline": {"bound": "tensor", "kernel": r["kernel"],
                     "achieved": r["kernel_tflops"], "peak": r["peak_tflops"],
                     "peak_kind": r["peak_kind"], "unit": "TFLOP/s",
                     "frac": r["kernel_frac_of_peak"], "kernel_ms": r["kernel_ms"],
                     "flops_per_launch": r["kernel_flops_executed"],
                     "note": "fp16 dense tensor rate = the measured bf16 sustained rate"},
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def main():
    global BATCH, SEQ, RAGGED, PEAKED
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-requests", type=int, default=64)
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other configurations (C0, C1, C3, ragged, E4M3, prefill)")
    ap.add_argument("--batch", type=int, default=BATCH)
    ap.add_argument("--seq-len", type=int, default=SEQ)
    ap.add_argument("--ragged", type=str, default=None,
                    help="LO,HI: per-sequence lengths uniform in [LO, HI] (seeded)")
    ap.add_argument("--workload", choices=["decode", "prefill"], default="decode")
    ap.add_argument("--prefill-batch", type=int, default=16)
    ap.add_argument("--prefill-variant", choices=["auto", "rank", "reconstruct"], default="auto")
    ap.add_argument("--pages", choices=["fp16", "fp8_e4m3", "int4"], default="fp16",
                    help="decode page format (fp16 is the measured configuration)")
    ap.add_argument("--prefill-prior", type=int, default=4096)
    ap.add_argument("--prefill-chunk", type=int, default=256)
    ap.add_argument("--peaked", action="store_true",
                    help="decode on peaked attention: 42%% of pages hold background keys")
    ap.add_argument("--sparse", type=float, default=None, metavar="THRESHOLD",
                    help="decode step with the block-sparse decode at this weight threshold")
    args = ap.parse_args()
    BATCH, SEQ = args.batch, args.seq_len
    PEAKED = args.peaked
    if args.workload == "prefill" and args.pages == "int4":
        ap.error("the prefill reads fp16 or E4M3 pages")
    if args.ragged:
        RAGGED = tuple(int(x) for x in args.ragged.split(","))
    rank, world, local_rank = dist_env()
    if world > 1:
        import torch.distributed as dist
        backend = "gloo" if args.impl == "reference" else "nccl"
        if backend == "nccl":
            import torch
            torch.cuda.set_device(local_rank)
        dist.init_process_group(backend)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        elif args.workload == "prefill":
            run_prefill(args)
        else:
            run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
