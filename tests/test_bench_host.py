"""Host-side logic of bench.py (no GPU): clock-sample windowing, the source hash that gates
recorded DRAM traffic, byte accounting, and the reference arm's JSON line."""
import datetime
import json
import os
import subprocess
import sys
import time

import numpy as np

import bench
import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _sample_line(ts, sm, reasons=("Not Active",) * 4):
    stamp = datetime.datetime.fromtimestamp(ts).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return f"{stamp}, {sm}, 2070, 900.00, 0x0, " + ", ".join(reasons) + "\n"


def test_clock_summary_keeps_only_samples_inside_the_timed_region():
    c = bench.ClockSampler(0)
    now = time.time()
    c.t0, c.t1 = now, now + 0.1
    c.proc = object()                       # as if nvidia-smi had been started
    with open(c.path, "w") as f:
        f.write(_sample_line(now - 0.2, 1000, ("Active",) * 4))   # before: ignored
        f.write(_sample_line(now + 0.02, 2070))
        f.write(_sample_line(now + 0.05, 2060, ("Not Active", "Not Active", "Not Active",
                                                "Active")))
        f.write(_sample_line(now + 0.08, 2070))
        f.write(_sample_line(now + 0.3, 900, ("Active",) * 4))    # after: ignored
        f.write("garbage line\n")
    s = c.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"] and s["window"] == "timed region"
    assert not os.path.exists(c.path)


def test_clock_summary_widens_the_window_for_a_short_region():
    c = bench.ClockSampler(0)
    now = time.time()
    c.t0, c.t1 = now, now + 0.001
    c.proc = object()
    with open(c.path, "w") as f:
        f.write(_sample_line(now + 0.02, 2070))
    s = c.summary()
    assert s["samples"] == 1 and s["window"] == "timed region +- 50 ms"


def test_clock_summary_describes_the_first_region_and_counts_all_marked_ones():
    c = bench.ClockSampler(0)
    now = time.time()
    c.t0, c.t1 = now, now + 1.0
    c.regions = [(now, now + 0.1), (now + 0.3, now + 0.4), (now + 0.6, now + 0.7)]
    c.proc = object()
    with open(c.path, "w") as f:
        f.write(_sample_line(now + 0.05, 2070))                   # first region
        f.write(_sample_line(now + 0.2, 1000, ("Active",) * 4))   # between regions: ignored
        f.write(_sample_line(now + 0.35, 1980))                   # second region
        f.write(_sample_line(now + 0.65, 2070, ("Not Active", "Not Active", "Not Active",
                                                "Active")))       # third region
    s = c.summary()
    assert s["samples"] == 1 and s["sm_mhz"] == 2070.0 and s["reasons"] == []
    a = s["all_timed_regions"]
    assert a["regions"] == 3 and a["samples"] == 3 and a["sm_min_mhz"] == 1980.0
    assert a["sm_mhz"] == 2070.0 and a["reasons"] == ["sw_power_cap"]


def test_source_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("int a = 1;  // one\n\n// a comment line\nint b = 2;\n")
    monkeypatch.setattr(bench, "KERNEL_SRC", str(src))
    h0 = bench.kernel_src_hash()
    src.write_text("int a = 1;  // changed comment\nint b = 2;   \n")
    assert bench.kernel_src_hash() == h0
    src.write_text("int a = 1;\nint b = 3;\n")
    assert bench.kernel_src_hash() != h0


def test_recorded_traffic_is_used_only_for_the_matching_source(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("int a = 1;\n")
    monkeypatch.setattr(bench, "KERNEL_SRC", str(src))
    prof = tmp_path / "p.md"
    prof.write_text(f"kernel_source_sha256_16: {bench.kernel_src_hash()}\n"
                    "dram_bytes_per_launch_full_size: 12345\n")
    assert bench.ncu_traffic_per_launch(str(prof)) == 12345
    src.write_text("int a = 2;\n")
    assert bench.ncu_traffic_per_launch(str(prof)) is None
    assert bench.ncu_traffic_per_launch(str(tmp_path / "missing.md")) is None


def test_byte_accounting():
    shape = wl.SHAPES["mha32"]
    coeff = wl.algorithmic_bytes_decode(shape, np.full(64, 8192))
    assert coeff == 64 * 8192 * (32 * 64 + 1024) * 2 == 3221225472
    assert wl.factor_bytes(shape) == (32 * 64 * 128 + 1024 * 32 * 128) * 2 == 8912896
    assert wl.algorithmic_bytes_decode(shape, [100], "fp8_e4m3") * 2 == \
        wl.algorithmic_bytes_decode(shape, [100])
    # 4-bit pages: 32 heads x 64 codes / 2 + 32 scales x 2 + 1024 / 2 + 16 scales x 2 bytes
    assert wl.page_bytes_per_token(shape, "int4") == 1024 + 64 + 512 + 32 == 1632
    per_req = bench.bytes_per_request()
    assert abs(per_req * bench.BATCH - (coeff + wl.factor_bytes(shape))) < 1e-3


def test_reference_arm_prints_one_json_line_with_the_contract_keys():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--seq-len", "256"], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "impl", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1


def test_decode_step_flop_count():
    f = bench.decode_step_flops(np.full(64, 8192))
    assert f["pv"] == 2 * 64 * 8192 * 32 * 1024 == 34359738368
    assert f["scores"] == 2 * 64 * 8192 * 32 * 64
    assert f["upproj"] == 2 * 64 * 32 * 1024 * 128
    assert f["total"] == sum(v for k, v in f.items() if k != "total")
    assert bench.decode_step_flops([16, 16], kept_tokens=16)["pv"] == 2 * 16 * 32 * 1024


def test_bench_int4_page_preparation_matches_the_oracle_encoding():
    """The bench stores its seeded fp16 pages as 4-bit pages with torch ops; the bytes must
    be the oracle's encoding of the same coefficients."""
    import torch
    from oracle import rcp_oracle as orc
    rng = np.random.default_rng(5)
    H, rk, R = 4, 16, 128
    kp = wl.fp16(rng.standard_normal((3, H, 16, rk)))
    vp = wl.fp16(rng.standard_normal((3, 16, R)) * 3)
    kp[1, 2, 5] = 0.0                      # an all-zero group
    kb, vb = bench.int4_pages_torch(torch.from_numpy(kp), torch.from_numpy(vp))
    kc, ks, vc, vs = orc.int4_pages(kp, vp)
    ko, vo = orc.int4_pack_pages(kc, ks, vc, vs)
    assert np.array_equal(kb.numpy(), ko)
    assert np.array_equal(vb.numpy(), vo)


def test_key_and_value_bytes_per_token_split_the_page_bytes():
    """Per cached token at (32, 128, 64, 1024): fp16 4096 + 2048, E4M3 2048 + 1024, 4-bit
    (32*64/2 code bytes + 32 fp16 row scales) + (512 code bytes + 16 fp16 group scales)."""
    import workloads as wl
    s = wl.SHAPES["mha32"]
    want = {"fp16": (4096, 2048), "fp8_e4m3": (2048, 1024), "int4": (1088, 544)}
    for pages, (k, v) in want.items():
        assert wl.key_bytes_per_token(s, pages) == k
        assert wl.value_bytes_per_token(s, pages) == v
        assert wl.page_bytes_per_token(s, pages) == k + v
