"""Host-side pieces of bench.py that decide what its JSON line reports (no GPU).

The per-launch DRAM traffic recorded from an ncu capture is reported only
while the kernel sources still match the capture; the match ignores comments
and layout, so it must strip exactly those and keep every token of code --
including string literals, where PTX text may contain "//"."""
import importlib.util
import json
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_host_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_comments_and_layout_do_not_count(bench):
    a = "int x = 1;  // the count\n/* block\n comment */ int y = x + 2;\n"
    b = "int x = 1;\nint y = x + 2;  // other words\n"
    assert bench.code_tokens(a) == bench.code_tokens(b)


def test_code_and_literals_count(bench):
    base = 'asm volatile("mov.u32 %0, 1;" : "=r"(v));'
    assert bench.code_tokens(base) != bench.code_tokens(base.replace("1;", "2;"))
    # "//" and "/*" inside a literal are code, not the start of a comment
    lit = 'const char* s = "a // b /* c */"; char q = \'"\'; int z = 3;'
    assert bench.code_tokens(lit) == lit
    assert bench.code_tokens('x = "\\" // still inside";') == 'x = "\\" // still inside";'


def test_recorded_traffic_follows_the_sources(bench):
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        rec = json.load(f)
    current = bench.source_hash()
    for tag, entry in rec.items():
        if not isinstance(entry, dict):
            continue
        got = bench.recorded_traffic(tag)
        if entry.get("source_hash") == current:
            assert got == entry["dram_bytes_per_launch"]
        else:
            assert got is None


PEAKS = {"hbm_gbs": 6689.1, "bf16_tflops": 1936.4, "bf16_tflops_sustained": 1742.0}


def test_peak_follows_the_timed_region_length(bench):
    flops, alg = 2.0 * 8192 ** 3, 2.0 * 3 * 8192 ** 2
    short = bench.roofline_of(flops, alg, 0.5856, PEAKS, "measured", 0.0117)
    assert short["bound"] == "tensor" and short["peak"] == PEAKS["bf16_tflops"]
    assert short["frac"] == pytest.approx(flops / 0.5856e-3 / 1e12 / PEAKS["bf16_tflops"])
    assert "under 1 s" in short["peak_source"]
    long = bench.roofline_of(flops, alg, 0.658, PEAKS, "measured", 2.0)
    assert long["peak"] == PEAKS["bf16_tflops_sustained"]
    assert long["frac"] == pytest.approx(long["achieved"] / PEAKS["bf16_tflops_sustained"])
    assert long["frac_of_burst_peak"] == pytest.approx(long["achieved"] / PEAKS["bf16_tflops"])


def test_skinny_shape_is_hbm_bound(bench):
    M, N, K = 128, 14336, 4096
    flops, alg = 2.0 * M * N * K, 2.0 * (M * K + N * K + M * N)
    r = bench.roofline_of(flops, alg, 0.02448, PEAKS, "measured", 0.01)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(alg / 0.02448e-3 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / PEAKS["hbm_gbs"])


def test_tensor_nominal_fraction(bench):
    n = bench.tensor_nominal(1877.6, 152, 2070.0, 1500.0)
    assert n["max_clock"]["peak_tflops"] == pytest.approx(152 * 8192 * 2.07e9 / 1e12)
    assert n["max_clock"]["frac"] == pytest.approx(1877.6 / (152 * 8192 * 2.07e9 / 1e12))
    assert n["sampled_clock"]["peak_tflops"] == pytest.approx(152 * 8192 * 1.5e9 / 1e12)
    assert "sampled_clock" not in bench.tensor_nominal(1.0, 152, 2070.0, None)


def test_parity_stats_counts_ulps_across_zero(bench):
    import numpy as np
    ref = np.array([0x3C00, 0x0000, 0x8001, 0x3C00], dtype=np.uint16)   # 1, +0, -tiny, 1
    got = np.array([0x3C00, 0x8000, 0x0001, 0x3C01], dtype=np.uint16)   # 1, -0, +tiny, 1+ulp
    st = bench.parity_stats(got, ref, K=1, amax=1.0, bmax=1.0)
    assert st["max_ulps"] == 2 and not st["bit_exact"]
    assert st["exact_frac"] == 0.25 and st["out_of_bound"] == 0
    far = np.array([0x4000, 0x0000, 0x8001, 0x3C00], dtype=np.uint16)  # 2 where 1 is expected
    assert bench.parity_stats(far, ref, K=1, amax=1e-3, bmax=1e-3)["out_of_bound"] == 1
    assert bench.parity_stats(ref, ref, K=1, amax=1.0, bmax=1.0)["bit_exact"]


def test_clock_region_picks_samples_in_the_window(bench):
    s = bench.ClockSampler("00000000:00:00.0")
    s.max_mhz = 2070.0
    s.samples = [(0.00, 2070.0, 300.0, 0), (0.01, 1800.0, 900.0, 0x4),
                 (0.02, 1600.0, 1300.0, 0x4), (0.05, 2000.0, 200.0, 0)]
    r = s.region(0.005, 0.025)
    assert r["samples"] == 2 and r["sm_mhz"] == 1700.0 and r["reasons"] == ["sw_power_cap"]
    assert r["power_w_max"] == 1300.0
    near = s.region(0.041, 0.042)        # shorter than the period: the nearest sample
    assert near["samples"] == 1 and near["sm_mhz"] == 2000.0
