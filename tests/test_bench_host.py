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
