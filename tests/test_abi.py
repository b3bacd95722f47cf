"""C-ABI checks that need no GPU: the library loads, exports every function
include/gemm_tn_f16.h declares, and rejects bad arguments on the host before
touching the device."""
import ctypes
import os
import re

import pytest

from conftest import cuda_available

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemm_tn_f16.h")


@pytest.fixture(scope="module")
def binding():
    from multistage_smem_pipeline_gb300 import build
    build.build()
    from multistage_smem_pipeline_gb300 import binding as b
    return b


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(gemm_[a-z0-9_]+)\s*\(", text,
                       flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for want in ("gemm_tn_f16", "gemm_tn_f16_ex", "gemm_f16_scaled", "gemm_f16_padded",
                 "gemm_padded_workspace_bytes", "gemm_get_device_error",
                 "gemm_minimum_stages",
                 "gemm_query_config", "gemm_probe_latencies", "gemm_status_string"):
        assert want in names


def test_library_exports_every_declared_symbol(binding):
    lib = ctypes.CDLL(binding.library_path())
    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} declared in the header but not exported"
    assert set(binding.EXPORTED) <= set(_declared_functions())


def test_library_is_in_tree_and_built_for_sm103a(binding):
    path = binding.library_path()
    assert path.startswith(os.path.join(ROOT, "multistage_smem_pipeline_gb300"))
    from multistage_smem_pipeline_gb300 import build
    assert "arch=compute_103a,code=sm_103a" in build.ARCH


def test_minimum_stages_matches_page_examples(binding):
    # same golden rows the oracle is pinned to
    with open(os.path.join(ROOT, "tests", "golden", "minimum_stages.txt")) as f:
        rows = [tuple(map(int, l.split())) for l in f if l.strip() and not l.startswith("#")]
    for copy, compute, want in rows:
        assert binding.minimum_stages(copy, compute) == want
    assert binding.minimum_stages(241, 120) == 4
    assert binding.minimum_stages(0, 5) == -1 and binding.minimum_stages(5, -1) == -1
    assert binding.minimum_stages(2**62, 1) == 2**62 + 1        # no overflow


def _call(binding, D, A, B, M, N, K, opts=None):
    if opts is None:
        return binding.LIB.gemm_tn_f16(D, A, B, M, N, K, None)
    return binding.LIB.gemm_tn_f16_ex(D, A, B, M, N, K, ctypes.byref(opts), None)


# fake, never dereferenced device addresses: validation rejects them first
P0, P1, P2 = 0x10000000, 0x20000000, 0x30000000


def test_rejects_bad_sizes(binding):
    for M, N, K in [(-1, 8, 8), (8, -8, 8), (8, 8, -8), (2**31, 8, 8), (8, 8, 2**40)]:
        assert _call(binding, P0, P1, P2, M, N, K) == binding.GEMM_ERR_INVALID_VALUE


def test_rejects_misalignment(binding):
    assert _call(binding, P0 + 2, P1, P2, 16, 16, 16) == binding.GEMM_ERR_MISALIGNED
    assert _call(binding, P0, P1 + 8, P2, 16, 16, 16) == binding.GEMM_ERR_MISALIGNED
    assert _call(binding, P0, P1, P2, 16, 12, 16) == binding.GEMM_ERR_MISALIGNED   # N % 8
    assert _call(binding, P0, P1, P2, 16, 16, 20) == binding.GEMM_ERR_MISALIGNED   # K % 8


def test_rejects_null_and_overlap(binding):
    assert _call(binding, 0, P1, P2, 16, 16, 16) == binding.GEMM_ERR_INVALID_VALUE
    assert _call(binding, P0, 0, P2, 16, 16, 16) == binding.GEMM_ERR_INVALID_VALUE
    # D = [P1, P1 + 512) overlaps A = [P1 + 256, ...)
    assert _call(binding, P1, P1 + 256, P2, 16, 16, 16) == binding.GEMM_ERR_INVALID_VALUE


def test_empty_output_is_a_noop_without_device(binding):
    assert _call(binding, 0, 0, 0, 0, 16, 16) == binding.GEMM_OK
    assert _call(binding, 0, 0, 0, 16, 0, 16) == binding.GEMM_OK


def test_rejects_bad_options(binding):
    for kw in [dict(bn=48), dict(bn=512), dict(kstage=1), dict(kstage=17), dict(path=4),
               dict(inject=3), dict(max_ctas=-1), dict(path=binding.PATH_SKINNY),
               dict(katoms=3), dict(katoms=-1), dict(epi_warps=6), dict(epi_warps=16),
               dict(acc_f16=2), dict(b_resident=3), dict(b_resident=-1),
               dict(b_resident=2, path=binding.PATH_PAIR),
               dict(b_resident=2, bn=32, group_m=4), dict(wide=3), dict(wide=-1),
               dict(wide=2, path=binding.PATH_SQUARE), dict(check=2), dict(check=-1),
               dict(split_k=3), dict(small_m=3), dict(multicast=3), dict(multicast=-1),
               dict(multicast=2, split_k=1)]:
        o = binding._options(**kw)
        M = 256 if kw.get("path") == binding.PATH_SKINNY else 64
        assert _call(binding, P0, P1, P2, M, 64, 64, o) == binding.GEMM_ERR_INVALID_VALUE, kw


@pytest.mark.skipif(cuda_available(), reason="checks the no-device error path")
def test_valid_call_without_a_device_reports_cuda_error(binding):
    assert _call(binding, P0, P1, P2, 64, 64, 64) in (binding.GEMM_ERR_CUDA,
                                                      binding.GEMM_ERR_UNSUPPORTED_DEVICE)


def test_query_config_plans(binding):
    c = binding.query_config(8192, 8192, 8192)
    assert c["path"] == binding.PATH_PAIR and c["bm"] == 256 and c["bk"] == 64 * c["katoms"]
    assert c["katoms"] in (1, 2)
    assert c["ctas"] % 2 == 0
    assert c["bn"] % 32 == 0 and 32 <= c["bn"] <= 256
    assert c["kstage"] >= 2 and c["smem_bytes"] <= 232448
    assert c["tmem_cols"] >= 2 * c["bn"] and c["tmem_cols"] <= 512
    assert c["tmem_cols"] & (c["tmem_cols"] - 1) == 0
    s = binding.query_config(128, 14336, 4096)
    assert s["path"] == binding.PATH_SKINNY and s["tiles"] <= s["ctas"] * 2
    # every explicit (path, bn, katoms, kstage) that is accepted fits the shared-memory budget
    for path in (binding.PATH_SQUARE, binding.PATH_PAIR):
        for katoms in (1, 2):
            for bn in range(32, 257, 32):
                q = dict(path=path, bn=bn, katoms=katoms)
                deepest = binding.query_config(1024, 1024, 1024, **q)["kstage"]
                for ks in range(2, deepest + 1):
                    cc = binding.query_config(1024, 1024, 1024, kstage=ks, **q)
                    assert cc["smem_bytes"] <= 232448 and cc["kstage"] == ks
                    assert cc["path"] == path and cc["katoms"] == katoms
                    assert cc["bm"] == (256 if path == binding.PATH_PAIR else 128)
                with pytest.raises(binding.GemmError):
                    binding.query_config(1024, 1024, 1024, kstage=deepest + 1, **q)
    # a pair stage holds half of B, so the pair ring is deeper at the same width
    assert binding.query_config(4096, 4096, 4096, path=binding.PATH_PAIR, bn=256, katoms=1,
                                wide=1)["kstage"] > \
        binding.query_config(4096, 4096, 4096, path=binding.PATH_SQUARE, bn=256,
                             katoms=1)["kstage"]
    # a wide pair stage holds A once for two tiles' B halves: the deepest ring at bn 256
    wide = binding.query_config(8192, 8192, 8192, path=binding.PATH_PAIR, bn=256, wide=2)
    assert wide["wide"] == 1 and wide["katoms"] == 1 and wide["kstage"] == 4
    # two K slices per stage only where the ring keeps at least 3 stages
    for shape in [(8192, 8192, 8192), (128, 14336, 4096), (256, 256, 256)]:
        cc = binding.query_config(*shape)
        assert cc["katoms"] == 1 or cc["kstage"] >= 3


def _scaled(binding, D, C, A, B, M, N, K, alpha=1.0, beta=0.0, layout=1, opts=None):
    o = binding._options(**(opts or {}))
    return binding.LIB.gemm_f16_scaled(D, C, A, B, M, N, K, alpha, beta, layout,
                                       ctypes.byref(o), None)


def test_scaled_entry_rejects_bad_arguments(binding):
    E = binding.GEMM_ERR_INVALID_VALUE
    assert _scaled(binding, P0, P1, P1 + 4096, P2, 16, 16, 16, layout=2) == E
    assert _scaled(binding, P0, P1, P1 + 4096, P2, 16, 16, 16, alpha=float("nan")) == E
    assert _scaled(binding, P0, P1, P1 + 4096, P2, 16, 16, 16, beta=float("inf")) == E
    # beta != 0 needs C; C partially overlapping D is refused; C == D is allowed (in place)
    assert _scaled(binding, P0, 0, P1, P2, 16, 16, 16, beta=0.5) == E
    assert _scaled(binding, P0, P0 + 256, P1, P2, 16, 16, 16, beta=0.5) == E
    assert _scaled(binding, P0, P0 + 8, P1, P2, 16, 16, 16, beta=0.5) == \
        binding.GEMM_ERR_MISALIGNED
    # a K x N B is loaded in 64-column boxes: the tile width must be whole boxes
    assert _scaled(binding, P0, 0, P1, P2, 256, 256, 256, opts=dict(bn=96, path=1)) == E
    assert _scaled(binding, P0, 0, P1, P2, 256, 256, 256, opts=dict(bn=64, path=3)) == E
    assert _scaled(binding, 0, 0, 0, 0, 0, 16, 16, beta=0.5) == binding.GEMM_OK


def test_status_strings(binding):
    assert binding.status_string(0) == "GEMM_OK"
    assert binding.status_string(5) == "GEMM_ERR_TIMEOUT"
    assert binding.status_string(7) == "GEMM_ERR_INVARIANT"
    assert binding.status_string(99) == "GEMM_ERR_UNKNOWN"


def _ws_bytes(binding, D, C, A, B, M, N, K, beta=0.0, layout=0):
    n = ctypes.c_uint64(12345)
    rc = binding.LIB.gemm_padded_workspace_bytes(D, C, A, B, M, N, K, beta, layout, ctypes.byref(n))
    return rc, n.value


def test_padded_workspace_sizes(binding):
    # nothing misaligned: no workspace
    assert _ws_bytes(binding, P0, P1, P1 + 4096, P2, 10, 16, 16, beta=1.0) == (0, 0)
    # K = 15: A (10 x 16) and an N x K B (16 x 16) repacked, 256-byte regions
    assert _ws_bytes(binding, P0, 0, P1, P2, 10, 16, 15) == (0, 512 + 512)
    # N = 13 with a K x N B: B (16 x 16) repacked; A as given; D is stored
    # directly by the kernel (C not read), so it needs no region
    assert _ws_bytes(binding, P0, 0, P1, P2, 10, 13, 16, layout=1) == (0, 512)
    # ... while an N x K B (13 x 16) is aligned as it is
    assert _ws_bytes(binding, P0, 0, P1, P2, 10, 13, 16, layout=0) == (0, 0)
    # with C read, D (10 x 16 padded) holds C during the GEMM
    assert _ws_bytes(binding, P0, P1 + 8192, P2, P2 + 65536, 10, 13, 16, beta=1.0) == (0, 512)
    assert _ws_bytes(binding, P0 + 2, P1 + 8192, P2, P2 + 65536, 10, 16, 16, beta=1.0) == (0, 512)
    # a base address alone forces a repack of that operand it reads
    assert _ws_bytes(binding, P0 + 2, 0, P1, P2, 10, 16, 16) == (0, 0)
    assert _ws_bytes(binding, P0, 0, P1 + 6, P2, 10, 16, 16) == (0, 512)
    assert _ws_bytes(binding, P0, 0, P1, P2 + 4, 300, 16, 16) == (0, 512)
    # a misaligned C with an aligned D is copied into D: no region of its own
    assert _ws_bytes(binding, P0, P1 + 2, P2, P2 + 65536, 10, 16, 16, beta=0.5) == (0, 0)
    # nothing reaches the GEMM kernel: no workspace
    assert _ws_bytes(binding, P0 + 2, 0, P1 + 2, P2 + 2, 10, 13, 0) == (0, 0)
    assert _ws_bytes(binding, P0 + 2, 0, P1 + 2, P2 + 2, 0, 13, 7) == (0, 0)
    # large sizes: 8191^3 repacks A and B, each 8191 x 8192 fp16 (D is stored
    # directly); with C read, D's padded copy adds a third region
    region = (8191 * 8192 * 2 + 255) // 256 * 256
    assert _ws_bytes(binding, P0, 0, P1, P2, 8191, 8191, 8191) == (0, 2 * region)
    assert _ws_bytes(binding, P0, 1 << 40, P1, P2, 8191, 8191, 8191, beta=0.5) == (0, 3 * region)
    E = binding.GEMM_ERR_INVALID_VALUE
    assert _ws_bytes(binding, P0, 0, P1, P2, -1, 16, 16)[0] == E
    # K or N that rounds up past the kernel's int32 extents, and a workspace
    # whose size would overflow, are refused
    assert _ws_bytes(binding, P0, 0, P1, P2, 1, 16, 2**31 - 1)[0] == E
    assert _ws_bytes(binding, P0, 0, P1, P2, 1, 2**31 - 1, 16)[0] == E
    assert _ws_bytes(binding, P0 + 2, 0, P1 + 2, P2 + 2, 2**31 - 1, 2**31 - 9, 2**31 - 9)[0] == E
    assert _ws_bytes(binding, P0, 0, P1, P2, 16, 16, 16, layout=2)[0] == E
    assert binding.LIB.gemm_padded_workspace_bytes(P0, 0, P1, P2, 1, 1, 1, 0.0, 0, None) == E


def _padded(binding, D, C, A, B, M, N, K, ws=0, ws_bytes=0, alpha=1.0, beta=0.0, layout=0):
    o = binding._options()
    return binding.LIB.gemm_f16_padded(D, C, A, B, M, N, K, alpha, beta, layout, ws, ws_bytes,
                                       ctypes.byref(o), None)


def test_padded_entry_rejects_bad_arguments(binding):
    E, MIS = binding.GEMM_ERR_INVALID_VALUE, binding.GEMM_ERR_MISALIGNED
    W = 0x40000000
    # odd (not fp16-aligned) pointers
    assert _padded(binding, P0 + 1, 0, P1, P2, 16, 16, 16) == MIS
    assert _padded(binding, P0, 0, P1 + 3, P2, 16, 16, 16) == MIS
    assert _padded(binding, P0, P1 + 8192 + 1, P2, P2 + 65536, 16, 16, 16, beta=1.0) == MIS
    # workspace missing, too small, misaligned, or overlapping an operand
    need = _ws_bytes(binding, P0, 0, P1, P2, 16, 13, 15)[1]
    assert need > 0
    assert _padded(binding, P0, 0, P1, P2, 16, 13, 15) == E
    assert _padded(binding, P0, 0, P1, P2, 16, 13, 15, ws=W, ws_bytes=need - 1) == E
    assert _padded(binding, P0, 0, P1, P2, 16, 13, 15, ws=W + 8, ws_bytes=need) == MIS
    assert _padded(binding, P0, 0, P1, P2, 16, 13, 15, ws=P0 - 64, ws_bytes=need) == E
    assert _padded(binding, P0, 0, P1, P2, 16, 13, 15, ws=P1 + 64, ws_bytes=need) == E
    # the checks of the scaled form
    assert _padded(binding, P0, 0, P1, P2, 16, 13, 15, ws=W, ws_bytes=need, layout=2) == E
    assert _padded(binding, P0, 0, P1, P2, 16, 13, 15, ws=W, ws_bytes=need,
                   alpha=float("nan")) == E
    assert _padded(binding, P0, 0, P1, P2, 16, 13, 15, ws=W, ws_bytes=need, beta=1.0) == E
    assert _padded(binding, P0, P0 + 2, P1, P2, 16, 13, 15, ws=W, ws_bytes=need, beta=1.0) == E
    assert _padded(binding, P0, 0, P0 + 64, P2, 16, 13, 15, ws=W, ws_bytes=need) == E
    assert _padded(binding, P0, 0, P1, P2, -3, 13, 15) == E
    assert _padded(binding, P0, 0, P1, P2, 16, 16, 2**31 - 1) == E
    # empty outputs are no-ops without a workspace or a device
    assert _padded(binding, 0, 0, 0, 0, 0, 13, 15) == binding.GEMM_OK
    assert _padded(binding, P0 + 2, 0, 0, 0, 7, 0, 15) == binding.GEMM_OK


@pytest.mark.skipif(cuda_available(), reason="checks the no-device error path")
def test_padded_call_without_a_device_reports_cuda_error(binding):
    need = _ws_bytes(binding, P0, 0, P1, P2, 16, 13, 15)[1]
    assert _padded(binding, P0, 0, P1, P2, 16, 13, 15, ws=0x40000000, ws_bytes=need) in \
        (binding.GEMM_ERR_CUDA, binding.GEMM_ERR_UNSUPPORTED_DEVICE)


def test_resident_b_plans(binding):
    # a tall shape whose resident B leaves A's ring deeper than streaming would:
    # each CTA holds its n-block of B and streams only A
    cfg = binding.query_config(81920, 1024, 128)
    assert cfg["b_resident"] == 1 and cfg["path"] == binding.PATH_SQUARE
    assert cfg["smem_bytes"] <= 232448
    # the page's 81920 x 256 x 256: the same depth of A either way, one n-block
    # (streamed B is an L2 hit for every tile), so B streams unless asked for
    assert binding.query_config(81920, 256, 256)["b_resident"] == 0
    assert binding.query_config(81920, 256, 256, b_resident=2)["b_resident"] == 1
    # off on request, and never for many n-blocks, the pair path or a K x N B
    assert binding.query_config(81920, 256, 256, b_resident=1)["b_resident"] == 0
    assert binding.query_config(8192, 8192, 8192)["b_resident"] == 0
    assert binding.query_config(81920, 4096, 256)["b_resident"] == 0
    assert binding.query_config(81920, 256, 256, b_layout=1)["b_resident"] == 0
    # too few tiles per CTA to pay for loading B up front
    assert binding.query_config(1024, 256, 256)["b_resident"] == 0
    # a few n-blocks: tiles n-fastest over a grid that is a multiple of num_n,
    # so every CTA meets a single n-block
    for shape, opts in [((81920, 512, 256), {}), ((81920, 256, 256), dict(bn=128)),
                        ((7680, 384, 64), dict(bn=128, b_resident=2)),
                        ((300, 256, 256), dict(path=1, b_resident=2))]:
        cfg = binding.query_config(*shape, **opts)
        num_n = -(-shape[1] // cfg["bn"])
        assert cfg["b_resident"] == 1 and cfg["ctas"] % num_n == 0, (shape, cfg)
        assert num_n == 1 or cfg["group_m"] == 1
    # a rasterisation group that would mix n-blocks on one CTA excludes it
    assert binding.query_config(81920, 256, 256, bn=128, group_m=4)["b_resident"] == 0
    # a B too large for shared memory is refused when forced
    with pytest.raises(binding.GemmError):
        binding.query_config(4096, 256, 4096, path=1, b_resident=2)
