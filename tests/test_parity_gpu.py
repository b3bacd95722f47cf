"""GPU parity: the CUDA path (called through the C-ABI) against the CPU oracle
on the same seeded fp16 inputs, element by element.

Shapes span several tiles and ragged tails in M, N and K; the five workload
configurations are checked in the launch configuration the bench times
(8192^3 on 4096 seeded samples plus tile-seam points, the rest in full).
"""
import numpy as np
import pytest
import torch

import oracle
from multistage_smem_pipeline_gb300 import synthetic
from tolerance import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib(gpu):
    from multistage_smem_pipeline_gb300 import binding
    return binding


def _dev(bits, gpu):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.float16)).to(gpu)


def _run(lib, a_bits, b_bits, gpu, **opts):
    a, b = _dev(a_bits, gpu), _dev(b_bits, gpu)
    d = lib.gemm_tn_f16_ex(a, b, **opts) if opts else lib.gemm_tn_f16(a, b)
    torch.cuda.synchronize()
    status, raw = lib.get_device_error()
    assert status == 0, f"device error word {raw:#x}"
    return d.cpu().numpy().view(np.uint16)


def _check(got, a_bits, b_bits, ref=None):
    K = a_bits.shape[1]
    if ref is None:
        ref = oracle.gemm_tn(a_bits, b_bits)
    st = compare(got, ref, K, a_bits, b_bits)
    assert st["bad"] == 0, st
    return st


# ----------------------------------------------------------------- shapes and tails
SHAPES = [
    (128, 256, 64),      # exactly one tile, one k-block
    (1, 8, 8),           # smallest legal shape: almost all of the box is out of range
    (7, 24, 40),         # sub-tile everything, K tail inside one k-block
    (129, 264, 72),      # one past a tile edge in M, N and K
    (300, 520, 200),     # several tiles, ragged in all three
    (256, 256, 256),     # the 256^3 workload's shape
    (384, 96, 1000),     # K tail of 40 after 15 full k-blocks
    (64, 4096, 128),     # skinny M, many n tiles
]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_shapes_with_tails(lib, gpu, M, N, K):
    a = synthetic.uniform_pm1(M * 7 + 1, (M, K))
    b = synthetic.uniform_pm1(N * 11 + 2, (N, K))
    _check(_run(lib, a, b, gpu), a, b)


SQUARE, PAIR = 1, 3


@pytest.mark.parametrize("path", [SQUARE, PAIR])
@pytest.mark.parametrize("bn", list(range(32, 257, 32)))
def test_every_tile_width(lib, gpu, bn, path):
    M, N, K = 272, 8 * 83, 328          # ragged m-blocks, ragged n, 6 k-blocks (tail 8)
    a = synthetic.uniform_pm1(bn, (M, K))
    b = synthetic.uniform_pm1(bn + 1, (N, K))
    _check(_run(lib, a, b, gpu, bn=bn, path=path), a, b)


@pytest.mark.parametrize("path,bn", [(SQUARE, 256), (SQUARE, 128), (SQUARE, 64),
                                     (PAIR, 256), (PAIR, 128), (PAIR, 64)])
def test_every_ring_depth_and_wrap(lib, gpu, path, bn):
    # K = BK * (kstage +- 1) around every depth: the ring wraps mid-tile and
    # the phase bits flip at different k-blocks; one CTA (pair) walks all
    # tiles so both TMEM accumulators are reused many times.
    fixed = dict(bn=bn, path=path, katoms=1, epi_warps=4)   # the ring depth alone varies
    deepest = lib.query_config(256, 512, 4096, **fixed)["kstage"]
    a_full = synthetic.uniform_pm1(5, (512, 64 * (deepest + 2)))
    b_full = synthetic.uniform_pm1(6, (512, 64 * (deepest + 2)))
    for ks in range(2, deepest + 1):
        for kb in (ks - 1, ks, ks + 1):
            K = 64 * kb
            a = np.ascontiguousarray(a_full[:, :K])
            b = np.ascontiguousarray(b_full[:, :K])
            got = _run(lib, a, b, gpu, kstage=ks, max_ctas=2 if path == PAIR else 1, **fixed)
            _check(got, a, b)


@pytest.mark.parametrize("path,bn", [(SQUARE, 256), (SQUARE, 96), (PAIR, 256), (PAIR, 128)])
def test_two_k_slices_per_stage(lib, gpu, path, bn):
    # katoms = 2: each ring stage holds two 64-wide K slices; K values put the
    # tail in the first or the second slice, or leave the second slice entirely
    # past K (its loads read zeros), and the ring wraps at every depth
    fixed = dict(bn=bn, path=path, katoms=2, epi_warps=8)
    deepest = lib.query_config(384, 520, 4096, **fixed)["kstage"]
    for ks in range(2, deepest + 1):
        for K in (64, 120, 128, 136, 64 * 2 * ks + 64, 64 * 2 * (ks + 1) + 8):
            a = synthetic.uniform_pm1(K + ks, (384, K))
            b = synthetic.uniform_pm1(K + ks + 1, (520, K))
            got = _run(lib, a, b, gpu, kstage=ks, max_ctas=2 if path == PAIR else 1, **fixed)
            _check(got, a, b)


@pytest.mark.parametrize("epi", [4, 8])
@pytest.mark.parametrize("path,bn", [(SQUARE, 32), (SQUARE, 96), (SQUARE, 256), (PAIR, 64),
                                     (PAIR, 160), (PAIR, 256)])
def test_both_epilogue_widths(lib, gpu, epi, path, bn):
    # 4 epilogue warps (one per TMEM lane quadrant) or 8 (two per quadrant,
    # alternate 32-column chunks); N tails leave odd chunk counts per warp
    for M, N, K in [(300, 8 * 41, 192), (129, 264, 64), (520, 1000, 320)]:
        a = synthetic.uniform_pm1(M + epi, (M, K))
        b = synthetic.uniform_pm1(N + epi, (N, K))
        _check(_run(lib, a, b, gpu, path=path, bn=bn, epi_warps=epi, max_ctas=4), a, b)


def test_two_k_slices_ternary_is_bit_exact(lib, gpu):
    a, b, spec = synthetic.workload("c2")
    for path in (SQUARE, PAIR):
        got = _run(lib, a, b, gpu, katoms=2, path=path)
        assert np.array_equal(got, oracle.gemm_tn(a, b))


@pytest.mark.parametrize("path", [SQUARE, PAIR])
@pytest.mark.parametrize("ctas,group_m", [(2, 1), (6, 2), (10, 16), (0, 3)])
def test_persistent_schedules(lib, gpu, ctas, group_m, path):
    M, N, K = 128 * 5 + 17, 256 * 3 + 40, 192
    a = synthetic.uniform_pm1(ctas + 40, (M, K))
    b = synthetic.uniform_pm1(group_m + 50, (N, K))
    _check(_run(lib, a, b, gpu, max_ctas=ctas, group_m=group_m, bn=128, path=path), a, b)


@pytest.mark.parametrize("M", [129, 200, 256, 300, 384, 385, 640])
def test_pair_row_tails(lib, gpu, M):
    # M not a multiple of 256: the odd CTA of the last pair has few or no
    # valid rows but still feeds its zero-filled half of the MMA
    N, K = 264, 136
    a = synthetic.uniform_pm1(M, (M, K))
    b = synthetic.uniform_pm1(M + 3, (N, K))
    _check(_run(lib, a, b, gpu, path=PAIR), a, b)


@pytest.mark.parametrize("path", [SQUARE, PAIR])
def test_one_m_block_rotated_k_is_bit_exact_on_ternary(lib, gpu, path):
    # M <= 128 rotates each tile's k loop; integer partial sums are exact in
    # any order, so the result must still match bit for bit
    a = synthetic.ternary(21, (128, 1024))
    b = synthetic.ternary(22, (1000, 1024))
    got = _run(lib, a, b, gpu, path=path)
    ai = a.view(np.float16).astype(np.int64)
    bi = b.view(np.float16).astype(np.int64)
    assert np.array_equal(got, (ai @ bi.T).astype(np.float16).view(np.uint16))
    assert np.array_equal(got, oracle.gemm_tn(a, b))


@pytest.mark.parametrize("bn", [64, 192, 256])
def test_pair_path_with_one_row_block(lib, gpu, bn):
    # M <= 128 on the pair path: the odd CTA's A rows are all out of range
    for M in (1, 77, 128):
        a = synthetic.gaussian(M + 5, (M, 640))
        b = synthetic.gaussian(M + 6, (1400, 640), 0.02)
        _check(_run(lib, a, b, gpu, path=PAIR, bn=bn), a, b)


def test_skinny_path_small(lib, gpu):
    for M in (1, 16, 100, 128):
        a = synthetic.gaussian(M, (M, 512))
        b = synthetic.gaussian(M + 1, (1000, 512), 0.02)
        _check(_run(lib, a, b, gpu, path=lib.PATH_SKINNY), a, b)


# ----------------------------------------------------------------- degenerate sizes
def test_zero_k_writes_zeros(lib, gpu):
    a = torch.empty((33, 0), dtype=torch.float16, device=gpu)
    b = torch.empty((40, 0), dtype=torch.float16, device=gpu)
    d = torch.full((33, 40), 7.0, dtype=torch.float16, device=gpu)
    lib.gemm_tn_f16(a, b, out=d)
    torch.cuda.synchronize()
    assert torch.count_nonzero(d).item() == 0


def test_empty_m_or_n_is_noop(lib, gpu):
    a = torch.ones((0, 64), dtype=torch.float16, device=gpu)
    b = torch.ones((16, 64), dtype=torch.float16, device=gpu)
    assert lib.gemm_tn_f16(a, b).shape == (0, 16)
    b0 = torch.ones((0, 64), dtype=torch.float16, device=gpu)
    assert lib.gemm_tn_f16(b, b0).shape == (16, 0)


def test_misaligned_tensor_is_rejected(lib, gpu):
    base = torch.zeros(64 * 64 + 1, dtype=torch.float16, device=gpu)
    a = base[1:].view(64, 64)                 # 2-byte offset
    b = torch.zeros((64, 64), dtype=torch.float16, device=gpu)
    with pytest.raises(lib.GemmError) as e:
        lib.gemm_tn_f16(a, b)
    assert e.value.status == lib.GEMM_ERR_MISALIGNED


def test_large_values_and_overflow(lib, gpu):
    # sums beyond 65504 become inf on both sides; exact small-int sums stay exact
    a = np.full((128, 64), np.float16(64.0)).view(np.uint16)
    b = np.full((256, 64), np.float16(32.0)).view(np.uint16)     # 64 * 2048 = 131072 -> inf
    got = _run(lib, a, b, gpu)
    assert np.all(got == 0x7C00)


# ----------------------------------------------------------------- the five workloads
def _workload_check(lib, gpu, tag, sampled=False):
    a, b, spec = synthetic.workload(tag)
    got = _run(lib, a, b, gpu)
    if sampled:
        rows, cols = synthetic.sample_coords(synthetic.seeds(tag)[2], spec["M"], spec["N"])
        ref = oracle.gemm_tn_sampled(a, b, rows, cols)
        st = compare(got[rows, cols], ref, spec["K"], a, b)
        assert st["bad"] == 0, st
        # properties that hold at any size: finite everywhere, |D| bounded by K*max|a||b|
        g = got.view(np.float16)
        assert np.isfinite(g).all()
        return st
    return _check(got, a, b)


def test_workload_256(lib, gpu):
    _workload_check(lib, gpu, "c1")


def test_workload_1024_ternary_is_bit_exact(lib, gpu):
    a, b, spec = synthetic.workload("c2")
    got = _run(lib, a, b, gpu)
    ref = oracle.gemm_tn(a, b)
    assert np.array_equal(got, ref)
    ai = a.view(np.float16).astype(np.int64)
    bi = b.view(np.float16).astype(np.int64)
    assert np.array_equal(ref, (ai @ bi.T).astype(np.float16).view(np.uint16))


def test_workload_4096(lib, gpu):
    st = _workload_check(lib, gpu, "c3")
    assert st["exact_frac"] > 0.95


def test_workload_8192_sampled(lib, gpu):
    st = _workload_check(lib, gpu, "c4", sampled=True)
    assert st["n"] >= 4096


def test_workload_skinny(lib, gpu):
    st = _workload_check(lib, gpu, "c5")
    assert st["exact_frac"] > 0.95


def test_workload_tall(lib, gpu):
    # the shape the multistage page times (section 11): 81920 x 256 x 256
    st = _workload_check(lib, gpu, "c6")
    assert st["exact_frac"] > 0.95


def test_host_buffers_end_to_end(lib, gpu):
    a, b, spec = synthetic.workload("c1")
    ah = torch.from_numpy(a.view(np.float16)).pin_memory()
    bh = torch.from_numpy(b.view(np.float16)).pin_memory()
    d = lib.gemm_tn_f16_from_host(ah, bh)
    _check(d.numpy().view(np.uint16), a, b)


def test_side_stream(lib, gpu):
    a = synthetic.uniform_pm1(77, (300, 256))
    b = synthetic.uniform_pm1(78, (264, 256))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        da, db = _dev(a, gpu), _dev(b, gpu)
        d = lib.gemm_tn_f16(da, db, stream=s)
    s.synchronize()
    _check(d.cpu().numpy().view(np.uint16), a, b)
