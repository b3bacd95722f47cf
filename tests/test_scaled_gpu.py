"""GPU parity of the scaled form D = alpha * A op(B) + beta * C against the
oracle, with B K x N (the layout of "CUDA 算子笔记 2", GEMM section) or N x K,
on both kernel paths, through the C-ABI entry gemm_f16_scaled."""
import numpy as np
import pytest
import torch

import oracle
from multistage_smem_pipeline_gb300 import synthetic
from tolerance import compare_scaled

pytestmark = pytest.mark.gpu
SQUARE, PAIR = 1, 3


@pytest.fixture(scope="module")
def lib(gpu):
    from multistage_smem_pipeline_gb300 import binding
    return binding


def _t(bits, gpu):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.float16)).to(gpu)


def _operands(M, N, K, kn, seed):
    a = synthetic.uniform_pm1(seed, (M, K))
    b = synthetic.uniform_pm1(seed + 1, (K, N) if kn else (N, K))
    c = synthetic.uniform_pm1(seed + 2, (M, N))
    return a, b, c


def _run(lib, gpu, a, b, c, alpha, beta, kn, in_place=False, **opts):
    ta, tb = _t(a, gpu), _t(b, gpu)
    tc = _t(c, gpu) if c is not None else None
    out = tc if in_place else None
    d = lib.gemm_f16_scaled(ta, tb, tc, alpha, beta, "kn" if kn else "nk", out=out, **opts)
    torch.cuda.synchronize()
    status, raw = lib.get_device_error()
    assert status == 0, f"device error word {raw:#x}"
    return d.cpu().numpy().view(np.uint16)


def _check(got, a, b, c, alpha, beta, kn):
    ref = oracle.gemm_scaled(a, b, c, alpha, beta, kn)
    st = compare_scaled(got, ref, a.shape[1], a, b, c, alpha, beta)
    assert st["bad"] == 0, st
    return st


@pytest.mark.parametrize("kn", [True, False])
@pytest.mark.parametrize("path,bn", [(SQUARE, 64), (SQUARE, 128), (SQUARE, 256), (PAIR, 128),
                                     (PAIR, 256)])
def test_scaled_shapes(lib, gpu, kn, path, bn):
    for (M, N, K), (alpha, beta) in [((300, 520, 200), (1.5, -0.5)), ((129, 264, 72), (-1.0, 2.0)),
                                      ((640, 384, 1088), (0.25, 0.0)), ((64, 1000, 64), (1.0, 1.0))]:
        a, b, c = _operands(M, N, K, kn, M + N + K)
        got = _run(lib, gpu, a, b, c, alpha, beta, kn, path=path, bn=bn)
        _check(got, a, b, c, alpha, beta, kn)


@pytest.mark.parametrize("kn", [True, False])
def test_scaled_ring_and_slices(lib, gpu, kn):
    # the NN loads at every ring depth and slice count (wraps and K tails)
    for path, bn in [(SQUARE, 128), (PAIR, 256)]:
        for katoms in (1, 2):
            fixed = dict(path=path, bn=bn, katoms=katoms, epi_warps=4)
            deepest = lib.query_config(512, 512, 4096, **fixed)["kstage"]
            for ks in range(2, deepest + 1):
                K = 64 * katoms * (ks + 1) + 8
                a, b, c = _operands(512, 512, K, kn, ks * 7 + katoms)
                got = _run(lib, gpu, a, b, c, 0.75, -1.25, kn, kstage=ks,
                           max_ctas=2 if path == PAIR else 1, **fixed)
                _check(got, a, b, c, 0.75, -1.25, kn)


def test_scaled_small_integers_bit_exact(lib, gpu):
    # integer operands and dyadic scalars: every partial sum and alpha*S + beta*C
    # is exact in fp32, so the result must match the oracle bit for bit
    rng = np.random.default_rng(5)
    M, N, K = 256, 384, 512
    ai = rng.integers(-2, 3, (M, K))
    bi = rng.integers(-2, 3, (K, N))
    ci = rng.integers(-64, 65, (M, N))
    a = ai.astype(np.float16).view(np.uint16)
    c = ci.astype(np.float16).view(np.uint16)
    for kn in (True, False):
        b = (bi if kn else bi.T).astype(np.float16).view(np.uint16)
        for path in (SQUARE, PAIR):
            got = _run(lib, gpu, a, b, c, 0.5, -2.0, kn, path=path)
            assert np.array_equal(got, oracle.gemm_scaled(a, b, c, 0.5, -2.0, kn))


def test_in_place_update(lib, gpu):
    # C = alpha A B + beta C with D the same buffer as C
    a, b, c = _operands(384, 520, 264, True, 99)
    got = _run(lib, gpu, a, b, c, 1.25, 0.5, True, in_place=True)
    _check(got, a, b, c, 1.25, 0.5, True)


def test_beta_zero_never_reads_c(lib, gpu):
    a, b, _ = _operands(256, 256, 128, True, 7)
    c_nan = np.full((256, 256), 0x7E00, np.uint16)
    got = _run(lib, gpu, a, b, c_nan, 2.0, 0.0, True)
    assert not np.isnan(got.view(np.float16)).any()
    _check(got, a, b, None, 2.0, 0.0, True)


def test_alpha_zero_copies_c_and_k_zero_scales_c(lib, gpu):
    a, b, c = _operands(200, 136, 64, True, 3)
    got = _run(lib, gpu, a, b, c, 0.0, 1.0, True)
    assert np.array_equal(got, c)
    ta = torch.empty((200, 0), dtype=torch.float16, device=gpu)
    tb = torch.empty((0, 136), dtype=torch.float16, device=gpu)
    d = lib.gemm_f16_scaled(ta, tb, _t(c, gpu), 1.0, -0.5, "kn")
    torch.cuda.synchronize()
    want = (c.view(np.float16).astype(np.float32) * np.float32(-0.5)).astype(np.float16)
    assert np.array_equal(d.cpu().numpy(), want)


def test_scaled_skinny_and_tall(lib, gpu):
    for (M, N, K) in [(128, 4096, 1024), (4096, 256, 256)]:
        for kn in (True, False):
            a, b, c = _operands(M, N, K, kn, M + K)
            got = _run(lib, gpu, a, b, c, 1.0, 1.0, kn)
            _check(got, a, b, c, 1.0, 1.0, kn)


def test_workload_nn_scaled_8192_seeded_rows(lib, gpu):
    # the 8192^3 scaled NN workload in the launch configuration the bench uses;
    # the oracle computes 24 seeded rows plus the tile-seam rows in full
    a, b, spec = synthetic.workload("c7")
    c = synthetic.workload_c("c7")
    d = lib.gemm_f16_scaled(_t(a, gpu), _t(b, gpu), _t(c, gpu), spec["alpha"], spec["beta"], "kn")
    torch.cuda.synchronize()
    got = d.cpu().numpy().view(np.uint16)
    M = spec["M"]
    u = synthetic.uniform01(3007, 24)
    rows = sorted(set((u * M).astype(int).tolist()) | {0, 127, 128, 255, 256, M - 1})
    ref = oracle.gemm_scaled(a[rows], b, c[rows], spec["alpha"], spec["beta"], True)
    st = compare_scaled(got[rows], ref, spec["K"], a, b, c, spec["alpha"], spec["beta"])
    assert st["bad"] == 0, st
    assert np.isfinite(got.view(np.float16)).all()
