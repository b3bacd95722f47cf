"""GPU parity of the pair kernel's wide units (two adjacent n-tiles sharing
each A slice, one TMEM accumulator each) against the oracle, through the
C-ABI.  Each accumulator receives the same MMAs in the same order as with
one tile per unit, so the two schedules must agree bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from multistage_smem_pipeline_gb300 import synthetic
from tolerance import compare, compare_scaled

pytestmark = pytest.mark.gpu
PAIR = 3
WIDE = dict(path=PAIR, wide=2)
NARROW = dict(path=PAIR, wide=1)


@pytest.fixture(scope="module")
def lib(gpu):
    from multistage_smem_pipeline_gb300 import binding
    return binding


def _dev(bits, gpu):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.float16)).to(gpu)


def _host(d):
    return d.cpu().numpy().view(np.uint16)


def _run(lib, gpu, a_bits, b_bits, **opts):
    d = lib.gemm_tn_f16_ex(_dev(a_bits, gpu), _dev(b_bits, gpu), **opts)
    torch.cuda.synchronize()
    status, raw = lib.get_device_error()
    assert status == 0, f"device error word {raw:#x}"
    return _host(d)


# (M, N, K, bn): whole units, a ragged last unit whose second tile is partly
# or wholly past N, a single unit with an empty second tile, narrow tiles
SHAPES = [(600, 1000, 1152, 256), (300, 304, 200, 256), (257, 256, 520, 256),
          (1024, 1536, 2048, 256), (513, 2600, 136, 256), (700, 720, 264, 64),
          (384, 96, 96, 32), (1300, 1000, 1032, 160), (256, 512, 8, 128)]


@pytest.mark.parametrize("M,N,K,bn", SHAPES)
def test_wide_matches_oracle_and_narrow(lib, gpu, M, N, K, bn):
    a = synthetic.uniform_pm1(M * 7 + K, (M, K))
    b = synthetic.uniform_pm1(N * 3 + K, (N, K))
    cfg = lib.query_config(M, N, K, bn=bn, **WIDE)
    num_n = -(-N // bn)
    units = -(-M // 256) * -(-num_n // 2)
    assert cfg["wide"] == 1 and cfg["ctas"] <= 2 * units
    got = _run(lib, gpu, a, b, bn=bn, **WIDE)
    st = compare(got, oracle.gemm_tn(a, b), K, a, b)
    assert st["bad"] == 0, st
    assert np.array_equal(got, _run(lib, gpu, a, b, bn=bn, **NARROW))


@pytest.mark.parametrize("epi", [4, 8])
def test_wide_every_ring_depth_one_pair(lib, gpu, epi):
    # one pair walks every unit: the ring wraps many times and the
    # accumulator phase flips once per unit
    M, N, K = 1024, 1280, 520
    a = synthetic.uniform_pm1(201 + epi, (M, K))
    b = synthetic.uniform_pm1(202 + epi, (N, K))
    ref = oracle.gemm_tn(a, b)
    fixed = dict(bn=128, katoms=1, epi_warps=epi, **WIDE)
    deepest = lib.query_config(M, N, K, **fixed)["kstage"]
    assert deepest >= 4
    for ks in range(2, deepest + 1):
        got = _run(lib, gpu, a, b, kstage=ks, max_ctas=2, **fixed)
        st = compare(got, ref, K, a, b)
        assert st["bad"] == 0, (ks, st)


@pytest.mark.parametrize("katoms", [1, 2])
def test_wide_slices_per_stage(lib, gpu, katoms):
    M, N, K = 800, 1024, 1000
    a = synthetic.uniform_pm1(211 + katoms, (M, K))
    b = synthetic.uniform_pm1(212 + katoms, (N, K))
    got = _run(lib, gpu, a, b, katoms=katoms, **WIDE)
    st = compare(got, oracle.gemm_tn(a, b), K, a, b)
    assert st["bad"] == 0, st
    assert np.array_equal(got, _run(lib, gpu, a, b, katoms=katoms, **NARROW))


def test_wide_ternary_bit_exact(lib, gpu):
    M, N, K = 1000, 1304, 2048
    a = synthetic.ternary(221, (M, K))
    b = synthetic.ternary(222, (N, K))
    got = _run(lib, gpu, a, b, **WIDE)
    assert np.array_equal(got.view(np.float16).astype(np.float64),
                          oracle.gemm_tn(a, b).view(np.float16).astype(np.float64))


@pytest.mark.parametrize("layout", ["nk", "kn"])
def test_wide_scaled_in_place(lib, gpu, layout):
    M, N, K = 700, 904, 1104
    kn = layout == "kn"
    a = synthetic.uniform_pm1(231, (M, K))
    b = synthetic.uniform_pm1(232, (K, N) if kn else (N, K))
    c = synthetic.uniform_pm1(233, (M, N))
    ref = oracle.gemm_scaled(a, b, c, 0.75, -0.5, kn)
    d = _dev(c, gpu)
    lib.gemm_f16_scaled(_dev(a, gpu), _dev(b, gpu), d, 0.75, -0.5, layout, out=d, **WIDE)
    torch.cuda.synchronize()
    got = _host(d)
    st = compare_scaled(got, ref, K, a, b, c, 0.75, -0.5)
    assert st["bad"] == 0, st
    narrow = lib.gemm_f16_scaled(_dev(a, gpu), _dev(b, gpu), _dev(c, gpu), 0.75, -0.5, layout,
                                 **NARROW)
    torch.cuda.synchronize()
    assert np.array_equal(got, _host(narrow))


def test_wide_fp16_accumulator_matches_narrow(lib, gpu):
    M, N, K = 600, 1024, 1536
    a = synthetic.uniform_pm1(241, (M, K))
    b = synthetic.uniform_pm1(242, (N, K))
    # (the narrow schedule's fp16 accumulator is checked against the oracle's
    # per-slice rounding in test_f16acc_gpu)
    got = _run(lib, gpu, a, b, acc_f16=1, **WIDE)
    assert np.array_equal(got, _run(lib, gpu, a, b, acc_f16=1, **NARROW))


@pytest.mark.parametrize("beta", [0.0, 0.5])
def test_wide_padded_entry(lib, gpu, beta):
    # N and K odd: D's rows are misaligned, so with beta = 0 the epilogue
    # stores D directly; with beta != 0 it updates a padded copy of C
    M, N, K = 520, 777, 1035
    a = synthetic.uniform_pm1(251, (M, K))
    b = synthetic.uniform_pm1(252, (N, K))
    c = synthetic.uniform_pm1(253, (M, N))
    d = lib.gemm_f16_padded(_dev(a, gpu), _dev(b, gpu), _dev(c, gpu) if beta else None, 1.25,
                            beta, "nk", **WIDE)
    torch.cuda.synchronize()
    got = _host(d)
    ref = oracle.gemm_scaled(a, b, c if beta else None, 1.25, beta, False)
    st = compare_scaled(got, ref, K, a, b, c, 1.25, beta)
    assert st["bad"] == 0, st
