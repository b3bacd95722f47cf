"""GPU parity of the fp16-accumulate option (acc_f16=1) against the oracle's
slice-by-slice fp16 accumulation -- the arithmetic of the F16F16F16F16 MMA
atom of "cute(9) multistage_gemm" (one fp16 rounding per 16-deep K slice).

How the tensor core rounds inside one slice is not specified, so general
inputs are compared within a per-slice bound: each of the ceil(K/16)
roundings may differ by an ulp of the running sum, which never exceeds
sum_k |a_k b_k|.  Where every partial sum is exact in fp16 ({-1,0,1}
operands) the result must match bit for bit; with a single slice (K <= 16)
it must be within one ulp.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from multistage_smem_pipeline_gb300 import synthetic
from tolerance import fp16_ulp

pytestmark = pytest.mark.gpu
SQUARE, PAIR = 1, 3


@pytest.fixture(scope="module")
def lib(gpu):
    from multistage_smem_pipeline_gb300 import binding
    return binding


def _run(lib, gpu, a_bits, b_bits, **opts):
    a = torch.from_numpy(np.ascontiguousarray(a_bits).view(np.float16)).to(gpu)
    b = torch.from_numpy(np.ascontiguousarray(b_bits).view(np.float16)).to(gpu)
    d = lib.gemm_tn_f16_ex(a, b, acc_f16=1, **opts)
    torch.cuda.synchronize()
    status, raw = lib.get_device_error()
    assert status == 0, f"device error word {raw:#x}"
    return d.cpu().numpy().view(np.uint16)


def _slice_bound_check(got, a_bits, b_bits):
    ref = oracle.gemm_tn_f16acc(a_bits, b_bits)
    a = np.abs(a_bits.view(np.float16).astype(np.float64))
    b = np.abs(b_bits.view(np.float16).astype(np.float64))
    s_abs = a @ b.T
    slices = math.ceil(a.shape[1] / 16)
    g = got.view(np.float16).astype(np.float64)
    r = ref.view(np.float16).astype(np.float64)
    tol = 2 * slices * fp16_ulp(s_abs) + fp16_ulp(r)
    err = np.abs(g - r)
    assert np.isfinite(g).all()
    assert int(np.count_nonzero(err > tol)) == 0, float(err.max())
    return float(np.mean(got == ref))


@pytest.mark.parametrize("path", [SQUARE, PAIR])
def test_f16acc_ternary_is_bit_exact(lib, gpu, path):
    a, b, _ = synthetic.workload("c2")
    got = _run(lib, gpu, a, b, path=path)
    assert np.array_equal(got, oracle.gemm_tn_f16acc(a, b))


@pytest.mark.parametrize("K", [8, 16])
def test_f16acc_single_slice_within_one_ulp(lib, gpu, K):
    a = synthetic.uniform_pm1(K, (300, K))
    b = synthetic.uniform_pm1(K + 1, (264, K))
    got = _run(lib, gpu, a, b)
    ref = oracle.gemm_tn_f16acc(a, b)
    g = got.view(np.float16).astype(np.float64)
    r = ref.view(np.float16).astype(np.float64)
    assert np.all(np.abs(g - r) <= fp16_ulp(r))


@pytest.mark.parametrize("path", [SQUARE, PAIR])
@pytest.mark.parametrize("K", [200, 512, 1032])
def test_f16acc_general_within_slice_bound(lib, gpu, path, K):
    a = (synthetic.uniform01(K, 384 * K) * 0.125 - 0.0625).astype(np.float16).view(np.uint16)
    a = a.reshape(384, K)
    b = synthetic.uniform_pm1(K + 2, (520, K))
    got = _run(lib, gpu, a, b, path=path)
    _slice_bound_check(got, a, b)


def test_f16acc_scaled_form(lib, gpu):
    a, b = synthetic.ternary(61, (256, 512)), synthetic.ternary(62, (512, 384))
    c = synthetic.ternary(63, (256, 384))
    ta, tb, tc = (torch.from_numpy(x.view(np.float16)).to(gpu) for x in (a, b, c))
    d = lib.gemm_f16_scaled(ta, tb, tc, 2.0, -1.0, "kn", acc_f16=1)
    torch.cuda.synchronize()
    # integer partial sums (exact in fp16), dyadic scalars: exact
    ai = a.view(np.float16).astype(np.int64); bi = b.view(np.float16).astype(np.int64)
    ci = c.view(np.float16).astype(np.int64)
    want = (2 * (ai @ bi) - ci).astype(np.float16).view(np.uint16)
    assert np.array_equal(d.cpu().numpy().view(np.uint16), want)


def test_workload_tall_f16acc(lib, gpu):
    # the shape and the accumulator of the multistage page's own measurement
    a, b, spec = synthetic.workload("c8")
    got = _run(lib, gpu, a, b)
    _slice_bound_check(got, a, b)
