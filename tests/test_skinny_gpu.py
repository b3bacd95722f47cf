"""GPU parity of the small-M kernel (gemm_tn_f16_skinny) against the oracle,
through the C-ABI.  The kernel computes one 128 x bn tile per CTA and stages
its epilogue in its ring once the tile's MMAs are done, so its whole shared
memory holds the ring.  It is the skinny path's default (M <= 128, at most one
n-tile per SM); small_m=1 selects the single-CTA kernel instead, and with the
same K slices per stage the two must agree bit for bit (same MMAs in the same
order)."""
import numpy as np
import pytest
import torch

import oracle
from multistage_smem_pipeline_gb300 import synthetic
from tolerance import compare, compare_scaled

pytestmark = pytest.mark.gpu
SKINNY = 2


@pytest.fixture(scope="module")
def lib(gpu):
    from multistage_smem_pipeline_gb300 import binding
    return binding


def _dev(bits, gpu):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.float16)).to(gpu)


def _run(lib, a_bits, b_bits, gpu, **opts):
    a, b = _dev(a_bits, gpu), _dev(b_bits, gpu)
    d = lib.gemm_tn_f16_ex(a, b, **opts)
    torch.cuda.synchronize()
    status, raw = lib.get_device_error()
    assert status == 0, f"device error word {raw:#x}"
    return d.cpu().numpy().view(np.uint16)


def _check(got, a_bits, b_bits):
    st = compare(got, oracle.gemm_tn(a_bits, b_bits), a_bits.shape[1], a_bits, b_bits)
    assert st["bad"] == 0, st
    return st


def test_skinny_shapes_plan_the_small_m_kernel(lib, gpu):
    cfg = lib.query_config(128, 14336, 4096)
    assert cfg["path"] == SKINNY and cfg["small_m"] == 1
    assert cfg["ctas"] == cfg["tiles"] and cfg["epi_warps"] == 4
    # the ring takes the staging buffers' room: one stage deeper than the single-CTA kernel's
    assert cfg["kstage"] > lib.query_config(128, 14336, 4096, small_m=1)["kstage"]
    assert lib.query_config(128, 14336, 4096, small_m=1)["small_m"] == 0
    assert lib.query_config(256, 14336, 4096)["small_m"] == 0       # two m-blocks
    # more n-tiles than SMs: the persistent single-CTA kernel, and small_m=2 is refused
    sms = torch.cuda.get_device_properties(gpu).multi_processor_count
    wide_n = 256 * (sms + 8)
    assert lib.query_config(128, wide_n, 1024, bn=256)["small_m"] == 0
    with pytest.raises(lib.GemmError):
        lib.query_config(128, wide_n, 1024, bn=256, small_m=2)


@pytest.mark.parametrize("katoms", [1, 2])
@pytest.mark.parametrize("M", [1, 16, 33, 100, 128])
def test_rows_and_k_tails(lib, gpu, M, katoms):
    # ragged N (last tile partial) and a K tail inside the last slice
    a = synthetic.gaussian(M, (M, 520))
    b = synthetic.gaussian(M + 1, (1000, 520), 0.02)
    _check(_run(lib, a, b, gpu, path=SKINNY, katoms=katoms), a, b)


@pytest.mark.parametrize("katoms,kstage", [(1, 2), (1, 5), (1, 7), (2, 2), (2, 3), (2, 4)])
def test_every_ring_depth_and_wrap(lib, gpu, katoms, kstage):
    # K one k-block past two passes of the ring, plus a tail inside a slice
    K = 64 * katoms * (2 * kstage + 1) + 24
    a = synthetic.uniform_pm1(kstage, (128, K))
    b = synthetic.uniform_pm1(kstage + 1, (1000, K))
    got = _run(lib, a, b, gpu, path=SKINNY, katoms=katoms, kstage=kstage, bn=96, small_m=2)
    _check(got, a, b)


@pytest.mark.parametrize("bn", [32, 96, 128, 160, 256])
def test_tile_widths(lib, gpu, bn):
    a = synthetic.gaussian(bn, (128, 1024))
    b = synthetic.gaussian(bn + 1, (2000, 1024), 0.02)
    _check(_run(lib, a, b, gpu, path=SKINNY, bn=bn), a, b)


@pytest.mark.parametrize("katoms", [1, 2])
def test_bit_identical_to_the_single_cta_kernel(lib, gpu, katoms):
    a = synthetic.gaussian(31, (128, 2048))
    b = synthetic.gaussian(32, (3000, 2048), 0.02)
    small = _run(lib, a, b, gpu, path=SKINNY, katoms=katoms, small_m=2)
    single = _run(lib, a, b, gpu, path=SKINNY, katoms=katoms, small_m=1)
    assert np.array_equal(small, single)
    _check(small, a, b)


def test_ternary_is_bit_exact(lib, gpu):
    a = synthetic.ternary(41, (128, 1024))
    b = synthetic.ternary(42, (1000, 1024))
    got = _run(lib, a, b, gpu, path=SKINNY)
    ai = a.view(np.float16).astype(np.int64)
    bi = b.view(np.float16).astype(np.int64)
    assert np.array_equal(got, (ai @ bi.T).astype(np.float16).view(np.uint16))


def test_fp16_accumulator_matches_the_single_cta_kernel(lib, gpu):
    # the fp16 accumulator's arithmetic is checked against its oracle on the
    # other kernels; here the small-M kernel must issue the same MMAs
    a = synthetic.uniform_pm1(51, (100, 768))
    b = synthetic.uniform_pm1(52, (904, 768))
    small = _run(lib, a, b, gpu, path=SKINNY, acc_f16=1, katoms=2, small_m=2)
    single = _run(lib, a, b, gpu, path=SKINNY, acc_f16=1, katoms=2, small_m=1)
    assert np.array_equal(small, single)


@pytest.mark.parametrize("kn", [False, True])
def test_scaled_and_kn_layout(lib, gpu, kn):
    for (M, N, K), (alpha, beta) in [((100, 640, 200), (1.5, -0.5)), ((128, 1024, 1088), (-1.0, 2.0)),
                                      ((7, 128, 64), (0.25, 0.0))]:
        a = synthetic.uniform_pm1(M + N, (M, K))
        b = synthetic.uniform_pm1(M + N + 1, (K, N) if kn else (N, K))
        c = synthetic.uniform_pm1(M + N + 2, (M, N))
        for in_place in (False, True):
            tc = _dev(c, gpu)
            d = lib.gemm_f16_scaled(_dev(a, gpu), _dev(b, gpu), tc, alpha, beta,
                                    "kn" if kn else "nk", out=tc if in_place else None,
                                    path=SKINNY, bn=128, small_m=2)
            torch.cuda.synchronize()
            assert lib.get_device_error()[0] == 0
            got = d.cpu().numpy().view(np.uint16)
            ref = oracle.gemm_scaled(a, b, c, alpha, beta, kn)
            st = compare_scaled(got, ref, K, a, b, c, alpha, beta)
            assert st["bad"] == 0, st


def test_direct_store_of_unaligned_rows(lib, gpu):
    # N odd: D's rows are not 16-byte aligned, so the padded entry has the
    # kernel store D itself (beta == 0)
    M, N, K = 77, 1001, 300
    a = synthetic.uniform_pm1(61, (M, K))
    b = synthetic.uniform_pm1(62, (N, K))
    d = lib.gemm_f16_padded(_dev(a, gpu), _dev(b, gpu), None, 1.0, 0.0, "nk", path=SKINNY,
                            small_m=2)
    torch.cuda.synchronize()
    assert lib.get_device_error()[0] == 0
    _check(d.cpu().numpy().view(np.uint16), a, b)


def test_stalled_stage_times_out_and_context_survives(lib, gpu):
    a_bits = synthetic.uniform_pm1(71, (128, 512))
    b_bits = synthetic.uniform_pm1(72, (512, 512))
    a, b = _dev(a_bits, gpu), _dev(b_bits, gpu)
    assert lib.get_device_error()[0] == lib.GEMM_OK
    lib.gemm_tn_f16_ex(a, b, inject=1, timeout_ns=50_000_000, path=SKINNY, small_m=2)
    status, raw = lib.get_device_error()
    assert status == lib.GEMM_ERR_TIMEOUT
    assert (raw >> 8) in (1, 2, 3, 4)
    for _ in range(2):
        d = lib.gemm_tn_f16_ex(a, b, path=SKINNY, small_m=2)
        torch.cuda.synchronize()
        _check(d.cpu().numpy().view(np.uint16), a_bits, b_bits)
    assert lib.get_device_error()[0] == lib.GEMM_OK


def test_workload_skinny_in_full(lib, gpu):
    a, b, spec = synthetic.workload("c5")
    got = _run(lib, a, b, gpu, small_m=2)
    st = _check(got, a, b)
    assert st["exact_frac"] > 0.95
