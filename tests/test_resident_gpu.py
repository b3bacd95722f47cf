"""GPU parity of the resident-B mode of the single-CTA kernel (one n-block:
every CTA loads all of B into shared memory once and streams only A) against
the oracle, through the C-ABI.  The MMAs are issued in the same order as
with B streamed through the ring, so the two modes must agree bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from multistage_smem_pipeline_gb300 import synthetic
from tolerance import compare, compare_scaled

pytestmark = pytest.mark.gpu
SQUARE = 1


@pytest.fixture(scope="module")
def lib(gpu):
    from multistage_smem_pipeline_gb300 import binding
    return binding


def _dev(bits, gpu):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.float16)).to(gpu)


def _run(lib, gpu, a_bits, b_bits, **opts):
    d = lib.gemm_tn_f16_ex(_dev(a_bits, gpu), _dev(b_bits, gpu), **opts)
    torch.cuda.synchronize()
    status, raw = lib.get_device_error()
    assert status == 0, f"device error word {raw:#x}"
    return d.cpu().numpy().view(np.uint16)


SHAPES = [(300, 256, 256), (1000, 200, 304), (640, 96, 600), (129, 8, 72), (257, 64, 136),
          (1, 8, 8), (4000, 256, 64)]


@pytest.mark.parametrize("M,N,K,bn", [(7680, 384, 64, 128), (4100, 256, 256, 128),
                                      (2000, 512, 128, 256), (3000, 200, 192, 64)])
def test_resident_several_n_blocks(lib, gpu, M, N, K, bn):
    # each CTA keeps the one n-block its tiles share (grid a multiple of num_n)
    a = synthetic.uniform_pm1(M + 7 * K, (M, K))
    b = synthetic.uniform_pm1(N + 11 * K, (N, K))
    cfg = lib.query_config(M, N, K, path=SQUARE, bn=bn, b_resident=2)
    num_n = -(-N // bn)
    assert cfg["b_resident"] == 1 and cfg["ctas"] % num_n == 0
    res = _run(lib, gpu, a, b, path=SQUARE, bn=bn, b_resident=2)
    st = compare(res, oracle.gemm_tn(a, b), K, a, b)
    assert st["bad"] == 0, st
    streamed = _run(lib, gpu, a, b, path=SQUARE, bn=bn, b_resident=1, katoms=cfg["katoms"],
                    epi_warps=cfg["epi_warps"])
    assert np.array_equal(res, streamed)


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_resident_matches_oracle_and_streamed(lib, gpu, M, N, K):
    a = synthetic.uniform_pm1(M * 3 + K, (M, K))
    b = synthetic.uniform_pm1(N * 5 + K, (N, K))
    cfg = lib.query_config(M, N, K, path=SQUARE, b_resident=2)
    assert cfg["b_resident"] == 1
    res = _run(lib, gpu, a, b, path=SQUARE, b_resident=2)
    st = compare(res, oracle.gemm_tn(a, b), K, a, b)
    assert st["bad"] == 0, st
    streamed = _run(lib, gpu, a, b, path=SQUARE, b_resident=1, bn=cfg["bn"],
                    katoms=cfg["katoms"], epi_warps=cfg["epi_warps"])
    assert np.array_equal(res, streamed)


@pytest.mark.parametrize("katoms", [1, 2])
@pytest.mark.parametrize("epi", [4, 8])
def test_resident_every_ring_depth(lib, gpu, katoms, epi):
    # the A ring wraps many times per CTA while B stays put
    M, N, K = 2048, 128, 320
    a = synthetic.uniform_pm1(91 + katoms, (M, K))
    b = synthetic.uniform_pm1(92 + epi, (N, K))
    ref = oracle.gemm_tn(a, b)
    fixed = dict(path=SQUARE, bn=128, katoms=katoms, epi_warps=epi, b_resident=2)
    deepest = lib.query_config(M, N, K, **fixed)["kstage"]
    assert deepest >= 2
    for ks in range(2, deepest + 1):
        got = _run(lib, gpu, a, b, kstage=ks, max_ctas=3, **fixed)
        st = compare(got, ref, K, a, b)
        assert st["bad"] == 0, (ks, st)


@pytest.mark.parametrize("bn", [32, 64, 160, 256])
def test_resident_tile_widths(lib, gpu, bn):
    M, N, K = 1500, bn, 192
    a = synthetic.uniform_pm1(bn, (M, K))
    b = synthetic.uniform_pm1(bn + 1, (N, K))
    got = _run(lib, gpu, a, b, path=SQUARE, bn=bn, b_resident=2)
    st = compare(got, oracle.gemm_tn(a, b), K, a, b)
    assert st["bad"] == 0, st


def test_resident_ternary_bit_exact(lib, gpu):
    M, N, K = 3000, 256, 256
    a = synthetic.ternary(101, (M, K))
    b = synthetic.ternary(102, (N, K))
    got = _run(lib, gpu, a, b, path=SQUARE, b_resident=2)
    ref = oracle.gemm_tn(a, b)
    assert np.array_equal(got.view(np.float16).astype(np.float64),
                          ref.view(np.float16).astype(np.float64))


def test_resident_scaled_and_fp16_accumulator(lib, gpu):
    M, N, K = 1200, 256, 256
    a = synthetic.uniform_pm1(111, (M, K))
    b = synthetic.uniform_pm1(112, (N, K))
    c = synthetic.uniform_pm1(113, (M, N))
    d = lib.gemm_f16_scaled(_dev(a, gpu), _dev(b, gpu), _dev(c, gpu), -1.5, 0.25, "nk",
                            path=SQUARE, b_resident=2)
    torch.cuda.synchronize()
    got = d.cpu().numpy().view(np.uint16)
    ref = oracle.gemm_scaled(a, b, c, -1.5, 0.25, False)
    st = compare_scaled(got, ref, K, a, b, c, -1.5, 0.25)
    assert st["bad"] == 0, st
    # the fp16 accumulator: same MMA order as streamed B, so identical bits
    res = _run(lib, gpu, a, b, path=SQUARE, b_resident=2, acc_f16=1)
    cfg = lib.query_config(M, N, K, path=SQUARE, b_resident=2)
    streamed = _run(lib, gpu, a, b, path=SQUARE, b_resident=1, acc_f16=1, bn=cfg["bn"],
                    katoms=cfg["katoms"], epi_warps=cfg["epi_warps"])
    assert np.array_equal(res, streamed)


def test_tall_shapes_choose_resident_where_it_keeps_more_a_in_flight(lib, gpu):
    # resident B when it leaves A's ring deeper than streaming B would (or as deep, with
    # several n-blocks); the page's 81920 x 256 x 256 (one n-block, the same depth either
    # way) and its fp16-accumulator variant stream B
    assert lib.query_config(81920, 1024, 128)["b_resident"] == 1
    assert lib.query_config(81920, 512, 256)["b_resident"] == 1
    assert lib.query_config(65536, 128, 512)["b_resident"] == 0
    for tag in ("c6", "c8"):
        spec = synthetic.WORKLOADS[tag]
        assert lib.query_config(spec["M"], spec["N"], spec["K"])["b_resident"] == 0
        assert lib.query_config(spec["M"], spec["N"], spec["K"], b_resident=2)["b_resident"] == 1


def test_resident_stall_times_out_and_context_survives(lib, gpu):
    M, N, K = 1024, 256, 256
    a_bits = synthetic.uniform_pm1(121, (M, K))
    b_bits = synthetic.uniform_pm1(122, (N, K))
    a, b = _dev(a_bits, gpu), _dev(b_bits, gpu)
    assert lib.get_device_error()[0] == lib.GEMM_OK
    lib.gemm_tn_f16_ex(a, b, inject=1, timeout_ns=50_000_000, max_ctas=2, path=SQUARE,
                       b_resident=2)
    status, raw = lib.get_device_error()
    assert status == lib.GEMM_ERR_TIMEOUT
    assert (raw >> 8) in (1, 2, 3, 4)
    d = lib.gemm_tn_f16_ex(a, b, path=SQUARE, b_resident=2)
    torch.cuda.synchronize()
    st = compare(d.cpu().numpy().view(np.uint16), oracle.gemm_tn(a_bits, b_bits), K, a_bits,
                 b_bits)
    assert st["bad"] == 0
    assert lib.get_device_error()[0] == lib.GEMM_OK
