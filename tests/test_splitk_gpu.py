"""GPU parity of the split-K kernel (gemm_tn_f16_splitk) against the oracle,
through the C-ABI.  A cluster of two CTAs computes each 128 x bn tile, each
CTA half of the k range; the two exchange their fp32 partials through
distributed shared memory and each rounds and stores half of the tile.  The
sum differs from a single accumulator's only in fp32 rounding, so the usual
bound applies, and integer-valued inputs must still match bit for bit.  With
multicast operands a cluster holds two or four such tiles, and the CTAs that
share a block of A or B each load half of it for both: the MMAs and the sums
are the same, so the results must equal the 2-CTA form's bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from multistage_smem_pipeline_gb300 import synthetic
from tolerance import compare, compare_scaled

pytestmark = pytest.mark.gpu


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


def test_1024_cube_plans_a_split(lib, gpu):
    cfg = lib.query_config(1024, 1024, 1024)
    assert cfg["split_k"] == 1 and cfg["ctas"] == 2 * cfg["tiles"] and cfg["bn"] % 64 == 0
    assert lib.query_config(1024, 1024, 1024, split_k=1)["split_k"] == 0
    assert lib.query_config(8192, 8192, 8192)["split_k"] == 0          # long k loops: the pair path


@pytest.mark.parametrize("M,N,K", [(1024, 1024, 1024), (300, 520, 1000), (129, 264, 136),
                                   (200, 328, 264), (77, 1000, 520), (1, 64, 200),
                                   (640, 384, 1088), (256, 256, 256)])
def test_shapes_with_tails(lib, gpu, M, N, K):
    a = synthetic.uniform_pm1(M + K, (M, K))
    b = synthetic.uniform_pm1(N + K, (N, K))
    _check(_run(lib, a, b, gpu, split_k=2), a, b)


@pytest.mark.parametrize("bn", [64, 128, 192, 256])
@pytest.mark.parametrize("katoms", [1, 2])
def test_tile_widths_and_slices(lib, gpu, bn, katoms):
    if bn == 256 and katoms == 2:
        # two 96 KiB stages and the 64 KiB region for the peer's partial do not fit
        with pytest.raises(lib.GemmError):
            lib.query_config(520, 600, 776, split_k=2, bn=bn, katoms=katoms)
        return
    a = synthetic.gaussian(bn + katoms, (520, 776))
    b = synthetic.gaussian(bn + katoms + 1, (600, 776))
    _check(_run(lib, a, b, gpu, split_k=2, bn=bn, katoms=katoms), a, b)


@pytest.mark.parametrize("kstage", [2, 3])
def test_ring_depths_and_wrap(lib, gpu, kstage):
    # each CTA's half runs through its ring twice and a k-block more
    K = 2 * 128 * (2 * kstage + 1)
    a = synthetic.uniform_pm1(kstage, (384, K))
    b = synthetic.uniform_pm1(kstage + 1, (512, K))
    _check(_run(lib, a, b, gpu, split_k=2, bn=128, katoms=2, kstage=kstage), a, b)


def test_odd_k_block_count(lib, gpu):
    # 5 k-blocks: the even CTA takes 3, the odd one 2
    a = synthetic.uniform_pm1(81, (256, 640))
    b = synthetic.uniform_pm1(82, (384, 640))
    _check(_run(lib, a, b, gpu, split_k=2, bn=128, katoms=2), a, b)


def test_ternary_1024_is_bit_exact_and_deterministic(lib, gpu):
    a, b, _ = synthetic.workload("c2")
    first = _run(lib, a, b, gpu, split_k=2)
    ai = a.view(np.float16).astype(np.int64)
    bi = b.view(np.float16).astype(np.int64)
    assert np.array_equal(first, (ai @ bi.T).astype(np.float16).view(np.uint16))
    assert np.array_equal(first, _run(lib, a, b, gpu, split_k=2))


def test_random_inputs_are_deterministic(lib, gpu):
    a = synthetic.gaussian(91, (1024, 1024))
    b = synthetic.gaussian(92, (1024, 1024))
    runs = [_run(lib, a, b, gpu, split_k=2) for _ in range(3)]
    assert all(np.array_equal(runs[0], r) for r in runs[1:])
    _check(runs[0], a, b)


def test_scaled_epilogue(lib, gpu):
    M, N, K = 300, 512, 704
    a = synthetic.uniform_pm1(101, (M, K))
    b = synthetic.uniform_pm1(102, (N, K))
    c = synthetic.uniform_pm1(103, (M, N))
    for alpha, beta in [(1.5, -0.5), (-2.0, 0.0)]:
        for in_place in (False, True):
            tc = _dev(c, gpu)
            d = lib.gemm_f16_scaled(_dev(a, gpu), _dev(b, gpu), tc, alpha, beta, "nk",
                                    out=tc if in_place else None, split_k=2)
            torch.cuda.synchronize()
            assert lib.get_device_error()[0] == 0
            ref = oracle.gemm_scaled(a, b, c, alpha, beta, False)
            st = compare_scaled(d.cpu().numpy().view(np.uint16), ref, K, a, b, c, alpha, beta)
            assert st["bad"] == 0, st


def test_unsupported_forms_are_refused(lib, gpu):
    a = torch.zeros((256, 512), dtype=torch.float16, device=gpu)
    b = torch.zeros((512, 256), dtype=torch.float16, device=gpu)       # K x N
    with pytest.raises(lib.GemmError):
        lib.gemm_f16_scaled(a, b, None, 1.0, 0.0, "kn", split_k=2)
    with pytest.raises(lib.GemmError):
        lib.gemm_tn_f16_ex(a, b.t().contiguous(), acc_f16=1, split_k=2)
    # odd N: the padded entry's kernel would store D itself, which this kernel does not
    with pytest.raises(lib.GemmError):
        lib.gemm_f16_padded(a, torch.zeros((255, 512), dtype=torch.float16, device=gpu), None,
                            1.0, 0.0, "nk", split_k=2)


def test_stalled_stage_times_out_and_context_survives(lib, gpu):
    a_bits = synthetic.uniform_pm1(111, (512, 1024))
    b_bits = synthetic.uniform_pm1(112, (512, 1024))
    a, b = _dev(a_bits, gpu), _dev(b_bits, gpu)
    assert lib.get_device_error()[0] == lib.GEMM_OK
    lib.gemm_tn_f16_ex(a, b, inject=1, timeout_ns=50_000_000, split_k=2)
    status, raw = lib.get_device_error()
    assert status == lib.GEMM_ERR_TIMEOUT
    assert (raw >> 8) in (1, 2, 3, 4)
    for _ in range(2):
        d = lib.gemm_tn_f16_ex(a, b, split_k=2)
        torch.cuda.synchronize()
        _check(d.cpu().numpy().view(np.uint16), a_bits, b_bits)
    assert lib.get_device_error()[0] == lib.GEMM_OK


def test_multicast_cluster_shapes(lib, gpu):
    # chosen by itself with partners along n and m (8 CTAs), when every cluster of 8 fits
    # at once; asked for, also along n only (one m-block) or m only (one n-block): 4
    assert lib.query_config(1024, 1024, 1024)["cluster"] in (2, 8)
    assert lib.query_config(256, 256, 256)["cluster"] == 8
    assert lib.query_config(100, 1024, 1024, split_k=2)["cluster"] == 2
    assert lib.query_config(100, 1024, 1024, split_k=2, multicast=2)["cluster"] == 4
    assert lib.query_config(1024, 64, 1024, split_k=2, multicast=2)["cluster"] == 4
    assert lib.query_config(100, 64, 1024, split_k=2)["cluster"] == 2
    assert lib.query_config(1024, 1024, 1024, multicast=1)["cluster"] == 2
    assert lib.query_config(1024, 1024, 1024, check=1)["cluster"] == 2
    with pytest.raises(lib.GemmError):
        lib.query_config(100, 64, 1024, split_k=2, multicast=2)   # no partner to share with


@pytest.mark.parametrize("M,N,K", [(1024, 1024, 1024), (300, 520, 1000), (129, 264, 136),
                                   (77, 1000, 520), (640, 384, 1088), (256, 256, 256),
                                   (1000, 120, 512), (384, 640, 320), (136, 136, 768)])
def test_multicast_matches_the_pair_form_bit_for_bit(lib, gpu, M, N, K):
    a = synthetic.uniform_pm1(3 * M + K, (M, K))
    b = synthetic.uniform_pm1(3 * N + K + 1, (N, K))
    cfg = lib.query_config(M, N, K, split_k=2, multicast=2)
    assert cfg["cluster"] in (4, 8)
    print(cfg["cluster"], end=" ")
    mc = _run(lib, a, b, gpu, split_k=2, multicast=2)
    pair = _run(lib, a, b, gpu, split_k=2, multicast=1)
    assert np.array_equal(mc, pair)
    _check(mc, a, b)


@pytest.mark.parametrize("bn,katoms,kstage", [(64, 2, 2), (128, 1, 3), (192, 1, 2), (256, 1, 2)])
def test_multicast_tile_widths_and_ring_wrap(lib, gpu, bn, katoms, kstage):
    # halves of B of bn / 2 rows per CTA; each CTA's k-half wraps its ring
    M, N, K = 520, 4 * bn + 40, 2 * 64 * katoms * (2 * kstage + 1)
    a = synthetic.gaussian(bn + kstage, (M, K))
    b = synthetic.gaussian(bn + kstage + 1, (N, K))
    got = _run(lib, a, b, gpu, split_k=2, multicast=2, bn=bn, katoms=katoms, kstage=kstage)
    assert np.array_equal(got, _run(lib, a, b, gpu, split_k=2, multicast=1, bn=bn, katoms=katoms,
                                    kstage=kstage))
    _check(got, a, b)


def test_multicast_stalled_stage_times_out_and_context_survives(lib, gpu):
    a_bits = synthetic.uniform_pm1(121, (512, 1024))
    b_bits = synthetic.uniform_pm1(122, (512, 1024))
    a, b = _dev(a_bits, gpu), _dev(b_bits, gpu)
    assert lib.get_device_error()[0] == lib.GEMM_OK
    lib.gemm_tn_f16_ex(a, b, inject=1, timeout_ns=50_000_000, split_k=2, multicast=2)
    status, raw = lib.get_device_error()
    assert status == lib.GEMM_ERR_TIMEOUT
    assert (raw >> 8) in (1, 2, 3, 4)
    for _ in range(2):
        d = lib.gemm_tn_f16_ex(a, b, split_k=2, multicast=2)
        torch.cuda.synchronize()
        _check(d.cpu().numpy().view(np.uint16), a_bits, b_bits)
    assert lib.get_device_error()[0] == lib.GEMM_OK
