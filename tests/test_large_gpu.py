"""GPU parity at sizes past 32-bit element offsets: D with more than 2^31
elements (40960 x 65536 fp16, 5.4 GB), through every way a kernel writes D
or reads C -- the TMA store on the single-CTA and the pair paths, the scaled
epilogue's copies of C (in place, C = D), and the padded call's plain stores
to rows that are not 16-byte aligned.  K is small, so the launches are short
and the oracle checks whole rows: the first and last, and the rows on either
side of 2^31 bytes (row 16384) and of 2^31 elements (row 32768) of D."""
import numpy as np
import pytest
import torch

import oracle
from multistage_smem_pipeline_gb300 import synthetic
from tolerance import compare, compare_scaled

pytestmark = pytest.mark.gpu

M, N = 40960, 65536
ROWS = [0, 16383, 16384, 32767, 32768, M - 1]


@pytest.fixture(scope="module")
def lib(gpu):
    from multistage_smem_pipeline_gb300 import binding
    return binding


def _dev(bits, gpu):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.float16)).to(gpu)


def _rows(d, rows):
    idx = torch.tensor(rows, device=d.device)
    return d.index_select(0, idx).cpu().numpy().view(np.uint16)


def _check_clean(lib):
    status, raw = lib.get_device_error()
    assert status == 0, f"device error word {raw:#x}"


def test_index_range_is_past_32_bits():
    assert M * N > 2 ** 31 and ROWS[3] * N < 2 ** 31 <= ROWS[4] * N
    assert ROWS[1] * N * 2 < 2 ** 31 <= ROWS[2] * N * 2


@pytest.mark.parametrize("path", [1, 3])
def test_output_past_2_31_elements(lib, gpu, path):
    K = 64 if path == 1 else 1088      # the pair path needs K > 1024 in its plan
    a = synthetic.uniform_pm1(401 + path, (M, K))
    b = synthetic.uniform_pm1(402 + path, (N, K))
    d = lib.gemm_tn_f16_ex(_dev(a, gpu), _dev(b, gpu), path=path)
    torch.cuda.synchronize()
    _check_clean(lib)
    got = _rows(d, ROWS)
    del d
    ref = oracle.gemm_tn(a[ROWS], b)
    st = compare(got, ref, K, a, b)
    assert st["bad"] == 0, st


def test_scaled_in_place_past_2_31_elements(lib, gpu):
    # C = D = c_row[i] * c_col[j], products of powers of two: exact in fp16,
    # built on the device without a host copy of the 5.4 GB matrix
    K = 1088
    a = synthetic.uniform_pm1(411, (M, K))
    b = synthetic.uniform_pm1(412, (N, K))
    pick = np.array([0.25, -0.5, 1.0, -2.0], dtype=np.float16)
    c_row = pick[(synthetic.uniform01(413, M) * 4).astype(np.int64)]
    c_col = pick[(synthetic.uniform01(414, N) * 4).astype(np.int64)]
    d = torch.from_numpy(c_row).to(gpu)[:, None] * torch.from_numpy(c_col).to(gpu)[None, :]
    assert d.dtype == torch.float16 and d.is_contiguous()
    lib.gemm_f16_scaled(_dev(a, gpu), _dev(b, gpu), d, 0.75, -0.5, "nk", out=d, path=3)
    torch.cuda.synchronize()
    _check_clean(lib)
    got = _rows(d, ROWS)
    del d
    c = (c_row[ROWS][:, None] * c_col[None, :]).astype(np.float16).view(np.uint16)
    ref = oracle.gemm_scaled(a[ROWS], b, c, 0.75, -0.5, False)
    st = compare_scaled(got, ref, K, a, b, c, 0.75, -0.5)
    assert st["bad"] == 0, st


def test_padded_direct_stores_past_2_31_elements(lib, gpu):
    # N and K odd: no row of A, B or D is 16-byte aligned, so A and B are
    # repacked and the epilogue writes D with plain stores at 64-bit offsets
    n, K = N - 1, 1087
    a = synthetic.uniform_pm1(421, (M, K))
    b = synthetic.uniform_pm1(422, (n, K))
    d = lib.gemm_f16_padded(_dev(a, gpu), _dev(b, gpu), None, 1.0, 0.0, "nk", path=3)
    torch.cuda.synchronize()
    _check_clean(lib)
    got = _rows(d, ROWS)
    del d
    ref = oracle.gemm_tn(a[ROWS], b)
    st = compare(got, ref, K, a, b)
    assert st["bad"] == 0, st
