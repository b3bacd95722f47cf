"""Seeded random shapes and options through the C-ABI against the oracle: the
plain, scaled and padded entries, both B layouts, both kernel paths, forced
tile widths, ring depths, slices per stage, epilogue warps, resident B, wide
pair units and the fp16 accumulator."""
import numpy as np
import pytest
import torch

import oracle
from multistage_smem_pipeline_gb300 import synthetic
from tolerance import compare_scaled, fp16_ulp

pytestmark = pytest.mark.gpu
N_CASES = 48


@pytest.fixture(scope="module")
def lib(gpu):
    from multistage_smem_pipeline_gb300 import binding
    return binding


def _case(i):
    """Shape, entry and options of case i, drawn from a seeded stream."""
    u = synthetic.uniform01(7000 + i, 17)
    pick = lambda x, options: options[min(int(x * len(options)), len(options) - 1)]
    entry = pick(u[0], ["plain", "scaled", "padded"])
    kn = entry != "plain" and u[1] < 0.5
    M = 1 + int(u[2] * 700)
    N = 8 * (1 + int(u[3] * 90))
    K = 8 * (1 + int(u[4] * 140))
    if entry == "padded":              # any N and K
        N = 1 + int(u[3] * 720)
        K = 1 + int(u[4] * 1120)
    opts = {}
    path = pick(u[5], [0, 0, 1, 3])
    if path:
        opts["path"] = path
    if u[6] < 0.4:
        step = 64 if kn else 32
        if kn and path == 3:
            step = 128
        opts["bn"] = pick(u[7], list(range(step, 257, step)))
    if u[8] < 0.3:
        opts["katoms"] = pick(u[9], [1, 2])
    if u[10] < 0.3:
        opts["epi_warps"] = pick(u[11], [4, 8])
    if u[12] < 0.15 and not kn:
        opts["acc_f16"] = 1
    if u[13] < 0.2:
        opts["b_resident"] = pick(u[14], [1, 2])
    if path == 3 and u[16] < 0.5:
        opts["wide"] = 2
    alpha, beta = (1.0, 0.0)
    if entry != "plain":
        alpha = pick(u[15], [1.0, -0.5, 2.0])
        beta = pick(u[14], [0.0, 0.5, -1.0])
    return entry, kn, M, N, K, opts, alpha, beta


def _dev(bits, gpu):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.float16)).to(gpu)


@pytest.mark.parametrize("i", range(N_CASES))
def test_fuzz_case(lib, gpu, i):
    entry, kn, M, N, K, opts, alpha, beta = _case(i)
    a = synthetic.uniform_pm1(7100 + i, (M, K))
    b = synthetic.uniform_pm1(7200 + i, (K, N) if kn else (N, K))
    c = synthetic.uniform_pm1(7300 + i, (M, N))
    layout = "kn" if kn else "nk"
    try:
        if entry == "plain":
            d = lib.gemm_tn_f16_ex(_dev(a, gpu), _dev(b, gpu), **opts)
        elif entry == "scaled":
            d = lib.gemm_f16_scaled(_dev(a, gpu), _dev(b, gpu), _dev(c, gpu), alpha, beta, layout,
                                    **opts)
        else:
            d = lib.gemm_f16_padded(_dev(a, gpu), _dev(b, gpu), _dev(c, gpu), alpha, beta, layout,
                                    **opts)
    except lib.GemmError as e:
        # an explicit option the shape cannot honour is refused before any launch
        assert e.status == lib.GEMM_ERR_INVALID_VALUE and opts, (entry, M, N, K, opts)
        return
    torch.cuda.synchronize()
    status, raw = lib.get_device_error()
    assert status == 0, f"device error word {raw:#x}"
    got = d.cpu().numpy().view(np.uint16)
    if opts.get("acc_f16"):
        ref = oracle.gemm_tn_f16acc(a, b) if entry == "plain" else None
        if ref is None:  # scaled/padded with fp16 accumulation: the bound below, from the slices
            s = oracle.gemm_tn_f16acc(a, b.T.copy() if kn else b)
            ref = oracle.gemm_scaled(s, np.eye(N, dtype=np.float16).view(np.uint16), c, alpha,
                                     beta, False)
        g = got.view(np.float16).astype(np.float64)
        r = ref.view(np.float16).astype(np.float64)
        s_abs = np.abs(a.view(np.float16).astype(np.float64)) @ \
            np.abs((b.T if kn else b).view(np.float16).astype(np.float64)).T
        tol = (2 * -(-K // 16) * fp16_ulp(s_abs) * abs(alpha) + 2 * fp16_ulp(r) +
               2.0 ** -20 * abs(beta))
        assert np.all(np.abs(g - r) <= tol), (entry, M, N, K, opts)
        return
    ref = oracle.gemm_scaled(a, b, c if beta else None, alpha, beta, kn)
    st = compare_scaled(got, ref, K, a, b, c, alpha, beta)
    assert st["bad"] == 0, (entry, kn, M, N, K, opts, alpha, beta, st)
