"""GEMMs launched back to back with programmatic dependent launch: each
kernel may start its set-up while the previous one finishes, so these tests
check that every kernel still sees its predecessor's complete results
(read-after-write), that a kernel never overwrites what its predecessor is
still reading (write-after-read), in plain streams and in CUDA graphs, and
that launching with and without it gives identical bits."""
import numpy as np
import pytest
import torch

import oracle
from multistage_smem_pipeline_gb300 import synthetic
from tolerance import compare, compare_scaled

pytestmark = pytest.mark.gpu
SQUARE, PAIR = 1, 3


@pytest.fixture(scope="module")
def lib(gpu):
    from multistage_smem_pipeline_gb300 import binding
    return binding


def _dev(bits, gpu):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.float16)).to(gpu)


def _bits(t):
    return t.cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("path", [SQUARE, PAIR])
def test_chain_reads_each_predecessor(lib, gpu, path):
    # X_{i+1} = (1/16) X_i W^T, eight launches back to back on one stream;
    # every step is checked against the oracle applied to the GPU's own X_i
    M, K = 1024, 256
    w_bits = synthetic.uniform_pm1(201, (K, K))
    xs = [_dev(synthetic.uniform_pm1(202, (M, K)), gpu)]
    w = _dev(w_bits, gpu)
    opts = dict(path=path, bn=256)
    for _ in range(8):
        xs.append(lib.gemm_f16_scaled(xs[-1], w, None, 1.0 / 16, 0.0, "nk", **opts))
    torch.cuda.synchronize()
    assert lib.get_device_error()[0] == lib.GEMM_OK
    for i in range(8):
        x_bits = _bits(xs[i])
        ref = oracle.gemm_scaled(x_bits, w_bits, None, 1.0 / 16, 0.0, False)
        st = compare_scaled(_bits(xs[i + 1]), ref, K, x_bits, w_bits, None, 1.0 / 16, 0.0)
        assert st["bad"] == 0, (i, st)


@pytest.mark.parametrize("path", [SQUARE, PAIR])
def test_next_kernel_overwrites_inputs_only_after_they_are_read(lib, gpu, path):
    # GEMM 1 reads A; GEMM 2, launched right after it, writes its result into
    # A's buffer.  GEMM 1's result must be that of the original A.
    M, N, K = 2048, 512, 2048
    a_bits = synthetic.uniform_pm1(211, (M, K))
    b_bits = synthetic.uniform_pm1(212, (N, K))
    e_bits = synthetic.uniform_pm1(213, (M, 256))
    f_bits = synthetic.uniform_pm1(214, (K, 256))
    a, b, e, f = (_dev(x, gpu) for x in (a_bits, b_bits, e_bits, f_bits))
    d = lib.gemm_tn_f16_ex(a, b, path=path)
    lib.gemm_tn_f16_ex(e, f, out=a, path=path)        # A <- E F^T (M x K)
    torch.cuda.synchronize()
    st = compare(_bits(d), oracle.gemm_tn(a_bits, b_bits), K, a_bits, b_bits)
    assert st["bad"] == 0, st
    st = compare(_bits(a), oracle.gemm_tn(e_bits, f_bits), 256, e_bits, f_bits)
    assert st["bad"] == 0, st


def test_chain_in_a_cuda_graph(lib, gpu):
    M, K = 512, 128
    w_bits = synthetic.uniform_pm1(221, (K, K))
    x0_bits = synthetic.uniform_pm1(222, (M, K))
    w = _dev(w_bits, gpu)
    bufs = [torch.empty((M, K), dtype=torch.float16, device=gpu) for _ in range(5)]
    side = torch.cuda.Stream(gpu)
    g = torch.cuda.CUDAGraph()
    side.wait_stream(torch.cuda.current_stream(gpu))
    with torch.cuda.graph(g, stream=side):
        s = torch.cuda.current_stream(gpu)
        for i in range(4):
            lib.gemm_f16_scaled(bufs[i], w, None, 0.125, 0.0, "nk", out=bufs[i + 1], stream=s)
    torch.cuda.current_stream(gpu).wait_stream(side)
    for rep in range(3):
        bufs[0].copy_(_dev(synthetic.uniform_pm1(223 + rep, (M, K)) if rep else x0_bits, gpu))
        g.replay()
        torch.cuda.synchronize()
        for i in range(4):
            x_bits = _bits(bufs[i])
            ref = oracle.gemm_scaled(x_bits, w_bits, None, 0.125, 0.0, False)
            st = compare_scaled(_bits(bufs[i + 1]), ref, K, x_bits, w_bits, None, 0.125, 0.0)
            assert st["bad"] == 0, (rep, i, st)


@pytest.mark.parametrize("M,N,K", [(1024, 1024, 1024), (81920, 256, 256), (128, 4096, 2048)])
def test_with_and_without_dependent_launch_identical(lib, gpu, M, N, K):
    a = _dev(synthetic.uniform_pm1(231, (M, K)), gpu)
    b = _dev(synthetic.uniform_pm1(232, (N, K)), gpu)
    assert lib.query_config(M, N, K)["pdl"] == 1
    assert lib.query_config(M, N, K, pdl=1)["pdl"] == 0
    outs = []
    for pdl in (0, 1, 0):
        d = torch.empty((M, N), dtype=torch.float16, device=gpu)
        for _ in range(3):
            lib.gemm_tn_f16_ex(a, b, out=d, pdl=pdl)
        outs.append(d)
    torch.cuda.synchronize()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert torch.equal(outs[0].view(torch.int16), outs[2].view(torch.int16))
