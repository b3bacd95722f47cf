"""The pipeline invariant check (option `check`): with it on, every ring slot
carries the sequence number of the fill that produced it and the MMA thread
compares it with its own count when it consumes the slot -- the read-after-
write discipline of "第 6 课：Shared Memory 布局与异步流水" (section 3) checked
slot by slot.  A mismatch is recorded as GEMM_ERR_INVARIANT (site 5) in the
device error word and the kernel runs on; nothing traps.

Each kernel runs with the check on and must report nothing and stay exact
against the oracle; the host-selected hook inject=2 makes the producer stamp
its first slot wrongly (nothing else changes), which the check must report,
after which the context serves the next call normally."""
import numpy as np
import pytest
import torch

import oracle
from multistage_smem_pipeline_gb300 import synthetic
from tolerance import compare

pytestmark = pytest.mark.gpu

# (M, N, K, options) covering every kernel: single-CTA, resident B, narrow and
# wide pairs, the small-M kernel and the split-K pair
KERNELS = {
    "single_cta": (300, 520, 640, dict(path=1, split_k=1)),
    "resident_b": (2048, 256, 256, dict(b_resident=2)),
    "pair_narrow": (512, 512, 2048, dict(path=3, wide=1)),
    "pair_wide": (512, 1024, 4096, dict(path=3, wide=2)),
    "small_m": (128, 2048, 1024, dict(small_m=2)),
    "split_k": (512, 512, 1024, dict(split_k=2)),
}


@pytest.fixture(scope="module")
def lib(gpu):
    from multistage_smem_pipeline_gb300 import binding
    return binding


def _ops(M, N, K, gpu, seed):
    a = synthetic.ternary(seed, (M, K))
    b = synthetic.ternary(seed + 1, (N, K))
    return a, b, torch.from_numpy(a.view(np.float16)).to(gpu), \
        torch.from_numpy(b.view(np.float16)).to(gpu)


@pytest.mark.parametrize("kind", sorted(KERNELS))
def test_check_on_reports_nothing_and_results_stay_exact(lib, gpu, kind):
    M, N, K, opts = KERNELS[kind]
    a_bits, b_bits, a, b = _ops(M, N, K, gpu, 11)
    assert lib.get_device_error()[0] == lib.GEMM_OK
    d = lib.gemm_tn_f16_ex(a, b, check=1, **opts)
    torch.cuda.synchronize()
    assert lib.get_device_error()[0] == lib.GEMM_OK
    st = compare(d.cpu().numpy().view(np.uint16), oracle.gemm_tn(a_bits, b_bits), K, a_bits, b_bits)
    assert st["bad"] == 0 and st["exact_frac"] == 1.0, st     # integer sums: exact


@pytest.mark.parametrize("kind", sorted(KERNELS))
def test_a_slot_out_of_sequence_is_reported(lib, gpu, kind):
    M, N, K, opts = KERNELS[kind]
    a_bits, b_bits, a, b = _ops(M, N, K, gpu, 21)
    assert lib.get_device_error()[0] == lib.GEMM_OK
    lib.gemm_tn_f16_ex(a, b, check=1, inject=2, **opts)
    status, raw = lib.get_device_error()
    assert status == lib.GEMM_ERR_INVARIANT and (raw >> 8) == 5, (status, hex(raw))
    assert lib.get_device_error()[0] == lib.GEMM_OK              # reading clears it
    # the planted stamp changed nothing else: the result of that call and of the next are exact
    d = lib.gemm_tn_f16_ex(a, b, **opts)
    torch.cuda.synchronize()
    assert lib.get_device_error()[0] == lib.GEMM_OK
    ref = oracle.gemm_tn(a_bits, b_bits)
    assert np.array_equal(d.cpu().numpy().view(np.uint16), ref)


def test_planted_stamp_without_the_check_is_silent(lib, gpu):
    M, N, K, opts = KERNELS["pair_wide"]
    a_bits, b_bits, a, b = _ops(M, N, K, gpu, 31)
    d = lib.gemm_tn_f16_ex(a, b, inject=2, **opts)
    torch.cuda.synchronize()
    assert lib.get_device_error()[0] == lib.GEMM_OK
    assert np.array_equal(d.cpu().numpy().view(np.uint16), oracle.gemm_tn(a_bits, b_bits))


def test_check_is_refused_where_it_is_not_built(lib, gpu):
    # built for the plain forms only: a scaled epilogue or a directly stored D is refused
    a = torch.zeros((256, 512), dtype=torch.float16, device=gpu)
    b = torch.zeros((256, 512), dtype=torch.float16, device=gpu)
    c = torch.zeros((256, 256), dtype=torch.float16, device=gpu)
    with pytest.raises(lib.GemmError) as e:
        lib.gemm_f16_scaled(a, b, c, 1.5, -0.5, "nk", check=1)
    assert e.value.status == lib.GEMM_ERR_INVALID_VALUE
    with pytest.raises(lib.GemmError) as e:
        lib.gemm_f16_padded(a, torch.zeros((255, 512), dtype=torch.float16, device=gpu), None,
                            1.0, 0.0, "nk", check=1)
    assert e.value.status == lib.GEMM_ERR_INVALID_VALUE
    assert lib.get_device_error()[0] == lib.GEMM_OK
