"""Failure detection without a GPU fault: every pipeline wait in the kernel has
a time limit.  The test hook makes the producer announce its first stage but
never load it (a barrier that nothing completes); the consumers' bounded
waits run out, the kernel records GEMM_ERR_TIMEOUT and exits cleanly (TMEM
freed, copies drained), and the context stays usable for the next call."""
import numpy as np
import pytest
import torch

import oracle
from multistage_smem_pipeline_gb300 import synthetic
from tolerance import compare, probes_agree

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib(gpu):
    from multistage_smem_pipeline_gb300 import binding
    return binding


@pytest.mark.parametrize("path", [1, 3])
def test_stalled_stage_times_out_and_context_survives(lib, gpu, path):
    a_bits = synthetic.uniform_pm1(1, (256, 512))
    b_bits = synthetic.uniform_pm1(2, (512, 512))
    a = torch.from_numpy(a_bits.view(np.float16)).to(gpu)
    b = torch.from_numpy(b_bits.view(np.float16)).to(gpu)
    assert lib.get_device_error()[0] == lib.GEMM_OK           # clean slate
    lib.gemm_tn_f16_ex(a, b, inject=1, timeout_ns=50_000_000, max_ctas=2, path=path)
    status, raw = lib.get_device_error()
    assert status == lib.GEMM_ERR_TIMEOUT
    assert (raw >> 8) in (1, 2, 3, 4)                          # the site that gave up
    assert lib.get_device_error()[0] == lib.GEMM_OK            # reading clears it
    # the same SMs run a normal GEMM correctly afterwards (TMEM was freed)
    for _ in range(2):
        d = lib.gemm_tn_f16_ex(a, b, path=path)
        torch.cuda.synchronize()
        st = compare(d.cpu().numpy().view(np.uint16), oracle.gemm_tn(a_bits, b_bits), 512,
                     a_bits, b_bits)
        assert st["bad"] == 0
    assert lib.get_device_error()[0] == lib.GEMM_OK


def test_error_words_are_per_stream(lib, gpu):
    """A timeout raised on one stream is reported by that stream's poll only."""
    a_bits = synthetic.uniform_pm1(3, (256, 512))
    b_bits = synthetic.uniform_pm1(4, (512, 512))
    a = torch.from_numpy(a_bits.view(np.float16)).to(gpu)
    b = torch.from_numpy(b_bits.view(np.float16)).to(gpu)
    sx, sy = torch.cuda.Stream(gpu), torch.cuda.Stream(gpu)
    for s in (sx, sy):
        s.wait_stream(torch.cuda.current_stream(gpu))
        assert lib.get_device_error(stream=s)[0] == lib.GEMM_OK
    assert lib.get_device_error()[0] == lib.GEMM_OK
    with torch.cuda.stream(sx):
        lib.gemm_tn_f16_ex(a, b, inject=1, timeout_ns=50_000_000, max_ctas=2, stream=sx)
    with torch.cuda.stream(sy):
        d = lib.gemm_tn_f16_ex(a, b, stream=sy)
    sx.synchronize()
    assert lib.get_device_error(stream=sy)[0] == lib.GEMM_OK      # Y's word is clean
    assert lib.get_device_error()[0] == lib.GEMM_OK               # so is the default stream's
    assert lib.get_device_error(stream=sx)[0] == lib.GEMM_ERR_TIMEOUT
    assert lib.get_device_error(stream=sx)[0] == lib.GEMM_OK      # reading clears it
    st = compare(d.cpu().numpy().view(np.uint16), oracle.gemm_tn(a_bits, b_bits), 512,
                 a_bits, b_bits)
    assert st["bad"] == 0


def test_latency_probes_give_a_stage_count(lib, gpu):
    copy, compute = lib.probe_latencies(bn=256, ctas=0, footprint_bytes=1 << 30, reps=32)
    assert copy > 0 and compute > 0
    s = lib.minimum_stages(int(np.ceil(copy)), int(np.ceil(compute)))
    assert s >= 2
    # a 128 x 256 x 64 k-block is 512 tensor-pipe cycles at the dense fp16 rate
    assert 400 < compute < 1000


def test_latency_probes_repeat_within_tolerance(lib, gpu):
    first = lib.probe_latencies(bn=256, ctas=0, footprint_bytes=16 << 20, reps=64)
    second = lib.probe_latencies(bn=256, ctas=0, footprint_bytes=16 << 20, reps=64)
    assert probes_agree(first, second), (first, second)
