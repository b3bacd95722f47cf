"""The allocation-free latency probe, gemm_probe_latencies_static.

Some callers cannot allocate device memory: a serving process whose memory
pool already holds nearly all of HBM, or a loop that must not call cudaMalloc
or cudaFree because those can synchronise the device.  For them the library
offers a probe entry point whose copy measurement loads from a fixed 16 MiB
array the library owns, instead of from a region the caller allocates.

This file calls that entry point through the C-ABI twice in a row and checks
each result against the allocating entry point (gemm_probe_latencies) run on
a caller-allocated region of the same size, within the probe tolerance the
other probe tests use.  It is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

from tolerance import probes_agree

pytestmark = pytest.mark.gpu

FOOTPRINT = 16 << 20     # the entry point's stated maximum


@pytest.fixture(scope="module")
def lib(gpu):
    from multistage_smem_pipeline_gb300 import binding
    return binding


def _static(lib, footprint, stream):
    c, m = ctypes.c_double(0), ctypes.c_double(0)
    rc = lib.LIB.gemm_probe_latencies_static(256, 0, footprint, 64, ctypes.byref(c),
                                             ctypes.byref(m), stream)
    return rc, (c.value, m.value)


def _allocating(lib, scratch, footprint, stream):
    c, m = ctypes.c_double(0), ctypes.c_double(0)
    rc = lib.LIB.gemm_probe_latencies(256, 0, scratch.data_ptr(), footprint, 64, ctypes.byref(c),
                                      ctypes.byref(m), stream)
    return rc, (c.value, m.value)


def test_static_scratch_probe_matches_allocating_probe(lib, gpu):
    stream = torch.cuda.current_stream(gpu).cuda_stream
    scratch = torch.zeros(FOOTPRINT // 2, dtype=torch.float16, device=gpu)
    for call in range(2):                    # two calls in a row share the library's array
        free_before = torch.cuda.mem_get_info(gpu)[0]
        rc, got = _static(lib, FOOTPRINT, stream)
        free_after = torch.cuda.mem_get_info(gpu)[0]
        assert rc == lib.GEMM_OK, lib.status_string(rc)
        if call == 1:
            # Set up by the first call, the second allocates nothing: device
            # memory is handed out in pages of at least 2 MiB, and a reload
            # of the array would take 16 MiB.
            assert free_before - free_after < (1 << 20), (free_before, free_after)
        rc, ref = _allocating(lib, scratch, FOOTPRINT, stream)
        assert rc == lib.GEMM_OK, lib.status_string(rc)
        assert got[0] > 0 and got[1] > 0
        assert probes_agree(got, ref), (got, ref)


def test_static_scratch_probe_rejects_footprint_beyond_its_array(lib, gpu):
    stream = torch.cuda.current_stream(gpu).cuda_stream
    rc, _ = _static(lib, FOOTPRINT + 128, stream)
    assert rc == lib.GEMM_ERR_INVALID_VALUE
