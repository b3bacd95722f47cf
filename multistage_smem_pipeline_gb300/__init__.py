"""GB300-native multi-stage pipelined fp16 TN GEMM (D = A * B^T).

The compute path is the C-ABI library built from ``csrc/`` (TMA + mbarrier
stage ring + tcgen05/TMEM kernels for sm_103a).  ``binding`` marshals torch
tensors into that library; it has no fallback of any kind.
"""
_EXPORTS = ("gemm_tn_f16", "gemm_tn_f16_ex", "gemm_f16_scaled", "gemm_tn_f16_from_host",
            "get_device_error",
            "minimum_stages", "query_config", "probe_latencies", "library_path", "status_string",
            "GemmError")
__all__ = list(_EXPORTS)


def __getattr__(name):
    # the CUDA library is loaded on first use, so that importing the package
    # (e.g. for ``synthetic``) works on machines without it
    if name in _EXPORTS:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
