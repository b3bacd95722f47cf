"""ctypes binding of libgemm_tn_f16.so: argument marshalling only.

Every step of the GEMM runs in the library's CUDA kernels.  There is no CPU
or PyTorch fallback: if the library is missing, importing this module raises.
PyTorch provides device memory and the current stream.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

GEMM_OK = 0
GEMM_ERR_INVALID_VALUE = 1
GEMM_ERR_MISALIGNED = 2
GEMM_ERR_UNSUPPORTED_DEVICE = 3
GEMM_ERR_LAUNCH = 4
GEMM_ERR_TIMEOUT = 5
GEMM_ERR_CUDA = 6
GEMM_ERR_INVARIANT = 7

PATH_AUTO, PATH_SQUARE, PATH_SKINNY, PATH_PAIR = 0, 1, 2, 3

B_NK, B_KN = 0, 1

EXPORTED = ("gemm_tn_f16", "gemm_tn_f16_ex", "gemm_f16_scaled", "gemm_f16_padded",
            "gemm_padded_workspace_bytes", "gemm_query_config", "gemm_get_device_error",
            "gemm_minimum_stages", "gemm_probe_latencies", "gemm_probe_latencies_static",
            "gemm_status_string")


class GemmOptions(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("bn", ctypes.c_int), ("kstage", ctypes.c_int),
                ("max_ctas", ctypes.c_int), ("group_m", ctypes.c_int),
                ("timeout_ns", ctypes.c_uint64), ("inject", ctypes.c_int), ("katoms", ctypes.c_int),
                ("epi_warps", ctypes.c_int), ("b_layout", ctypes.c_int), ("acc_f16", ctypes.c_int),
                ("b_resident", ctypes.c_int), ("pdl", ctypes.c_int), ("wide", ctypes.c_int),
                ("small_m", ctypes.c_int), ("check", ctypes.c_int), ("split_k", ctypes.c_int),
                ("multicast", ctypes.c_int)]


class GemmConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("path", "bm", "bn", "bk", "kstage", "ctas", "group_m",
                                            "tiles", "smem_bytes", "tmem_cols", "katoms",
                                            "epi_warps", "b_resident", "pdl", "wide",
                                            "small_m", "split_k", "cluster")]


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def library_path() -> str:
    return _build.LIB


def _load() -> ctypes.CDLL:
    if not os.path.exists(_build.LIB):
        raise ImportError(f"{_build.LIB} is missing: build it with "
                          "`python -m multistage_smem_pipeline_gb300.build` (needs nvcc)")
    lib = ctypes.CDLL(_build.LIB)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.gemm_tn_f16.argtypes = [vp, vp, vp, i64, i64, i64, vp]
    lib.gemm_tn_f16.restype = i32
    lib.gemm_tn_f16_ex.argtypes = [vp, vp, vp, i64, i64, i64, ctypes.POINTER(GemmOptions), vp]
    lib.gemm_tn_f16_ex.restype = i32
    lib.gemm_f16_scaled.argtypes = [vp, vp, vp, vp, i64, i64, i64, ctypes.c_float, ctypes.c_float,
                                    i32, ctypes.POINTER(GemmOptions), vp]
    lib.gemm_f16_scaled.restype = i32
    lib.gemm_f16_padded.argtypes = [vp, vp, vp, vp, i64, i64, i64, ctypes.c_float, ctypes.c_float,
                                    i32, vp, ctypes.c_uint64, ctypes.POINTER(GemmOptions), vp]
    lib.gemm_f16_padded.restype = i32
    lib.gemm_padded_workspace_bytes.argtypes = [vp, vp, vp, vp, i64, i64, i64, ctypes.c_float, i32,
                                                ctypes.POINTER(ctypes.c_uint64)]
    lib.gemm_padded_workspace_bytes.restype = i32
    lib.gemm_query_config.argtypes = [i64, i64, i64, ctypes.POINTER(GemmOptions),
                                      ctypes.POINTER(GemmConfig)]
    lib.gemm_query_config.restype = i32
    lib.gemm_get_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.gemm_get_device_error.restype = i32
    lib.gemm_minimum_stages.argtypes = [i64, i64]
    lib.gemm_minimum_stages.restype = i64
    lib.gemm_probe_latencies.argtypes = [i32, i32, vp, i64, i32, ctypes.POINTER(ctypes.c_double),
                                         ctypes.POINTER(ctypes.c_double), vp]
    lib.gemm_probe_latencies.restype = i32
    lib.gemm_probe_latencies_static.argtypes = [i32, i32, i64, i32, ctypes.POINTER(ctypes.c_double),
                                                ctypes.POINTER(ctypes.c_double), vp]
    lib.gemm_probe_latencies_static.restype = i32
    lib.gemm_status_string.argtypes = [i32]
    lib.gemm_status_string.restype = ctypes.c_char_p
    return lib


LIB = _load()


def status_string(status: int) -> str:
    return LIB.gemm_status_string(int(status)).decode()


def _stream_handle(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _options(path=0, bn=0, kstage=0, max_ctas=0, group_m=0, timeout_ns=0, inject=0,
             katoms=0, epi_warps=0, b_layout=0, acc_f16=0, b_resident=0,
             pdl=0, wide=0, small_m=0, check=0, split_k=0, multicast=0) -> GemmOptions:
    return GemmOptions(int(path), int(bn), int(kstage), int(max_ctas), int(group_m),
                       int(timeout_ns), int(inject), int(katoms), int(epi_warps), int(b_layout),
                       int(acc_f16), int(b_resident), int(pdl), int(wide), int(small_m),
                       int(check), int(split_k), int(multicast))


def _check_operands(a: torch.Tensor, b: torch.Tensor, out):
    if a.dtype != torch.float16 or b.dtype != torch.float16:
        raise TypeError("A and B must be float16")
    if a.dim() != 2 or b.dim() != 2 or a.shape[1] != b.shape[1]:
        raise ValueError(f"A must be M x K and B N x K, got {tuple(a.shape)} and {tuple(b.shape)}")
    if not (a.is_cuda and b.is_cuda):
        raise ValueError("A and B must be CUDA tensors")
    if not (a.is_contiguous() and b.is_contiguous()):
        raise ValueError("A and B must be contiguous (row-major)")
    M, K = a.shape
    N = b.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=a.device)
    elif out.dtype != torch.float16 or tuple(out.shape) != (M, N) or not out.is_contiguous() \
            or out.device != a.device:
        raise ValueError("out must be a contiguous float16 M x N tensor on A's device")
    return M, N, K, out


def gemm_tn_f16(a: torch.Tensor, b: torch.Tensor, out: torch.Tensor | None = None,
                stream=None) -> torch.Tensor:
    """out = A @ B^T (fp16 in, fp32 accumulate, fp16 out) via the C-ABI, async on the stream."""
    M, N, K, out = _check_operands(a, b, out)
    with torch.cuda.device(a.device):
        rc = LIB.gemm_tn_f16(out.data_ptr(), a.data_ptr(), b.data_ptr(), M, N, K,
                             _stream_handle(stream))
    if rc != GEMM_OK:
        raise GemmError(rc, "gemm_tn_f16")
    return out


def gemm_tn_f16_ex(a: torch.Tensor, b: torch.Tensor, out: torch.Tensor | None = None, stream=None,
                   **opts) -> torch.Tensor:
    """gemm_tn_f16 with explicit options: path, bn, kstage, max_ctas, group_m, timeout_ns,
    inject, katoms, epi_warps, acc_f16, b_resident, pdl, wide, small_m, check, split_k,
    multicast (the fields of gemm_options_t)."""
    M, N, K, out = _check_operands(a, b, out)
    o = _options(**opts)
    with torch.cuda.device(a.device):
        rc = LIB.gemm_tn_f16_ex(out.data_ptr(), a.data_ptr(), b.data_ptr(), M, N, K,
                                ctypes.byref(o), _stream_handle(stream))
    if rc != GEMM_OK:
        raise GemmError(rc, "gemm_tn_f16_ex")
    return out


def _scaled_operands(a, b, c, out, b_layout: str, contiguous_what: str):
    """Checks the tensors of the scaled form; returns (M, N, K, kn, out)."""
    if b_layout not in ("kn", "nk"):
        raise ValueError("b_layout must be 'kn' or 'nk'")
    kn = b_layout == "kn"
    if a.dtype != torch.float16 or b.dtype != torch.float16:
        raise TypeError("A and B must be float16")
    if a.dim() != 2 or b.dim() != 2 or not (a.is_cuda and b.is_cuda):
        raise ValueError("A and B must be 2-D CUDA tensors")
    if not (a.is_contiguous() and b.is_contiguous()):
        raise ValueError("A and B must be contiguous (row-major)")
    M, K = a.shape
    if kn:
        if b.shape[0] != K:
            raise ValueError(f"B must be K x N, got {tuple(b.shape)}")
        N = b.shape[1]
    else:
        if b.shape[1] != K:
            raise ValueError(f"B must be N x K, got {tuple(b.shape)}")
        N = b.shape[0]
    if c is not None and (c.dtype != torch.float16 or tuple(c.shape) != (M, N)
                          or not c.is_contiguous() or c.device != a.device):
        raise ValueError("C must be a contiguous float16 M x N tensor on A's device")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=a.device)
    elif out.dtype != torch.float16 or tuple(out.shape) != (M, N) or not out.is_contiguous() \
            or out.device != a.device:
        raise ValueError(f"out must be a {contiguous_what} float16 M x N tensor on A's device")
    return M, N, K, kn, out


def gemm_f16_scaled(a: torch.Tensor, b: torch.Tensor, c: torch.Tensor | None = None,
                    alpha: float = 1.0, beta: float = 0.0, b_layout: str = "kn",
                    out: torch.Tensor | None = None, stream=None, **opts) -> torch.Tensor:
    """out = alpha * A @ op(B) + beta * C via the C-ABI (fp32 accumulate, fp16 out).

    b_layout "kn": B is K x N (out = alpha A B + beta C); "nk": B is N x K
    (out = alpha A B^T + beta C).  C is read only when beta != 0; passing
    out=c updates C in place."""
    M, N, K, kn, out = _scaled_operands(a, b, c, out, b_layout, "contiguous")
    o = _options(**opts)
    with torch.cuda.device(a.device):
        rc = LIB.gemm_f16_scaled(out.data_ptr(), c.data_ptr() if c is not None else None,
                                 a.data_ptr(), b.data_ptr(), M, N, K, float(alpha), float(beta),
                                 B_KN if kn else B_NK, ctypes.byref(o), _stream_handle(stream))
    if rc != GEMM_OK:
        raise GemmError(rc, "gemm_f16_scaled")
    return out


def padded_workspace_bytes(a: torch.Tensor, b: torch.Tensor, c: torch.Tensor | None,
                           out: torch.Tensor, beta: float = 0.0, b_layout: str = "nk") -> int:
    """Workspace bytes gemm_f16_padded needs for exactly these tensors."""
    M, N, K, kn, out = _scaled_operands(a, b, c, out, b_layout, "contiguous")
    n = ctypes.c_uint64(0)
    rc = LIB.gemm_padded_workspace_bytes(out.data_ptr(), c.data_ptr() if c is not None else None,
                                         a.data_ptr(), b.data_ptr(), M, N, K, float(beta),
                                         B_KN if kn else B_NK, ctypes.byref(n))
    if rc != GEMM_OK:
        raise GemmError(rc, "gemm_padded_workspace_bytes")
    return int(n.value)


def gemm_f16_padded(a: torch.Tensor, b: torch.Tensor, c: torch.Tensor | None = None,
                    alpha: float = 1.0, beta: float = 0.0, b_layout: str = "nk",
                    out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                    stream=None, **opts) -> torch.Tensor:
    """gemm_f16_scaled for any K and N (and any fp16-aligned tensors): operands
    whose rows are not 16-byte aligned are repacked into `workspace` (a uint8
    CUDA tensor; allocated here when None) before the GEMM kernel."""
    M, N, K, kn, out = _scaled_operands(a, b, c, out, b_layout, "contiguous")
    need = padded_workspace_bytes(a, b, c, out, beta, b_layout)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=a.device)
    elif workspace.dtype != torch.uint8 or not workspace.is_contiguous() \
            or workspace.device != a.device:
        raise ValueError("workspace must be a contiguous uint8 tensor on A's device")
    o = _options(**opts)
    with torch.cuda.device(a.device):
        rc = LIB.gemm_f16_padded(out.data_ptr(), c.data_ptr() if c is not None else None,
                                 a.data_ptr(), b.data_ptr(), M, N, K, float(alpha), float(beta),
                                 B_KN if kn else B_NK, workspace.data_ptr(), workspace.numel(),
                                 ctypes.byref(o), _stream_handle(stream))
    if rc != GEMM_OK:
        raise GemmError(rc, "gemm_f16_padded")
    return out


def gemm_tn_f16_from_host(a_host: torch.Tensor, b_host: torch.Tensor, device=None,
                          stream=None) -> torch.Tensor:
    """End-to-end call from host buffers: copy A and B (pinned host fp16) to the
    device, run the GEMM, copy D back into a pinned host tensor.  All on one
    stream; returns after D is on the host."""
    dev = torch.device(device or "cuda")
    s = stream or torch.cuda.current_stream(dev)
    with torch.cuda.stream(s):
        a = a_host.to(dev, non_blocking=True)
        b = b_host.to(dev, non_blocking=True)
        d = gemm_tn_f16(a, b, stream=s)
        d_host = torch.empty(d.shape, dtype=d.dtype, pin_memory=True)
        d_host.copy_(d, non_blocking=True)
    s.synchronize()
    return d_host


def get_device_error(stream=None) -> tuple[int, int]:
    """(status, raw word) of the stream's device error word; synchronises the stream and clears it."""
    raw = ctypes.c_uint32(0)
    rc = LIB.gemm_get_device_error(_stream_handle(stream), ctypes.byref(raw))
    return rc, int(raw.value)


def minimum_stages(copy_cycles: int, compute_cycles: int) -> int:
    return int(LIB.gemm_minimum_stages(int(copy_cycles), int(compute_cycles)))


def query_config(M: int, N: int, K: int, **opts) -> dict:
    o = _options(**opts)
    c = GemmConfig()
    rc = LIB.gemm_query_config(int(M), int(N), int(K), ctypes.byref(o), ctypes.byref(c))
    if rc != GEMM_OK:
        raise GemmError(rc, "gemm_query_config")
    return {n: getattr(c, n) for n, _ in GemmConfig._fields_}


def probe_latencies(bn: int = 256, ctas: int = 0, footprint_bytes: int = 1 << 30, reps: int = 64,
                    device=None) -> tuple[float, float]:
    """(copy_cycles, compute_cycles) measured on the device; see gemm_probe_latencies."""
    dev = torch.device(device or "cuda")
    scratch = torch.zeros(footprint_bytes // 2, dtype=torch.float16, device=dev)
    c = ctypes.c_double(0)
    m = ctypes.c_double(0)
    with torch.cuda.device(dev):
        rc = LIB.gemm_probe_latencies(int(bn), int(ctas), scratch.data_ptr(), int(footprint_bytes),
                                      int(reps), ctypes.byref(c), ctypes.byref(m),
                                      _stream_handle(None))
    if rc != GEMM_OK:
        raise GemmError(rc, "gemm_probe_latencies")
    return c.value, m.value


def probe_latencies_static(bn: int = 256, ctas: int = 0, footprint_bytes: int = 16 << 20,
                           reps: int = 64, device=None) -> tuple[float, float]:
    """(copy_cycles, compute_cycles) like probe_latencies, for callers that cannot
    allocate device memory: the copy probe loads from the library's own 16 MiB
    device array, so nothing is allocated here or in the library."""
    dev = torch.device(device or "cuda")
    c = ctypes.c_double(0)
    m = ctypes.c_double(0)
    with torch.cuda.device(dev):
        rc = LIB.gemm_probe_latencies_static(int(bn), int(ctas), int(footprint_bytes), int(reps),
                                             ctypes.byref(c), ctypes.byref(m),
                                             _stream_handle(None))
    if rc != GEMM_OK:
        raise GemmError(rc, "gemm_probe_latencies_static")
    return c.value, m.value
