"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module draws random numbers and rounds them to fp16; it holds none of the
GEMM's arithmetic.  Both sides receive the very same fp16 bit patterns.

Generator: splitmix64 in counter form (Steele, Lea & Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014): the i-th 64-bit output for seed
s is mix(s + (i + 1) * 0x9E3779B97F4A7C15) with the published mixing
constants; a uniform double in [0, 1) is its top 53 bits times 2^-53.  Normals
use the Box-Muller transform on pairs of uniforms.

Workloads (the GEMM shapes the pipeline is measured and checked on, with the
value distributions they are checked with):

=====  =======================  ===========================================
name   M x N x K                values (A and B iid, then fp16 round-nearest)
=====  =======================  ===========================================
c1     256 x 256 x 256          U[-1, 1]
c2     1024 x 1024 x 1024       uniform over {-1, 0, 1}
c3     4096 x 4096 x 4096       N(0, 1) * K^(-1/4) on each operand
c4     8192 x 8192 x 8192       U[-1, 1]
c5     128 x 14336 x 4096       A ~ N(0, 1), B ~ N(0, 0.02^2)
c6     81920 x 256 x 256        U[-1, 1] (the tall shape "cute(9)
                                multistage_gemm" times in its section 11;
                                the page does not state its values)
c7     8192 x 8192 x 8192       U[-1, 1]; the scaled NN form of "CUDA 算子笔记
                                2" (GEMM section): D = 1.5 A B - 0.5 C with
                                B K x N and C U[-1, 1]
c8     81920 x 256 x 256        U[-1, 1] with an fp16 accumulator: the shape
                                and the accumulator of the page's own
                                measurement ("cute(9)", section 11)
c9     8191 x 8191 x 8191       U[-1, 1]; K and N not multiples of 8, so the
                                rows are not 16-byte aligned: the general
                                shapes the padding wrapper of "CUDA 算子笔记
                                2" (GEMM section) serves
=====  =======================  ===========================================
"""
from __future__ import annotations

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Outputs start .. start+count-1 of the counter-form splitmix64 stream."""
    i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def uniform01(seed: int, count: int) -> np.ndarray:
    out = np.empty(count, dtype=np.float64)
    for s in range(0, count, _CHUNK):
        n = min(_CHUNK, count - s)
        out[s:s + n] = (splitmix64(seed, s, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    return out


def normal(seed: int, count: int) -> np.ndarray:
    """Standard normals by Box-Muller: uniforms 2i, 2i+1 give normals 2i, 2i+1."""
    pairs = (count + 1) // 2
    out = np.empty(2 * pairs, dtype=np.float64)
    for s in range(0, pairs, _CHUNK):
        n = min(_CHUNK, pairs - s)
        u = (splitmix64(seed, 2 * s, 2 * n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
        u1 = 1.0 - u[0::2]                     # (0, 1]: log is finite
        u2 = u[1::2]
        r = np.sqrt(-2.0 * np.log(u1))
        out[2 * s:2 * (s + n):2] = r * np.cos(2.0 * np.pi * u2)
        out[2 * s + 1:2 * (s + n):2] = r * np.sin(2.0 * np.pi * u2)
    return out[:count]


def to_fp16_bits(x: np.ndarray) -> np.ndarray:
    """Round doubles to fp16 (nearest, ties to even) and return the bit patterns."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def uniform_pm1(seed: int, shape) -> np.ndarray:
    n = int(np.prod(shape))
    return to_fp16_bits(uniform01(seed, n) * 2.0 - 1.0).reshape(shape)


def ternary(seed: int, shape) -> np.ndarray:
    """-1, 0, 1 with probability 1/3 each: floor(3u) - 1."""
    n = int(np.prod(shape))
    return to_fp16_bits(np.floor(uniform01(seed, n) * 3.0) - 1.0).reshape(shape)


def gaussian(seed: int, shape, std: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    return to_fp16_bits(normal(seed, n) * std).reshape(shape)


WORKLOADS = {
    "c1": dict(M=256, N=256, K=256, kind="uniform"),
    "c2": dict(M=1024, N=1024, K=1024, kind="ternary"),
    "c3": dict(M=4096, N=4096, K=4096, kind="normal_k_quarter"),
    "c4": dict(M=8192, N=8192, K=8192, kind="uniform"),
    "c5": dict(M=128, N=14336, K=4096, kind="skinny"),
    "c6": dict(M=81920, N=256, K=256, kind="uniform"),
    "c7": dict(M=8192, N=8192, K=8192, kind="uniform", b_kn=True, alpha=1.5, beta=-0.5),
    "c8": dict(M=81920, N=256, K=256, kind="uniform", acc_f16=True),
    "c9": dict(M=8191, N=8191, K=8191, kind="uniform", padded=True),
}
WORKLOAD_NAMES = {
    "c1": "gemm_tn_f16 256x256x256 U[-1,1]",
    "c2": "gemm_tn_f16 1024x1024x1024 {-1,0,1}",
    "c3": "gemm_tn_f16 4096x4096x4096 N(0,1)*K^-1/4",
    "c4": "gemm_tn_f16 8192x8192x8192 U[-1,1]",
    "c5": "gemm_tn_f16 skinny M=128 N=14336 K=4096 A~N(0,1) B~N(0,0.02)",
    "c6": "gemm_tn_f16 tall M=81920 N=256 K=256 U[-1,1]",
    "c7": "gemm_f16_scaled NN 8192x8192x8192 D=1.5*A*B-0.5*C U[-1,1]",
    "c8": "gemm_tn_f16 tall M=81920 N=256 K=256 U[-1,1], fp16 accumulator",
    "c9": "gemm_f16_padded 8191x8191x8191 U[-1,1] (rows not 16-byte aligned)",
}


def seeds(tag: str) -> tuple[int, int, int]:
    """(seed_A, seed_B, seed_samples) for a workload tag c1..c9."""
    c = int(tag[1:])
    return 1000 + c, 2000 + c, 3000 + c


def make_operands(kind: str, M: int, N: int, K: int, seed_a: int, seed_b: int):
    """fp16 bit arrays A (M x K) and B (N x K) for one value distribution."""
    if kind == "uniform":
        return uniform_pm1(seed_a, (M, K)), uniform_pm1(seed_b, (N, K))
    if kind == "ternary":
        return ternary(seed_a, (M, K)), ternary(seed_b, (N, K))
    if kind == "normal_k_quarter":
        s = float(K) ** -0.25
        return gaussian(seed_a, (M, K), s), gaussian(seed_b, (N, K), s)
    if kind == "skinny":
        return gaussian(seed_a, (M, K), 1.0), gaussian(seed_b, (N, K), 0.02)
    raise ValueError(f"unknown value distribution {kind!r}")


def workload(tag: str):
    """(A_bits, B_bits, spec) for a workload tag c1..c9.  B is N x K, or K x N
    where spec["b_kn"] is set."""
    spec = WORKLOADS[tag]
    sa, sb, _ = seeds(tag)
    if spec.get("b_kn"):
        if spec["kind"] != "uniform":
            raise ValueError("K x N operands are generated for the uniform distribution only")
        return uniform_pm1(sa, (spec["M"], spec["K"])), uniform_pm1(sb, (spec["K"], spec["N"])), spec
    a, b = make_operands(spec["kind"], spec["M"], spec["N"], spec["K"], sa, sb)
    return a, b, spec


def workload_c(tag: str):
    """C (M x N fp16 bits) of a scaled workload (seed 4000 + c)."""
    spec = WORKLOADS[tag]
    return uniform_pm1(4000 + int(tag[1:]), (spec["M"], spec["N"]))


def sample_coords(seed: int, M: int, N: int, count: int = 4096, bm: int = 128, bn: int = 256):
    """`count` seeded (row, col) pairs plus structural points: the four corners
    and the rows/cols on either side of the first tile seams."""
    u = uniform01(seed, 2 * count)
    rows = np.minimum((u[0::2] * M).astype(np.int64), M - 1)
    cols = np.minimum((u[1::2] * N).astype(np.int64), N - 1)
    rs = sorted({0, M - 1} | {x for x in (bm - 1, bm, 2 * bm - 1, 2 * bm) if x < M})
    cs = sorted({0, N - 1} | {x for x in (bn - 1, bn, 2 * bn - 1, 2 * bn, bn // 2 - 1, bn // 2) if x < N})
    er = np.array([r for r in rs for _ in cs], dtype=np.int64)
    ec = np.array([c for _ in rs for c in cs], dtype=np.int64)
    return np.concatenate([rows, er]), np.concatenate([cols, ec])
