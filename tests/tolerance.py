"""Element-wise comparison of the GPU result with the oracle.

Bound per element (fp32 accumulation vs the oracle's exact-then-round):
    |D_gpu - D_ref| <= 2e-3 * sqrt(K) * max|A| * max|B| + ulp(D_ref)
where ulp(r) is the fp16 spacing at |r| (2^(max(e, -14) - 10) for
2^e <= |r| < 2^(e+1)).  The first term bounds the fp32 rounding of K
accumulated products with room to spare (each product is exact in fp32; the
running sum rounds at 2^-24 relative), the second the two sides rounding to
fp16 on either side of a tie.  Integer-valued inputs whose partial sums stay
exact in fp32 ({-1, 0, 1} at K = 1024) must match bit for bit instead.
"""
import numpy as np


def fp16_ulp(r: np.ndarray) -> np.ndarray:
    a = np.abs(r.astype(np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -14)))
    return np.exp2(e - 10)


def tolerance(ref_bits: np.ndarray, K: int, amax: float, bmax: float) -> np.ndarray:
    r = ref_bits.view(np.float16).astype(np.float64)
    return 2e-3 * np.sqrt(max(K, 1)) * amax * bmax + fp16_ulp(r)


def compare(got_bits: np.ndarray, ref_bits: np.ndarray, K: int, a_bits: np.ndarray,
            b_bits: np.ndarray) -> dict:
    """Returns stats; 'bad' counts elements outside the bound (NaN-aware)."""
    g = got_bits.view(np.float16).astype(np.float64)
    r = ref_bits.view(np.float16).astype(np.float64)
    amax = float(np.abs(a_bits.view(np.float16).astype(np.float64)).max()) if a_bits.size else 0.0
    bmax = float(np.abs(b_bits.view(np.float16).astype(np.float64)).max()) if b_bits.size else 0.0
    tol = tolerance(ref_bits, K, amax, bmax)
    both_nan = np.isnan(g) & np.isnan(r)
    err = np.where(both_nan, 0.0, np.abs(g - r))
    err = np.where(np.isnan(err), np.inf, err)
    bad = int(np.count_nonzero(err > tol))
    ulps = np.abs(got_bits.astype(np.int64) - ref_bits.astype(np.int64))
    return {"bad": bad, "max_err": float(err.max()) if err.size else 0.0,
            "max_ulps": int(ulps.max()) if ulps.size else 0,
            "exact_frac": float(np.mean(got_bits == ref_bits)) if got_bits.size else 1.0,
            "n": int(got_bits.size)}


# Latency probes report cycle counts measured on a live GPU, so two
# measurements of the same quantity agree only to within run-to-run noise.
# Relative bounds used wherever two probe results are compared: the copy
# latency (memory system, shared by all SMs) varies more than the MMA time.
PROBE_REL_TOL = {"copy": 0.25, "compute": 0.05}


def probes_agree(a: tuple, b: tuple) -> bool:
    """(copy_cycles, compute_cycles) pairs within PROBE_REL_TOL of each other."""
    (c1, m1), (c2, m2) = a, b
    return (abs(c1 - c2) <= PROBE_REL_TOL["copy"] * max(c1, c2)
            and abs(m1 - m2) <= PROBE_REL_TOL["compute"] * max(m1, m2))


def compare_scaled(got_bits, ref_bits, K, a_bits, b_bits, c_bits, alpha, beta) -> dict:
    """compare() for D = alpha * A op(B) + beta * C: the product term's bound
    scales with |alpha|, and beta * C adds fp32 rounding of its own
    (2^-20 |beta| max|C| is several fp32 ulps)."""
    g = got_bits.view(np.float16).astype(np.float64)
    r = ref_bits.view(np.float16).astype(np.float64)
    amax = float(np.abs(a_bits.view(np.float16).astype(np.float64)).max()) if a_bits.size else 0.0
    bmax = float(np.abs(b_bits.view(np.float16).astype(np.float64)).max()) if b_bits.size else 0.0
    cmax = 0.0
    if c_bits is not None and c_bits.size and beta != 0:
        cmax = float(np.abs(c_bits.view(np.float16).astype(np.float64)).max())
    tol = (2e-3 * np.sqrt(max(K, 1)) * abs(alpha) * amax * bmax + 2.0 ** -20 * abs(beta) * cmax
           + fp16_ulp(r))
    err = np.abs(g - r)
    err = np.where(np.isnan(g) & np.isnan(r), 0.0, err)
    err = np.where(np.isnan(err), np.inf, err)
    return {"bad": int(np.count_nonzero(err > tol)), "max_err": float(err.max()) if err.size else 0.0,
            "exact_frac": float(np.mean(got_bits == ref_bits)) if got_bits.size else 1.0,
            "n": int(got_bits.size)}
