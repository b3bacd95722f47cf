"""Pins for the CPU oracle, checked against things other than the oracle itself.

* converters: numpy's own binary16 conversions (exhaustive / constructed ties);
* the GEMM: exact integer arithmetic on tiny and structured inputs, the
  identity and rank-1 closed forms, and an independent integer rounding of the
  exact rational result;
* the stage helper: the worked examples of "第 6 课：Shared Memory 布局与异步流水"
  (section 4 and its exercise), stored in tests/golden/minimum_stages.txt.

Every plausible slip -- a dropped term, a sign, a transposed operand, a wrong
index, double rounding, a wrong tie rule -- fails at least one test here.
"""
import os

import numpy as np
import pytest

import oracle
from multistage_smem_pipeline_gb300 import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------- converters
def test_half_to_double_exhaustive_matches_numpy():
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.half_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_double_to_half_roundtrip_exhaustive():
    bits = np.arange(65536, dtype=np.uint16)
    vals = bits.view(np.float16).astype(np.float64)
    back = oracle.double_to_half(vals)
    finite = ~np.isnan(vals)
    assert np.array_equal(back[finite], bits[finite])
    assert np.all(np.isnan(back[~finite].view(np.float16)))


def _positive_finite_halves():
    b = np.arange(0, 0x7C00, dtype=np.uint16)        # +0 .. 65504
    return b.view(np.float16).astype(np.float64)


def test_double_to_half_ties_go_to_even():
    v = _positive_finite_halves()
    mids = (v[:-1] + v[1:]) / 2.0                    # exact in double
    ours = oracle.double_to_half(mids)
    ref = mids.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)
    # the winner of every tie has an even last fraction bit
    assert np.all(ours & 1 == 0)
    # just above / below a midpoint goes to the nearer neighbour
    up = oracle.double_to_half(np.nextafter(mids, np.inf))
    dn = oracle.double_to_half(np.nextafter(mids, -np.inf))
    lo = np.arange(0, 0x7BFF, dtype=np.uint16)
    assert np.array_equal(up, lo + 1)
    assert np.array_equal(dn, lo)


def test_double_to_half_special_edges():
    f = lambda x: int(oracle.double_to_half([x])[0])
    assert f(65504.0) == 0x7BFF
    assert f(65519.999) == 0x7BFF
    assert f(65520.0) == 0x7C00                      # tie to even = +inf
    assert f(-65520.0) == 0xFC00
    assert f(1e300) == 0x7C00
    assert f(float("inf")) == 0x7C00 and f(float("-inf")) == 0xFC00
    assert f(2.0 ** -25) == 0x0000                   # tie between 0 and 2^-24 -> 0
    assert f(np.nextafter(2.0 ** -25, 1.0)) == 0x0001
    assert f(3 * 2.0 ** -25) == 0x0002               # tie between 1 and 2 ulps -> 2
    assert f(-0.0) == 0x8000
    assert f(2.0 ** -14 - 2.0 ** -25) == 0x0400      # rounds up into the first normal
    assert (f(float("nan")) & 0x7C00) == 0x7C00 and (f(float("nan")) & 0x3FF) != 0


def test_double_to_half_random_matches_numpy():
    rng = np.random.default_rng(7)
    mant = rng.uniform(-1, 1, 200_000)
    expo = rng.integers(-30, 18, 200_000)
    x = np.ldexp(mant, expo)
    assert np.array_equal(oracle.double_to_half(x), x.astype(np.float16).view(np.uint16))


# --------------------------------------------------------------------------- exact references
def _exact_half_of_scaled_int(s: int) -> int:
    """fp16 bits of s * 2^-48 (s a Python int), rounded to nearest-even with
    integer arithmetic only -- independent of the oracle's converter."""
    neg = s < 0
    a = -s if neg else s
    if a == 0:
        return 0x8000 if neg else 0
    e = a.bit_length() - 1 - 48                   # 2^e <= value < 2^(e+1)
    q_exp = max(e, -14) - 10                      # fp16 spacing 2^q_exp
    Q = 1 << (q_exp + 48)                         # q_exp >= -24, so Q is an integer
    n, rem = divmod(a, Q)
    if 2 * rem > Q or (2 * rem == Q and n % 2 == 1):
        n += 1
    mag = float(n) * 2.0 ** q_exp                 # exactly representable (or overflow)
    bits = 0x7C00 if mag > 65504.0 else int(np.float16(mag).view(np.uint16))
    return bits | (0x8000 if neg else 0)


def _exact_reference(a_bits, b_bits):
    """D via exact integers: every fp16 value is an integer multiple of 2^-24."""
    a = (a_bits.view(np.float16).astype(np.float64) * 2.0 ** 24).astype(np.int64)
    b = (b_bits.view(np.float16).astype(np.float64) * 2.0 ** 24).astype(np.int64)
    M, N = a.shape[0], b.shape[0]
    out = np.zeros((M, N), dtype=np.uint16)
    for i in range(M):
        for j in range(N):
            s = sum(int(x) * int(y) for x, y in zip(a[i], b[j]))
            out[i, j] = _exact_half_of_scaled_int(s)
    return out


def _small_int_halves(rng, shape, lim=4):
    return rng.integers(-lim, lim + 1, size=shape).astype(np.float16).view(np.uint16)


SIZES = [1, 2, 3, 5, 8, 16, 17]


@pytest.mark.parametrize("M", SIZES)
def test_brute_force_small_integers(M):
    rng = np.random.default_rng(100 + M)
    for N in SIZES:
        for K in SIZES:
            a = _small_int_halves(rng, (M, K))
            b = _small_int_halves(rng, (N, K))
            ai = a.view(np.float16).astype(np.int64)
            bi = b.view(np.float16).astype(np.int64)
            want = (ai @ bi.T).astype(np.float16).view(np.uint16)   # |D| <= 272: exact
            got = oracle.gemm_tn(a, b, threads=2)
            assert np.array_equal(got, want), (M, N, K)


@pytest.mark.parametrize("shape", [(3, 5, 7), (7, 2, 33), (9, 11, 64), (1, 13, 130)])
def test_random_fp16_against_exact_rational(shape):
    M, N, K = shape
    rng = np.random.default_rng(sum(shape))
    a = rng.uniform(-1, 1, (M, K)).astype(np.float16).view(np.uint16)
    b = (rng.uniform(-1, 1, (N, K)) * np.ldexp(1.0, rng.integers(-12, 4, (N, K)))).astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.gemm_tn(a, b), _exact_reference(a, b))


@pytest.mark.parametrize("order", [(0, 1, 2), (2, 1, 0), (1, 2, 0)])
def test_accumulation_is_wider_than_float(order):
    # exact sum 1 + 2^-11 + 2^-25 lies just above the fp16 tie between 1 and
    # 1 + 2^-10, so it must round up.  A float accumulator (or a detour through
    # float before the fp16 rounding) loses the 2^-25 and lands on the tie,
    # which goes to the even neighbour 1.0 instead.
    a = np.array([1.0, 2.0 ** -11, 2.0 ** -12])[list(order)]
    b = np.array([1.0, 1.0, 2.0 ** -13])[list(order)]
    a = a.astype(np.float16).view(np.uint16)[None, :]
    b = b.astype(np.float16).view(np.uint16)[None, :]
    assert int(oracle.gemm_tn(a, b)[0, 0]) == 0x3C01
    assert int(_exact_reference(a, b)[0, 0]) == 0x3C01
    # the scaled form accumulates the same way (alpha = 1, beta = 0), in both layouts
    assert int(oracle.gemm_scaled(a, b, None, 1.0, 0.0, False)[0, 0]) == 0x3C01
    assert int(oracle.gemm_scaled(a, np.ascontiguousarray(b.T), None, 1.0, 0.0, True)[0, 0]) == 0x3C01


def test_subnormal_and_overflow_results():
    # products far below the normal range and sums beyond 65504
    a = np.full((2, 4), np.float16(2.0 ** -10)).view(np.uint16)
    b = np.full((3, 4), np.float16(2.0 ** -13)).view(np.uint16)
    assert np.array_equal(oracle.gemm_tn(a, b), _exact_reference(a, b))     # 4*2^-23 = 2^-21
    big = np.full((1, 8), np.float16(256.0)).view(np.uint16)
    d = oracle.gemm_tn(big, big)                                             # 8*65536 -> inf
    assert int(d[0, 0]) == 0x7C00


def test_identity_closed_forms():
    rng = np.random.default_rng(3)
    K = 40
    eye = np.eye(K).astype(np.float16).view(np.uint16)
    b = rng.standard_normal((23, K)).astype(np.float16).view(np.uint16)
    a = rng.standard_normal((31, K)).astype(np.float16).view(np.uint16)
    # A = I: D[i][j] = B[j][i], i.e. D = B^T
    assert np.array_equal(oracle.gemm_tn(eye, b), b.T)
    # B = I: D = A
    assert np.array_equal(oracle.gemm_tn(a, eye), a)


def test_rank_one_closed_form():
    rng = np.random.default_rng(11)
    M, N, K = 6, 9, 14
    u = rng.integers(-3, 4, M)
    v = rng.integers(-3, 4, N)
    x = rng.integers(-3, 4, K)
    y = rng.integers(-3, 4, K)
    a = np.outer(u, x).astype(np.float16).view(np.uint16)
    b = np.outer(v, y).astype(np.float16).view(np.uint16)
    want = (np.outer(u, v) * int(x @ y)).astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.gemm_tn(a, b), want)


@pytest.mark.parametrize("K", [1, 64, 1024])
def test_constant_closed_form(K):
    a = np.full((5, K), np.float16(0.75)).view(np.uint16)
    b = np.full((4, K), np.float16(-0.5)).view(np.uint16)
    want = np.float16(K * 0.75 * -0.5).view(np.uint16)
    assert np.all(oracle.gemm_tn(a, b) == want)


def test_ternary_exactness_case_equals_integer_gemm():
    a = synthetic.ternary(5, (64, 1024))
    b = synthetic.ternary(6, (48, 1024))
    ai = a.view(np.float16).astype(np.int64)
    bi = b.view(np.float16).astype(np.int64)
    want = (ai @ bi.T).astype(np.float16).view(np.uint16)       # |D| <= 1024: exact
    assert np.array_equal(oracle.gemm_tn(a, b), want)


def test_sampled_equals_full_and_thread_count_is_irrelevant():
    a = synthetic.uniform_pm1(1, (37, 96))
    b = synthetic.uniform_pm1(2, (29, 96))
    full1 = oracle.gemm_tn(a, b, threads=1)
    full5 = oracle.gemm_tn(a, b, threads=5)
    assert np.array_equal(full1, full5)
    rows, cols = synthetic.sample_coords(9, 37, 29, count=200, bm=8, bn=8)
    assert np.array_equal(oracle.gemm_tn_sampled(a, b, rows, cols), full1[rows, cols])


def test_empty_shapes():
    a = np.zeros((0, 8), np.uint16)
    b = np.zeros((3, 8), np.uint16)
    assert oracle.gemm_tn(a, b).shape == (0, 3)
    a = np.zeros((2, 0), np.uint16)
    b = np.zeros((3, 0), np.uint16)
    assert np.all(oracle.gemm_tn(a, b) == 0)      # empty sum is +0


def test_normal_scaled_case_is_unit_variance():
    # weak statistical check of the 4096^3 recipe at a reduced M, N
    K = 4096
    a, b = synthetic.make_operands("normal_k_quarter", 48, 40, K, 11, 12)
    d = oracle.gemm_tn(a, b).view(np.float16).astype(np.float64)
    assert abs(d.mean()) < 0.1 and 0.85 < d.var() < 1.15


# --------------------------------------------------------------------------- stage helper
def _golden_stages():
    rows = []
    with open(os.path.join(GOLDEN, "minimum_stages.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(tuple(int(t) for t in line.split()))
    return rows


def test_minimum_stages_matches_page_examples():
    rows = _golden_stages()
    assert len(rows) == 3
    for copy, compute, stages in rows:
        assert oracle.minimum_stages(copy, compute) == stages


@pytest.mark.parametrize("copy,compute,want", [
    (240, 120, 3), (241, 120, 4), (119, 120, 2), (1, 1, 2), (10**12, 1, 10**12 + 1),
    (0, 120, -1), (120, 0, -1), (-5, 3, -1), (3, -5, -1)])
def test_minimum_stages_boundaries(copy, compute, want):
    assert oracle.minimum_stages(copy, compute) == want


# --------------------------------------------------------------------------- generator
def test_splitmix64_published_vector():
    # first outputs of splitmix64 seeded with 1234567 (the generator's reference test values)
    want = [6457827717110365317, 3203168211198807973, 9817491932198370423,
            4593380528125082431, 16408922859458223821]
    assert [int(x) for x in synthetic.splitmix64(1234567, 0, 5)] == want


def test_generators_are_seeded_and_in_range():
    a1 = synthetic.uniform_pm1(42, (64, 64))
    a2 = synthetic.uniform_pm1(42, (64, 64))
    assert np.array_equal(a1, a2)
    v = a1.view(np.float16).astype(np.float64)
    assert v.min() >= -1 and v.max() <= 1 and abs(v.mean()) < 0.05
    t = synthetic.ternary(1, (100_000,)).view(np.float16).astype(np.float64)
    assert set(np.unique(t)) == {-1.0, 0.0, 1.0}
    n = synthetic.normal(3, 200_001)
    assert abs(n.mean()) < 0.01 and abs(n.std() - 1) < 0.01


# --------------------------------------------------------------------------- scaled form
# D = fp16(alpha * A op(B) + beta * C), "CUDA 算子笔记 2" (GEMM section):
# C = alpha A B + beta C, fp16 matrices, fp32 alpha and beta, B K x N (NN).
from fractions import Fraction  # noqa: E402


def _fraction_to_half_bits(x: Fraction) -> int:
    """Round an exact rational to binary16, nearest-even, by exact rational
    arithmetic (no floating point on the way)."""
    neg = x < 0
    a = -x if neg else x
    if a == 0:
        return 0x8000 if neg else 0
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    q = Fraction(2) ** (max(e, -14) - 10)           # binary16 spacing at a
    n, rem = divmod(a, q)
    half = q / 2
    if rem > half or (rem == half and n % 2 == 1):
        n += 1
    mag = n * q
    if mag > 65504:
        bits = 0x7C00
    else:
        bits = int(np.float16(float(mag)).view(np.uint16))   # exactly representable
    return bits | (0x8000 if neg else 0)


def _exact_scaled(a_bits, b_bits, c_bits, alpha, beta, b_kn):
    a = a_bits.view(np.float16).astype(np.float64)
    b = b_bits.view(np.float16).astype(np.float64)
    if not b_kn:
        b = b.T
    M, K = a.shape
    N = b.shape[1]
    al, be = Fraction(float(np.float32(alpha))), Fraction(float(np.float32(beta)))
    c = c_bits.view(np.float16).astype(np.float64) if c_bits is not None else None
    out = np.zeros((M, N), dtype=np.uint16)
    for i in range(M):
        for j in range(N):
            s = sum(Fraction(a[i, k]) * Fraction(b[k, j]) for k in range(K))
            v = al * s + (be * Fraction(c[i, j]) if be != 0 else 0)
            out[i, j] = _fraction_to_half_bits(v)
    return out


@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (0.5, -2.0), (-0.25, 1.0), (2.0, 0.75)])
@pytest.mark.parametrize("b_kn", [False, True])
def test_scaled_small_integers_exact(alpha, beta, b_kn):
    rng = np.random.default_rng(17)
    M, N, K = 7, 12, 9
    ai = rng.integers(-3, 4, (M, K))
    bi = rng.integers(-3, 4, (K, N))
    ci = rng.integers(-50, 51, (M, N))
    a = ai.astype(np.float16).view(np.uint16)
    b = (bi if b_kn else bi.T).astype(np.float16).view(np.uint16)
    c = ci.astype(np.float16).view(np.uint16)
    want = (alpha * (ai @ bi) + beta * ci).astype(np.float16).view(np.uint16)  # exact dyadics
    assert np.array_equal(oracle.gemm_scaled(a, b, c, alpha, beta, b_kn), want)


@pytest.mark.parametrize("b_kn", [False, True])
def test_scaled_random_against_exact_rational(b_kn):
    rng = np.random.default_rng(23 + b_kn)
    M, N, K = 5, 6, 40
    a = rng.uniform(-1, 1, (M, K)).astype(np.float16).view(np.uint16)
    b = rng.uniform(-1, 1, (K, N) if b_kn else (N, K)).astype(np.float16).view(np.uint16)
    c = rng.uniform(-4, 4, (M, N)).astype(np.float16).view(np.uint16)
    for alpha, beta in [(1.3, -0.7), (-0.01171875, 3.25), (0.1, 0.9)]:
        got = oracle.gemm_scaled(a, b, c, alpha, beta, b_kn)
        assert np.array_equal(got, _exact_scaled(a, b, c, alpha, beta, b_kn)), (alpha, beta)


def test_scaled_special_cases():
    rng = np.random.default_rng(29)
    M, N, K = 9, 16, 24
    a = rng.standard_normal((M, K)).astype(np.float16).view(np.uint16)
    b_kn = rng.standard_normal((K, N)).astype(np.float16).view(np.uint16)
    c = rng.standard_normal((M, N)).astype(np.float16).view(np.uint16)
    # alpha = 0, beta = 1: D is C, bit for bit
    assert np.array_equal(oracle.gemm_scaled(a, b_kn, c, 0.0, 1.0, True), c)
    # beta = 0: C is never read -- NaN in C, or no C at all, changes nothing
    c_nan = np.full((M, N), 0x7E00, np.uint16)
    d0 = oracle.gemm_scaled(a, b_kn, c_nan, 1.5, 0.0, True)
    assert np.array_equal(d0, oracle.gemm_scaled(a, b_kn, None, 1.5, 0.0, True))
    assert not np.isnan(d0.view(np.float16)).any()
    # NN on B equals TN on B's transpose, and alpha = 1, beta = 0 is the plain product
    b_nk = np.ascontiguousarray(b_kn.T)
    assert np.array_equal(oracle.gemm_scaled(a, b_kn, c, 0.8, -0.3, True),
                          oracle.gemm_scaled(a, b_nk, c, 0.8, -0.3, False))
    assert np.array_equal(oracle.gemm_scaled(a, b_nk, None, 1.0, 0.0, False),
                          oracle.gemm_tn(a, b_nk))


# --------------------------------------------------------------------------- fp16 accumulation
# "cute(9) multistage_gemm": its MMA atom accumulates in fp16, one rounding per
# 16-deep K slice.
def _f16acc_reference(a_bits, b_bits):
    """The slice-by-slice rounding written with exact rationals."""
    a = a_bits.view(np.float16).astype(np.float64)
    b = b_bits.view(np.float16).astype(np.float64)
    M, K = a.shape
    N = b.shape[0]
    out = np.zeros((M, N), dtype=np.uint16)
    for i in range(M):
        for j in range(N):
            acc = Fraction(0)
            for k0 in range(0, K, 16):
                s = acc + sum(Fraction(a[i, k]) * Fraction(b[j, k]) for k in range(k0, min(K, k0 + 16)))
                bits = _fraction_to_half_bits(s)
                acc = Fraction(float(np.uint16(bits).view(np.float16)))
            out[i, j] = _fraction_to_half_bits(acc)
    return out


def test_f16acc_loses_what_an_fp16_accumulator_loses():
    # slice 1 sums to 2048; slices 2 and 3 each add 1.  In fp16, 2049 is a tie
    # between 2048 and 2050 and goes to the even 2048, so each added 1 is lost
    # and D = 2048, where the exactly summed product is 2050.
    K = 48
    a = np.zeros((1, K)); b = np.zeros((1, K))
    a[0, :16] = 128.0; b[0, :16] = 1.0          # 16 * 128 = 2048
    a[0, 16] = 1.0; b[0, 16] = 1.0              # + 1 in slice 2
    a[0, 32] = 1.0; b[0, 32] = 1.0              # + 1 in slice 3
    ah = a.astype(np.float16).view(np.uint16); bh = b.astype(np.float16).view(np.uint16)
    assert float(oracle.gemm_tn_f16acc(ah, bh).view(np.float16)[0, 0]) == 2048.0
    assert float(oracle.gemm_tn(ah, bh).view(np.float16)[0, 0]) == 2050.0


def test_f16acc_single_slice_is_one_rounding():
    # K <= 16: one slice, so fp16 accumulation is the plain product, rounded once
    rng = np.random.default_rng(41)
    for K in (1, 8, 16):
        a = rng.uniform(-1, 1, (6, K)).astype(np.float16).view(np.uint16)
        b = rng.uniform(-1, 1, (5, K)).astype(np.float16).view(np.uint16)
        assert np.array_equal(oracle.gemm_tn_f16acc(a, b), oracle.gemm_tn(a, b))


def test_f16acc_integer_sums_are_exact():
    # {-1,0,1} at K = 1024: every partial sum is an integer of magnitude <= 1024,
    # exact in fp16, so slice-wise rounding changes nothing
    a = synthetic.ternary(51, (24, 1024))
    b = synthetic.ternary(52, (20, 1024))
    ai = a.view(np.float16).astype(np.int64); bi = b.view(np.float16).astype(np.int64)
    assert np.array_equal(oracle.gemm_tn_f16acc(a, b), (ai @ bi.T).astype(np.float16).view(np.uint16))


@pytest.mark.parametrize("K", [17, 40, 100])
def test_f16acc_random_against_exact_slices(K):
    rng = np.random.default_rng(K)
    a = rng.uniform(-2, 2, (4, K)).astype(np.float16).view(np.uint16)
    b = rng.uniform(-2, 2, (3, K)).astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.gemm_tn_f16acc(a, b), _f16acc_reference(a, b))
