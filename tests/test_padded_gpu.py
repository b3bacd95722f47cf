"""GPU parity of the padded entry gemm_f16_padded -- the general shapes of the
host wrapper in "CUDA 算子笔记 2" (GEMM section): K and N not multiples of 8,
operands at any fp16 alignment -- against the oracle, through the C-ABI.

Each misaligned operand is repacked by a copy kernel, so the cases below are
chosen to reach every branch of those copies: rows that start 16-, 4- and
2-byte aligned (odd K or N makes consecutive rows alternate), rows shorter
than one 8-element chunk, ragged last chunks, and each operand misaligned on
its own."""
import numpy as np
import pytest
import torch

import oracle
from multistage_smem_pipeline_gb300 import synthetic
from tolerance import compare, compare_scaled, fp16_ulp

pytestmark = pytest.mark.gpu
SQUARE, PAIR = 1, 3


@pytest.fixture(scope="module")
def lib(gpu):
    from multistage_smem_pipeline_gb300 import binding
    return binding


def _placed(bits, gpu, off=0):
    """A contiguous CUDA tensor holding `bits` whose address is 2*off bytes
    past a 16-byte boundary (off in 0..7)."""
    flat = np.ascontiguousarray(bits).reshape(-1).view(np.float16)
    store = torch.zeros(flat.size + 8, dtype=torch.float16, device=gpu)
    assert store.data_ptr() % 16 == 0
    t = store[off:off + flat.size]
    t.copy_(torch.from_numpy(flat).to(gpu))
    t = t.view(bits.shape)
    assert flat.size == 0 or t.data_ptr() % 16 == 2 * off  # an empty tensor's address is 0
    return t


def _empty(shape, gpu, off=0):
    n = int(np.prod(shape))
    store = torch.empty(n + 8, dtype=torch.float16, device=gpu)
    return store[off:off + n].view(shape)


def _operands(M, N, K, kn, seed):
    a = synthetic.uniform_pm1(seed, (M, K))
    b = synthetic.uniform_pm1(seed + 1, (K, N) if kn else (N, K))
    c = synthetic.uniform_pm1(seed + 2, (M, N))
    return a, b, c


def _run(lib, gpu, a, b, c, alpha, beta, kn, offs=(0, 0, 0, 0), in_place=False, **opts):
    """offs: element offsets of (A, B, C, D) from a 16-byte boundary."""
    oa, ob, oc, od = offs
    ta, tb = _placed(a, gpu, oa), _placed(b, gpu, ob)
    tc = _placed(c, gpu, oc) if c is not None else None
    out = tc if in_place else _empty((a.shape[0], c.shape[1] if c is not None else
                                      (b.shape[1] if kn else b.shape[0])), gpu, od)
    d = lib.gemm_f16_padded(ta, tb, tc, alpha, beta, "kn" if kn else "nk", out=out, **opts)
    torch.cuda.synchronize()
    status, raw = lib.get_device_error()
    assert status == 0, f"device error word {raw:#x}"
    return d.cpu().numpy().view(np.uint16)


def _check(got, a, b, c, alpha, beta, kn):
    ref = oracle.gemm_scaled(a, b, c, alpha, beta, kn)
    st = compare_scaled(got, ref, a.shape[1], a, b, c, alpha, beta)
    assert st["bad"] == 0, st
    return st


RAGGED = [(1, 1, 1), (5, 3, 7), (7, 13, 5), (130, 257, 123), (300, 129, 65), (257, 263, 1031),
          (64, 1001, 9), (129, 9, 300),
          # rows of 127 / 128+ elements: either side of the switch from the
          # chunk-per-thread copies to the warp-per-row ones
          (300, 128, 127), (130, 129, 129), (33, 2049, 4097)]


@pytest.mark.parametrize("kn", [False, True])
@pytest.mark.parametrize("M,N,K", RAGGED)
def test_padded_ragged_shapes(lib, gpu, kn, M, N, K):
    a, b, c = _operands(M, N, K, kn, 7 * M + 3 * N + K)
    for alpha, beta in [(1.0, 0.0), (1.5, -0.5)]:
        got = _run(lib, gpu, a, b, c, alpha, beta, kn)
        _check(got, a, b, c, alpha, beta, kn)


@pytest.mark.parametrize("kn", [False, True])
@pytest.mark.parametrize("path,bn", [(SQUARE, 64), (SQUARE, 256), (PAIR, 128), (PAIR, 256)])
def test_padded_both_paths(lib, gpu, kn, path, bn):
    # several tiles in both directions and a ragged K tail on each kernel path
    for M, N, K in [(520, 389, 1201), (260, 777, 2051)]:
        a, b, c = _operands(M, N, K, kn, M + N + K)
        got = _run(lib, gpu, a, b, c, -0.75, 1.25, kn, path=path, bn=bn)
        _check(got, a, b, c, -0.75, 1.25, kn)


@pytest.mark.parametrize("which", ["A", "B", "C", "D", "all"])
@pytest.mark.parametrize("off", [1, 2, 4])
def test_padded_misaligned_operands(lib, gpu, which, off):
    # K and N multiples of 8, so only the base address forces a repack; off 1
    # gives 2-byte, off 2 4-byte, off 4 8-byte alignment
    M, N, K = 200, 136, 264
    a, b, c = _operands(M, N, K, False, 11 + off)
    offs = {"A": (off, 0, 0, 0), "B": (0, off, 0, 0), "C": (0, 0, off, 0),
            "D": (0, 0, 0, off), "all": (off, off, off, off)}[which]
    got = _run(lib, gpu, a, b, c, 2.0, -1.0, False, offs=offs)
    _check(got, a, b, c, 2.0, -1.0, False)


@pytest.mark.parametrize("kn", [False, True])
def test_padded_in_place(lib, gpu, kn):
    # C = alpha A B + beta C with C itself misaligned and N ragged
    M, N, K = 190, 203, 77
    a, b, c = _operands(M, N, K, kn, 31)
    got = _run(lib, gpu, a, b, c, 0.5, 0.5, kn, offs=(0, 0, 3, 0), in_place=True)
    _check(got, a, b, c, 0.5, 0.5, kn)
    # and C aligned while N is ragged (the padded D holds C during the GEMM)
    got = _run(lib, gpu, a, b, c, 0.5, 0.5, kn, in_place=True)
    _check(got, a, b, c, 0.5, 0.5, kn)


def test_padded_ternary_bit_exact(lib, gpu):
    # {-1, 0, 1} operands: every partial sum is an integer below 2^11, exact in
    # fp32 and in fp16, so the padded path must match the oracle bit for bit
    M, N, K = 333, 205, 1023
    a = synthetic.ternary(41, (M, K))
    b = synthetic.ternary(42, (N, K))
    got = _run(lib, gpu, a, b, None, 1.0, 0.0, False, offs=(1, 3, 0, 5))
    ref = oracle.gemm_tn(a, b)
    g = got.view(np.float16).astype(np.float64)
    r = ref.view(np.float16).astype(np.float64)
    assert np.array_equal(g, r)


def test_padded_matches_scaled_when_aligned(lib, gpu):
    # nothing needs repacking: the padded entry is the scaled entry, bit for bit
    M, N, K = 300, 264, 200
    a, b, c = _operands(M, N, K, True, 51)
    tb = torch.from_numpy(b.view(np.float16)).to(gpu)
    ta = torch.from_numpy(a.view(np.float16)).to(gpu)
    tc = torch.from_numpy(c.view(np.float16)).to(gpu)
    d0 = torch.empty((M, N), dtype=torch.float16, device=gpu)
    assert lib.padded_workspace_bytes(ta, tb, tc, d0, -0.5, "kn") == 0
    d1 = lib.gemm_f16_scaled(ta, tb, tc, 1.5, -0.5, "kn")
    lib.gemm_f16_padded(ta, tb, tc, 1.5, -0.5, "kn", out=d0,
                        workspace=torch.empty(0, dtype=torch.uint8, device=gpu))
    torch.cuda.synchronize()
    assert torch.equal(d0.view(torch.int16), d1.view(torch.int16))


def test_padded_fp16_accumulator(lib, gpu):
    # the fp16-accumulate option through the padded path: the +0 pad columns
    # only add whole 16-deep slices of zeros, which leave an fp16 sum unchanged
    M, N, K = 260, 131, 251
    a = synthetic.uniform_pm1(61, (M, K))
    b = synthetic.uniform_pm1(62, (N, K))
    got = _run(lib, gpu, a, b, None, 1.0, 0.0, False, offs=(0, 1, 0, 0), acc_f16=1)
    ref = oracle.gemm_tn_f16acc(a, b)
    g = got.view(np.float16).astype(np.float64)
    r = ref.view(np.float16).astype(np.float64)
    # each of the ceil(K/16) slice roundings may differ by an ulp of the
    # running sum, which never exceeds sum_k |a b|
    s_abs = np.abs(a.view(np.float16).astype(np.float64)) @ \
        np.abs(b.view(np.float16).astype(np.float64)).T
    tol = 2 * -(-K // 16) * fp16_ulp(s_abs) + fp16_ulp(r)
    assert np.all(np.abs(g - r) <= tol)


def test_padded_empty_and_k0(lib, gpu):
    a = synthetic.uniform_pm1(71, (37, 0))
    b = synthetic.uniform_pm1(72, (21, 0))
    c = synthetic.uniform_pm1(73, (37, 21))
    got = _run(lib, gpu, a, b, c, 3.0, -2.0, False, offs=(0, 0, 1, 3))
    ref = oracle.gemm_scaled(a, b, c, 3.0, -2.0, False)
    assert np.array_equal(got, ref)
    # M == 0 and N == 0 are no-ops
    for M, N in [(0, 9), (9, 0)]:
        a = synthetic.uniform_pm1(74, (M, 5))
        b = synthetic.uniform_pm1(75, (N, 5))
        got = _run(lib, gpu, a, b, None, 1.0, 0.0, False, offs=(1, 1, 0, 1))
        assert got.shape == (M, N)


def test_padded_rejects_small_workspace(lib, gpu):
    M, N, K = 64, 61, 67
    a, b, c = _operands(M, N, K, False, 81)
    ta, tb = _placed(a, gpu), _placed(b, gpu)
    d = torch.empty((M, N), dtype=torch.float16, device=gpu)
    need = lib.padded_workspace_bytes(ta, tb, None, d, 0.0, "nk")
    assert need > 0
    small = torch.empty(need - 16, dtype=torch.uint8, device=gpu)
    with pytest.raises(lib.GemmError) as e:
        lib.gemm_f16_padded(ta, tb, None, out=d, workspace=small)
    assert e.value.status == lib.GEMM_ERR_INVALID_VALUE
    store = torch.empty(need + 16, dtype=torch.uint8, device=gpu)
    with pytest.raises(lib.GemmError) as e:
        lib.gemm_f16_padded(ta, tb, None, out=d, workspace=store[8:8 + need])
    assert e.value.status == lib.GEMM_ERR_MISALIGNED
    # a workspace of exactly the size asked for is enough
    got = lib.gemm_f16_padded(ta, tb, None, out=d, workspace=store[:need])
    torch.cuda.synchronize()
    st = compare(got.cpu().numpy().view(np.uint16), oracle.gemm_tn(a, b), K, a, b)
    assert st["bad"] == 0, st


def test_padded_odd_sizes_sampled(lib, gpu):
    # the 8191^3 workload timed by the benchmark, on seeded samples and seams
    tag = "c9"
    a_bits, b_bits, spec = synthetic.workload(tag)
    M, N, K = spec["M"], spec["N"], spec["K"]
    ta = torch.from_numpy(a_bits.view(np.float16)).to(gpu)
    tb = torch.from_numpy(b_bits.view(np.float16)).to(gpu)
    d = lib.gemm_f16_padded(ta, tb, None)
    torch.cuda.synchronize()
    status, raw = lib.get_device_error()
    assert status == 0, f"device error word {raw:#x}"
    rows, cols = synthetic.sample_coords(synthetic.seeds(tag)[2], M, N)
    got = d.cpu().numpy().view(np.uint16)[rows, cols]
    ref = oracle.gemm_tn_sampled(a_bits, b_bits, rows, cols)
    st = compare(got, ref, K, a_bits, b_bits)
    assert st["bad"] == 0, st
