"""Planner invariants over many seeded shapes and options (host only, no GPU):
every plan the library accepts fits the hardware and is self-consistent."""
import numpy as np
import pytest

from multistage_smem_pipeline_gb300 import synthetic

SMEM_LIMIT = 232448      # dynamic shared memory per CTA on sm_100-class parts
TMEM_COLS = 512


@pytest.fixture(scope="module")
def binding():
    from multistage_smem_pipeline_gb300 import build
    build.build()
    from multistage_smem_pipeline_gb300 import binding as b
    return b


def _shapes(n, seed):
    u = synthetic.uniform01(seed, 3 * n).reshape(n, 3)
    # log-uniform sizes: M in [1, 2^17], N and K in [8, 2^15], N and K multiples of 8
    M = np.maximum(1, np.exp2(u[:, 0] * 17)).astype(np.int64)
    N = np.maximum(1, np.exp2(u[:, 1] * 12)).astype(np.int64) * 8
    K = np.maximum(1, np.exp2(u[:, 2] * 12)).astype(np.int64) * 8
    return list(zip(M.tolist(), N.tolist(), K.tolist()))


def _check(cfg, M, N, K):
    assert cfg["smem_bytes"] <= SMEM_LIMIT
    assert 2 <= cfg["kstage"] <= 16
    assert cfg["katoms"] in (1, 2) and cfg["bk"] == 64 * cfg["katoms"]
    assert cfg["epi_warps"] in (4, 8)
    assert 32 <= cfg["bn"] <= 256 and cfg["bn"] % 32 == 0
    # two accumulators, or one in the small-M kernel (one tile per CTA)
    accs = 1 if (cfg["small_m"] or cfg["split_k"]) else 2
    assert cfg["tmem_cols"] >= accs * cfg["bn"] and cfg["tmem_cols"] <= TMEM_COLS
    assert cfg["tmem_cols"] & (cfg["tmem_cols"] - 1) == 0          # a power of two
    bm = 256 if cfg["path"] == 3 else 128
    assert cfg["bm"] == bm
    assert cfg["tiles"] == -(-M // bm) * -(-N // cfg["bn"])
    if cfg["split_k"]:
        # clusters of 2 (one tile), 4 or 8 (1 x 2, 2 x 1 or 2 x 2 tiles, operands multicast);
        # a ragged edge still gets whole clusters
        nm, nn = -(-M // 128), -(-N // cfg["bn"])
        packs = {2: [(1, 1)], 4: [(2, 1), (1, 2)], 8: [(2, 2)]}[cfg["cluster"]]
        assert cfg["ctas"] in [cfg["cluster"] * -(-nm // cm) * -(-nn // cn) for cm, cn in packs]
        assert cfg["cluster"] != 8 or (nm >= 2 and nn >= 2)     # a partner on both sides
        assert cfg["cluster"] != 4 or nm >= 2 or nn >= 2
        assert cfg["bn"] % 64 == 0 and cfg["path"] == 1
        assert cfg["epi_warps"] == 8 and not cfg["b_resident"] and not cfg["small_m"]
        # the ring holds the eight warps' staging buffers once the MMAs are done, and the
        # peer's 128 x bn/2 fp32 partial has a region of its own
        ring = cfg["kstage"] * cfg["katoms"] * (128 + cfg["bn"]) * 128
        assert ring >= 32768 and cfg["smem_bytes"] >= ring + 256 * cfg["bn"]
    else:
        assert 1 <= cfg["ctas"] <= cfg["tiles"] * (2 if cfg["path"] == 3 else 1)
        assert cfg["cluster"] == (2 if cfg["path"] == 3 else 1)
    if cfg["path"] == 3:
        assert cfg["ctas"] % 2 == 0                                    # whole clusters of 2
    if cfg["path"] == 2:
        assert M <= 128
    if cfg["small_m"]:
        assert cfg["path"] == 2 and cfg["ctas"] == cfg["tiles"] and cfg["epi_warps"] == 4
        assert not cfg["b_resident"] and not cfg["wide"]
    if cfg["wide"]:
        units = -(-M // 256) * -(-(-(-N // cfg["bn"])) // 2)
        assert cfg["path"] == 3 and cfg["ctas"] <= 2 * units and not cfg["b_resident"]
    if cfg["b_resident"]:
        num_n = -(-N // cfg["bn"])
        assert cfg["path"] != 3 and num_n <= 4 and cfg["ctas"] % num_n == 0
        assert num_n == 1 or cfg["group_m"] == 1
    # balanced grids: with one CTA fewer (one pair fewer; num_n CTAs fewer with
    # resident B) the same work would need another wave
    if cfg["path"] == 3:
        num_n = -(-N // cfg["bn"])
        work = -(-M // 256) * (-(-num_n // 2) if cfg["wide"] else num_n)
        slots, step = cfg["ctas"] // 2, 1
    elif cfg["split_k"]:
        return  # one cluster per tile group: nothing to balance
    else:
        work, slots = cfg["tiles"], cfg["ctas"]
        step = -(-N // cfg["bn"]) if cfg["b_resident"] else 1
    waves = -(-work // slots)
    assert slots - step < 1 or (slots - step) * waves < work, (cfg, work)


def test_default_plans_fit(binding):
    for M, N, K in _shapes(3000, 501):
        _check(binding.query_config(M, N, K), M, N, K)


@pytest.mark.parametrize("opts", [dict(path=1), dict(path=3), dict(katoms=1), dict(katoms=2),
                                  dict(epi_warps=4), dict(epi_warps=8), dict(b_resident=1),
                                  dict(acc_f16=1), dict(b_layout=1), dict(max_ctas=37),
                                  dict(wide=2), dict(wide=2, path=3, epi_warps=8),
                                  dict(wide=1), dict(small_m=1), dict(small_m=2),
                                  dict(small_m=2, katoms=1), dict(split_k=1), dict(split_k=2),
                                  dict(split_k=2, katoms=1), dict(split_k=2, bn=256),
                                  dict(split_k=2, multicast=1), dict(split_k=2, multicast=2),
                                  dict(split_k=2, multicast=2, max_ctas=32)])
def test_forced_plans_fit_or_are_refused(binding, opts):
    accepted = 0
    for M, N, K in _shapes(600, 502 + len(str(opts))):
        try:
            cfg = binding.query_config(M, N, K, **opts)
        except binding.GemmError as e:
            assert e.status == binding.GEMM_ERR_INVALID_VALUE
            continue
        accepted += 1
        _check(cfg, M, N, K)
        if "path" in opts and opts["path"] == 3:
            assert cfg["path"] == 3
        if "katoms" in opts:
            assert cfg["katoms"] == opts["katoms"]
        if "epi_warps" in opts:
            assert cfg["epi_warps"] == opts["epi_warps"]
        if "max_ctas" in opts:
            assert cfg["ctas"] <= opts["max_ctas"]
        if opts.get("wide") == 2:
            assert cfg["wide"] == 1
        if opts.get("wide") == 1:
            assert cfg["wide"] == 0
        if "split_k" in opts:
            assert cfg["split_k"] == (1 if opts["split_k"] == 2 else 0)
        if "multicast" in opts:
            assert cfg["split_k"] == 1 and (cfg["cluster"] > 2) == (opts["multicast"] == 2)
        if "small_m" in opts:
            assert cfg["small_m"] == (1 if opts["small_m"] == 2 else 0)
        if opts.get("b_resident") == 1:
            assert cfg["b_resident"] == 0
        if opts.get("b_layout") == 1:
            assert cfg["bn"] % (128 if cfg["path"] == 3 else 64) == 0 and not cfg["b_resident"]
    assert accepted > 0


def test_every_ring_depth_that_is_offered_fits(binding):
    for M, N, K in _shapes(200, 503):
        deepest = binding.query_config(M, N, K)["kstage"]
        for ks in range(2, deepest + 1):
            _check(binding.query_config(M, N, K, kstage=ks), M, N, K)
        if deepest < 16:
            with pytest.raises(binding.GemmError):
                binding.query_config(M, N, K, kstage=deepest + 1)
