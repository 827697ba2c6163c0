"""Invariants of the host planner over many seeded random problems (no GPU:
tp_gemm_plan only plans). For every shape, pitch, alignment and option mix:
the plan picks a compiled variant, its shared memory fits, the persistent
grid is a whole number of clusters no larger than the machine (or max_ctas),
it never has more clusters than work units, the last-wave bookkeeping adds
up, and the tile counts cover the problem exactly."""
import random

import pytest

import mbarrier_pipelined_tensor_gb300 as tp

SM_COUNT = 152
SMEM_LIMIT = 232448
AL = 1 << 20


def _cdiv(a, b):
    return (a + b - 1) // b


@pytest.fixture(scope="module")
def compiled():
    return {(k["atom"], k["tile_n"], k["pipe_depth"], k["out_f32"], k["conv"], k["ldg"], k["splitk"])
            for k in tp.tp_list_kernels()}


def _random_problem(rng):
    M = rng.choice([1, 7, 127, 128, 129, 255, 256, 300, 1000, 2048, 4096, 9728, 100352, rng.randint(1, 20000)])
    N = rng.choice([1, 8, 100, 128, 200, 256, 257, 1024, 8192, rng.randint(1, 20000)])
    K = rng.choice([0, 1, 8, 16, 64, 448, 1000, 4096, 16384, rng.randint(0, 70000)])
    pad = rng.choice([0, 0, 0, 8, 3])
    lda, ldb, ldc = K + pad, K + rng.choice([0, 8, 1]), N + rng.choice([0, 8, 5])
    base = rng.choice([0, 0, 0, 2, 16])
    opts = {}
    if rng.random() < 0.4:
        opts["atom"] = rng.choice([1, 2])
    if rng.random() < 0.4:
        opts["tile_n"] = rng.choice([64, 128, 256])
    if rng.random() < 0.2:
        opts["max_ctas"] = rng.choice([1, 2, 3, 8, 64, 151, 152, 300])
    if rng.random() < 0.2:
        opts["no_tail"] = 1
    if rng.random() < 0.2:
        opts["group_m"] = rng.choice([1, 4, 8, 33])
    return M, N, K, lda, ldb, ldc, base, rng.random() < 0.5, opts


def test_plans_satisfy_invariants(compiled):
    rng = random.Random(20261202)
    checked = 0
    for _ in range(3000):
        M, N, K, lda, ldb, ldc, base, out_f32, opts = _random_problem(rng)
        st, p = tp.tp_gemm_plan(AL + base, AL, AL, M, N, K, lda, ldb, ldc, out_f32=out_f32, sm_count=SM_COUNT,
                                **opts)
        if st != tp.TP_OK:
            # Only explicit choices the library does not offer may be refused:
            # a variant the planner picks by itself always exists.
            if "atom" not in opts and "tile_n" not in opts:
                assert st != tp.TP_ERR_UNSUPPORTED, (M, N, K, out_f32, opts)
            assert st in (tp.TP_ERR_UNSUPPORTED, tp.TP_ERR_INVALID_ARG, tp.TP_ERR_SMEM_BUDGET), (st, M, N, K, opts)
            if st == tp.TP_ERR_INVALID_ARG:
                assert base % 2 == 1 or (out_f32 and base % 4) or ldc < N or lda < K or ldb < K
            continue
        if K == 0:
            assert p["path"] == tp.TP_PATH_ZERO_FILL
            continue
        checked += 1
        assert p["path"] in (tp.TP_PATH_MAINLOOP, tp.TP_PATH_FALLBACK_MAINLOOP)
        ldg = 1 if p["path"] == tp.TP_PATH_FALLBACK_MAINLOOP else 0
        key = (p["atom"], p["tile_n"], p["pipe_depth"], int(out_f32), 0, ldg, 0)
        assert key in compiled, key
        assert 0 < p["smem_bytes"] <= SMEM_LIMIT
        assert p["cluster"] == p["atom"] and p["grid"] % p["atom"] == 0
        assert p["m_tiles"] == _cdiv(M, 128 * p["atom"]) and p["n_tiles"] == _cdiv(N, p["tile_n"])
        assert p["k_blocks"] == _cdiv(K, 64)
        tiles = p["m_tiles"] * p["n_tiles"]
        cap = opts.get("max_ctas", SM_COUNT)
        clusters = p["grid"] // p["atom"]
        parts = p["tail_parts"]
        assert 1 <= clusters <= max(1, cap // p["atom"]) or (p["tail_units"] and clusters <= parts * tiles)
        units = tiles if not p["tail_units"] else tiles - p["tail_units"] // parts + p["tail_units"]
        assert clusters <= units
        if p["tail_units"]:
            # Narrow tail: only the 2-SM, N = 256 variant, never with no_tail,
            # two or four narrow units per leftover tile, at most one wave of
            # them, quarters whenever they fit.
            assert (p["atom"], p["tile_n"]) == (2, 256) and not opts.get("no_tail")
            assert parts in (2, 4) and p["tail_units"] % parts == 0 and p["tail_units"] // parts <= tiles
            assert p["tail_units"] <= max(clusters, parts)
            wave = min(max(1, cap // 2), SM_COUNT // 2)
            assert (parts == 4) == (4 * (p["tail_units"] // parts) <= wave)
        else:
            assert parts == 0
        assert p["l2_hint"] in range(1, 7)
    assert checked > 1000


def test_plan_is_a_pure_function_of_its_inputs():
    rng = random.Random(7)
    for _ in range(200):
        M, N, K, lda, ldb, ldc, base, out_f32, opts = _random_problem(rng)
        a = tp.tp_gemm_plan(AL + base, AL, AL, M, N, K, lda, ldb, ldc, out_f32=out_f32, sm_count=SM_COUNT, **opts)
        b = tp.tp_gemm_plan(AL + base, AL, AL, M, N, K, lda, ldb, ldc, out_f32=out_f32, sm_count=SM_COUNT, **opts)
        assert a == b
