"""GPU parity of the 2-SM atom (a cluster of two CTAs issuing cta_group::2
MMAs, each CTA holding half of the B tile: "two-free-pipeline-stages", "The
atom changes the fragment") against the CPU oracle, for every compiled ring
depth, both MMA N, ragged pair tiles and the convolution."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import datagen  # noqa: E402
import oracle  # noqa: E402
import mbarrier_pipelined_tensor_gb300 as tp  # noqa: E402
from gpu_util import check_against_oracle, dev_bf16, expect_ok, host_f64, new_out, run_gemm  # noqa: E402

pytestmark = pytest.mark.gpu

ONE = np.uint16(0x3F80)


@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("out_f32", [True, False])
def test_atom2_ragged_config(tile_n, out_f32):
    M, N, K = 320, 200, 448       # pair tile 256 rows: the second pair's upper CTA is all out of bounds
    A, B = datagen.gemm_operands(M, N, K, seed=0)
    got, plan = run_gemm(A, B, M, N, K, K, K, out_f32=out_f32, atom=2, tile_n=tile_n)
    assert plan["atom"] == 2 and plan["cluster"] == 2 and plan["grid"] % 2 == 0
    ref, ab = oracle.gemm(A, B, M, N, K, K, K)
    check_against_oracle(got, ref, ab, out_f32, f"atom2 n{tile_n}")


def test_atom2_identity_bit_exact():
    M = K = 512
    N = 384
    A = np.where(np.eye(M, K, dtype=bool), ONE, np.uint16(0)).astype(np.uint16)
    B = datagen.Stream(13).uniform_bf16((N, K))
    for tile_n in (128, 256):
        got, _ = run_gemm(A, B, M, N, K, K, K, out_f32=True, atom=2, tile_n=tile_n)
        assert np.array_equal(got, datagen.bf16_to_f32(B).astype(np.float64).T)


ATOM2 = [(128, d) for d in range(2, 9)] + [(256, d) for d in range(2, 7)]


@pytest.mark.parametrize("tile_n,depth", ATOM2)
def test_atom2_every_depth(tile_n, depth):
    M, N, K = 600, 520, 1216
    A, B = datagen.gemm_operands(M, N, K, seed=32)
    got, plan = run_gemm(A, B, M, N, K, K, K, out_f32=False, atom=2, tile_n=tile_n, pipe_depth=depth)
    assert (plan["atom"], plan["tile_n"], plan["pipe_depth"]) == (2, tile_n, depth)
    ref, ab = oracle.gemm(A, B, M, N, K, K, K)
    check_against_oracle(got, ref, ab, False, f"atom2 n{tile_n} d{depth}")


def test_atom2_persistent_small_grid():
    M, N, K = 1280, 1024, 384
    A, B = datagen.gemm_operands(M, N, K, seed=42)
    for tile_n in (128, 256):
        got, plan = run_gemm(A, B, M, N, K, K, K, out_f32=True, atom=2, tile_n=tile_n, max_ctas=4, group_m=2)
        assert plan["grid"] == 4
        ref, ab = oracle.gemm(A, B, M, N, K, K, K)
        check_against_oracle(got, ref, ab, True, f"atom2 persistent n{tile_n}")


@pytest.mark.parametrize("tile_n,out_f32", [(128, False), (128, True), (256, False)])
def test_atom2_conv(tile_n, out_f32):
    N, H, W, C, K, R, S, st, pad = 2, 13, 11, 96, 256, 3, 3, 1, 1
    x, w = datagen.conv_operands(N, H, W, C, K, R, S, seed=22)
    P, Q = oracle.conv_out_hw(H, W, R, S, st, pad)
    y = new_out(N * P * Q, K, out_f32)
    tp.tp_conv2d_fprop_bf16_ex(dev_bf16(x), dev_bf16(w), y, N, H, W, C, K, R, S, st, pad, out_f32=out_f32,
                               atom=2, tile_n=tile_n)
    expect_ok()
    assert tp.tp_last_plan()["atom"] == 2
    ref, ab = oracle.conv(x, w, N, H, W, C, K, R, S, st, pad)
    check_against_oracle(host_f64(y), ref, ab, out_f32, "atom2 conv")


# ------------------------------------------------------ narrow tail ---

@pytest.mark.parametrize("M,N,K,max_ctas", [(1280, 512, 640, 8),     # 10 tiles on 4 clusters: 8 whole + 4 halves
                                             (2560, 2048, 384, 0),    # 80 tiles on 76 clusters: 76 + 16 quarters
                                             (2560, 2048, 384, 100000),  # the same, one cluster per unit (92)
                                             (600, 100, 448, 0),      # 3 tiles, all quarters; upper ones out of N
                                             (320, 200, 448, 0),
                                             (5120, 4096, 448, 0)])   # 320 tiles on 76: 304 whole + 32 halves
@pytest.mark.parametrize("out_f32", [True, False])
def test_narrow_tail_units(M, N, K, max_ctas, out_f32):
    A, B = datagen.gemm_operands(M, N, K, seed=M + N)
    ldc = (N + 7) // 8 * 8
    got, plan = run_gemm(A, B, M, N, K, K, K, ldc=ldc, out_f32=out_f32, atom=2, tile_n=256, max_ctas=max_ctas)
    assert plan["tail_units"] > 0 and plan["tail_parts"] in (2, 4)
    tiles = plan["m_tiles"] * plan["n_tiles"]
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    wave = min(pairs, max_ctas // 2) if max_ctas else pairs   # clusters that run at once
    r = tiles % wave
    assert plan["tail_parts"] == (4 if 4 * r <= wave else 2)  # quarters when they fit one wave
    ref, ab = oracle.gemm(A, B, M, N, K, K, K)
    check_against_oracle(got, ref, ab, out_f32, f"narrow tail {M}x{N}x{K}")
    got2, plan2 = run_gemm(A, B, M, N, K, K, K, ldc=ldc, out_f32=out_f32, atom=2, tile_n=256, max_ctas=max_ctas,
                           no_tail=1)
    assert plan2["tail_units"] == 0
    check_against_oracle(got2, ref, ab, out_f32, f"whole tiles {M}x{N}x{K}")
    if out_f32:
        assert np.array_equal(got, got2)   # same MMAs per output element, same order


def test_narrow_tail_conv():
    N, H, W, C, K, R, S = 4, 20, 18, 64, 256, 3, 3   # 1440 pixels: 6 pair tiles, all quarters
    x, w = datagen.conv_operands(N, H, W, C, K, R, S, seed=23)
    y = new_out(N * H * W, K, False)
    tp.tp_conv2d_fprop_bf16_ex(dev_bf16(x), dev_bf16(w), y, N, H, W, C, K, R, S, 1, 1, atom=2, tile_n=256)
    expect_ok()
    assert tp.tp_last_plan()["tail_units"] == 24 and tp.tp_last_plan()["tail_parts"] == 4
    ref, ab = oracle.conv(x, w, N, H, W, C, K, R, S, 1, 1)
    check_against_oracle(host_f64(y), ref, ab, False, "conv narrow tail")


# ------------------------------------------------------- role timeline ---

@pytest.mark.parametrize("atom,tile_n", [(2, 256), (1, 128)])
def test_role_timeline(atom, tile_n):
    M, N, K = 2560, 2048, 1024
    A, B = datagen.gemm_operands(M, N, K, seed=81)
    a, b = dev_bf16(A), dev_bf16(B)
    c1, c2 = new_out(M, N, True), new_out(M, N, True)
    tp.tp_gemm_bf16_ex(a, b, c1, M, N, K, K, K, N, out_f32=True, atom=atom, tile_n=tile_n)
    plan = tp.tp_last_plan()
    trace = torch.zeros(tp.TRACE_SLOTS * plan["grid"], dtype=torch.int64, device="cuda")
    tp.tp_gemm_bf16_ex(a, b, c2, M, N, K, K, K, N, out_f32=True, atom=atom, tile_n=tile_n, trace=trace)
    expect_ok()
    assert torch.equal(c1, c2)                                  # tracing does not change results
    t = trace.view(plan["grid"], tp.TRACE_SLOTS).cpu().numpy()
    issuers = t[::atom]                                         # the pair's leader issues the MMAs
    tiles = plan["m_tiles"] * plan["n_tiles"]
    parts = plan["tail_parts"] or 1
    # whole tiles, with each tail tile split into `parts` units
    assert issuers[:, 7].sum() == tiles - plan["tail_units"] // parts + plan["tail_units"]
    for rows, span, wait in ((t, 0, 1), (issuers, 2, 3), (issuers, 2, 4), (t, 5, 6)):
        assert np.all(rows[:, span] > 0) and np.all(rows[:, wait] <= rows[:, span])


@pytest.mark.parametrize("atom,tile_n", [(2, 256), (2, 128), (1, 128), (1, 64)])
def test_event_timeline(atom, tile_n):
    # The per-unit event timeline on a small grid (many units per CTA): every
    # CTA runs units cluster_id, cluster_id + clusters, ... in that order,
    # each role's events are in order, and the two TMEM accumulators
    # alternate: a unit's MMAs start only after the epilogue warps of its
    # CTA (both CTAs of a pair) handed back the accumulator of the unit two
    # before it.
    M, N, K = 2560, 2048, 1024
    A, B = datagen.gemm_operands(M, N, K, seed=84)
    a, b = dev_bf16(A), dev_bf16(B)
    c = new_out(M, N, False)
    opts = dict(atom=atom, tile_n=tile_n, max_ctas=16)
    tp.tp_gemm_bf16_ex(a, b, c, M, N, K, K, K, N, **opts)
    plan = tp.tp_last_plan()
    grid = plan["grid"]
    ev = torch.zeros(grid * tp.EVENT_SLOTS, dtype=torch.int64, device="cuda")
    tp.tp_gemm_bf16_ex(a, b, c, M, N, K, K, K, N, events=ev, **opts)
    expect_ok()
    e = ev.view(grid, tp.EVENT_UNITS, tp.EVENTS_PER_UNIT).cpu().numpy().astype(np.int64)
    P0, P1, M0, M1, E0, E1, E2, U = range(8)
    clusters = grid // atom
    parts = plan["tail_parts"] or 1
    units = plan["m_tiles"] * plan["n_tiles"] - plan["tail_units"] // parts + plan["tail_units"]
    assert units >= clusters * tp.EVENT_UNITS   # every CTA fills all its event slots
    for cta in range(grid):
        cid, leader = cta // atom, cta - (cta // atom) * atom == 0
        lead = cid * atom
        for k in range(tp.EVENT_UNITS):
            r = e[cta, k]
            assert r[U] == cid + k * clusters
            assert 0 < r[P0] <= r[P1]
            assert 0 < r[E0] <= r[E1] <= r[E2]
            m = e[lead, k]
            assert 0 < m[M0] <= m[M1] <= r[E0]      # accumulator complete only after its last MMAs
            if k >= 2:
                for peer in range(lead, lead + atom):
                    assert e[peer, k - 2, E1] <= m[M0], (cta, k)
        if not leader:
            assert np.all(e[cta, :, [M0, M1]] == 0)   # the MMA issuer runs on the pair's leader
    ref, ab = oracle.gemm(A, B, M, N, K, K, K, rows=np.arange(0, M, 97))
    check_against_oracle(host_f64(c)[::97], ref, ab, False, "events run")
