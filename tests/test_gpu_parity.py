"""GPU parity of the TMA copy, the 1-SM mainloop and the implicit-GEMM conv
against the CPU oracle, on seeded inputs small enough to check every element
yet spanning several tiles, ragged tails and varied K_TILES ("B200 Tma
Pipeline Designer", step 8: asymmetric small matrices, boundary tiles,
different K_TILES). Every call goes through the C ABI.

Tolerance (fp32 accumulator): |gpu - ref| <= 1e-3 * sum|a*b| + 1e-6 per
element; bf16 outputs add half a bf16 ulp, 2**-8 * |ref|. Copies, and GEMMs
whose every partial sum is exact in fp32 (identity, permutation, all-ones),
must match bit for bit.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import datagen  # noqa: E402
import oracle  # noqa: E402
import mbarrier_pipelined_tensor_gb300 as tp  # noqa: E402
from gpu_util import (check_against_oracle, dev_bf16, dev_u16, expect_ok, host_f64, host_u16,  # noqa: E402
                      new_out, run_gemm)

pytestmark = pytest.mark.gpu

ONE = np.uint16(0x3F80)


# ------------------------------------------------------------------ copy ---

@pytest.mark.parametrize("rows,cols,ld", [(300, 1000, 1000), (257, 130, 136), (1024, 64, 64), (128, 4096, 4104),
                                           (515, 1003, 1016)])
def test_tma_copy_bit_exact_ragged(rows, cols, ld):
    src_h = datagen.copy_source(rows, cols, seed=4, ld=ld)
    src = dev_u16(src_h)
    dst = torch.full_like(src, 0x5A5A)
    tp.tp_tma_copy_2d(src, dst, rows, cols, ld)
    expect_ok()
    assert tp.tp_last_plan()["path"] == tp.TP_PATH_TMA_COPY
    got = host_u16(dst)
    assert np.array_equal(got[:, :cols], src_h[:, :cols])
    assert np.all(got[:, cols:] == 0x5A5A), "copy wrote into the pitch padding"


@pytest.mark.parametrize("box_cols,box_rows,stages,per_sm", [(64, 128, 2, 1), (64, 128, 12, 1), (256, 32, 6, 2),
                                                             (128, 64, 4, 3), (8, 256, 3, 1)])
def test_tma_copy_ring_shapes(box_cols, box_rows, stages, per_sm):
    rows, cols, ld = 777, 1500, 1504
    src_h = datagen.copy_source(rows, cols, seed=5, ld=ld)
    src = dev_u16(src_h)
    dst = torch.zeros_like(src)
    tp.tp_tma_copy_2d_ex(src, dst, rows, cols, ld, box_cols=box_cols, box_rows=box_rows, stages=stages,
                         ctas_per_sm=per_sm)
    expect_ok()
    p = tp.tp_last_plan()
    assert p["path"] == tp.TP_PATH_TMA_COPY and p["pipe_depth"] == stages
    assert np.array_equal(host_u16(dst), src_h)


@pytest.mark.parametrize("rows,cols,ld,offset", [(100, 1001, 1001, 0), (64, 600, 600, 1), (3, 5, 7, 0),
                                                 (200, 512, 520, 3)])
def test_vectorized_fallback_copy(rows, cols, ld, offset):
    total = rows * ld + 16
    src_h = datagen.Stream(6).bits16((total,))
    src_all = dev_u16(src_h)
    dst_all = torch.full_like(src_all, 0x1234)
    src = src_all[offset:]
    dst = dst_all[offset:]
    tp.tp_tma_copy_2d(src, dst, rows, cols, ld)
    expect_ok()
    assert tp.tp_last_plan()["path"] == tp.TP_PATH_VEC_COPY
    got = host_u16(dst_all)
    want = np.full_like(src_h, 0x1234)
    for r in range(rows):
        s = offset + r * ld
        want[s:s + cols] = src_h[s:s + cols]
    assert np.array_equal(got, want)


@pytest.mark.parametrize("rows,cols,ld,so,do", [(64, 600, 600, 1, 0), (50, 1001, 1003, 0, 3), (7, 9, 9, 2, 5),
                                                 (33, 4096, 4097, 7, 1), (16, 100, 104, 4, 1), (5, 1, 3, 1, 6)])
def test_vectorized_copy_relative_misalignment(rows, cols, ld, so, do):
    # src and dst with different alignments: aligned 16-byte stores whose
    # bytes are cut from two aligned source chunks.
    total = rows * ld + 16
    src_h = datagen.Stream(60 + so + do).bits16((total,))
    src_all = dev_u16(src_h)
    dst_all = torch.full_like(src_all, 0x1234)
    tp.tp_tma_copy_2d(src_all[so:], dst_all[do:], rows, cols, ld)
    expect_ok()
    assert tp.tp_last_plan()["path"] == tp.TP_PATH_VEC_COPY
    got = host_u16(dst_all)
    want = np.full_like(src_h, 0x1234)
    for r in range(rows):
        want[do + r * ld:do + r * ld + cols] = src_h[so + r * ld:so + r * ld + cols]
    assert np.array_equal(got, want)


def test_forced_fallback_matches_tma():
    rows, cols = 512, 2048
    src_h = datagen.copy_source(rows, cols, seed=7)
    src = dev_u16(src_h)
    d1, d2 = torch.zeros_like(src), torch.zeros_like(src)
    tp.tp_tma_copy_2d(src, d1, rows, cols, cols)
    tp.tp_tma_copy_2d_ex(src, d2, rows, cols, cols, force_vec=True)
    expect_ok()
    assert torch.equal(d1, src) and torch.equal(d2, src)


def test_copy_empty_and_invalid():
    src = torch.zeros(16, dtype=torch.int16, device="cuda")
    tp.tp_tma_copy_2d(src, src, 0, 5, 5)
    with pytest.raises(tp.TPError):
        tp.tp_tma_copy_2d(src, src, 2, 5, 4)


# ------------------------------------------------------------ bounded wait ---

def test_bounded_wait_gives_up_with_status():
    tp.tp_selftest_wait_timeout(2000)
    st, site, block, thread = tp.tp_device_status_detail()
    assert st == tp.TP_ERR_TIMEOUT and site == 7
    assert tp.tp_device_status() == tp.TP_OK  # cleared
    # The context is still usable.
    src = dev_u16(datagen.copy_source(256, 256, seed=8))
    dst = torch.zeros_like(src)
    tp.tp_tma_copy_2d(src, dst, 256, 256, 256)
    expect_ok()
    assert torch.equal(src, dst)


def test_mainloop_lost_arrival_times_out_and_recovers():
    # The producer withholds its first stage's expect_tx arrival but issues the
    # loads (the lost-arrival bug): the MMA issuer's bounded wait must give up,
    # the kernel must drain and return, and the context must stay usable.
    M, N, K = 256, 256, 512
    A, B = datagen.gemm_operands(M, N, K, seed=95)
    a, b = dev_bf16(A), dev_bf16(B)
    c = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    tp.tp_selftest_mainloop_withheld_arrival(a, b, c, M, N, K, 200)
    st, site, block, thread = tp.tp_device_status_detail()
    # Whichever dependent bounded wait expires first records it: the MMA
    # issuer's (2), the epilogue's (4) or the producer's (1).
    assert st == tp.TP_ERR_TIMEOUT and site in (1, 2, 4), (st, site)
    assert tp.tp_device_status() == tp.TP_OK
    got, _ = run_gemm(A, B, M, N, K, K, K, out_f32=True, atom=1, tile_n=128)
    ref, ab = oracle.gemm(A, B, M, N, K, K, K)
    check_against_oracle(got, ref, ab, True, "after the lost-arrival self test")


# ---------------------------------------------------------- GEMM, 1-SM ---

@pytest.mark.parametrize("out_f32", [True, False])
def test_gemm_ragged_config_every_element(out_f32):
    M, N, K = 320, 200, 448
    A, B = datagen.gemm_operands(M, N, K, seed=0)
    got, plan = run_gemm(A, B, M, N, K, K, K, out_f32=out_f32)
    assert plan["path"] == tp.TP_PATH_MAINLOOP and plan["k_blocks"] == 7
    ref, ab = oracle.gemm(A, B, M, N, K, K, K)
    check_against_oracle(got, ref, ab, out_f32, "320x200x448")


def test_gemm_left_identity_bit_exact():
    M = K = 192
    N = 320
    A = np.where(np.eye(M, K, dtype=bool), ONE, np.uint16(0)).astype(np.uint16)
    B = datagen.Stream(11).uniform_bf16((N, K))
    got, _ = run_gemm(A, B, M, N, K, K, K, out_f32=True)
    assert np.array_equal(got, datagen.bf16_to_f32(B).astype(np.float64).T)


def test_gemm_permutation_bit_exact():
    M = K = 256
    N = 136
    perm = np.random.default_rng(3).permutation(K)
    A = np.zeros((M, K), dtype=np.uint16)
    A[np.arange(M), perm] = ONE
    B = datagen.Stream(12).uniform_bf16((N, K))
    got, _ = run_gemm(A, B, M, N, K, K, K, out_f32=True)
    assert np.array_equal(got, datagen.bf16_to_f32(B).astype(np.float64)[:, perm].T)
    got16, _ = run_gemm(A, B, M, N, K, K, K, out_f32=False)
    assert np.array_equal(got16, datagen.bf16_to_f32(B).astype(np.float64)[:, perm].T)


@pytest.mark.parametrize("K", [64, 1000, 4096])
def test_gemm_all_ones_is_k(K):
    M, N = 136, 264
    A = np.full((M, K), ONE, dtype=np.uint16)
    B = np.full((N, K), ONE, dtype=np.uint16)
    got, _ = run_gemm(A, B, M, N, K, K, K, out_f32=True)
    assert np.all(got == K)


@pytest.mark.parametrize("M", [1, 127, 129, 200])
@pytest.mark.parametrize("N", [1, 64, 129, 200])
@pytest.mark.parametrize("K", [16, 40, 448, 1001])
def test_gemm_shape_grid(M, N, K):
    lda = ldb = (K + 7) // 8 * 8
    A, B = datagen.gemm_operands(M, N, K, seed=M * 7 + N * 13 + K, lda=lda, ldb=ldb)
    ldc = (N + 7) // 8 * 8
    got, plan = run_gemm(A, B, M, N, K, lda, ldb, ldc=ldc, out_f32=(M + N) % 2 == 0)
    assert plan["k_blocks"] == (K + 63) // 64
    ref, ab = oracle.gemm(A, B, M, N, K, lda, ldb)
    check_against_oracle(got, ref, ab, (M + N) % 2 == 0, f"{M}x{N}x{K}")


def test_gemm_pitched_operands_with_poisoned_padding():
    M, N, K = 300, 260, 520
    lda, ldb, ldc = K + 24, K + 40, N + 20
    A, B = datagen.gemm_operands(M, N, K, seed=21, lda=lda, ldb=ldb)
    for out_f32 in (True, False):
        got, _ = run_gemm(A, B, M, N, K, lda, ldb, ldc=ldc, out_f32=out_f32)
        ref, ab = oracle.gemm(A, B, M, N, K, lda, ldb)
        check_against_oracle(got, ref, ab, out_f32, "pitched")


def test_gemm_k_zero_writes_zeros():
    M, N = 37, 70
    a = torch.zeros(8, dtype=torch.bfloat16, device="cuda")
    c = new_out(M, 72, True)
    tp.tp_gemm_bf16_ex(a, a, c, M, N, 0, 8, 8, 72, out_f32=True)
    expect_ok()
    h = c.cpu().numpy()
    assert np.all(h[:, :N] == 0) and np.all(np.isnan(h[:, N:]))


ATOM1 = [(128, d) for d in range(2, 7)] + [(256, d) for d in range(2, 5)]


@pytest.mark.parametrize("tile_n,depth", ATOM1)
def test_gemm_atom1_every_depth(tile_n, depth):
    M, N, K = 520, 600, 1216  # 19 K-blocks: more than, and not a multiple of, every depth
    A, B = datagen.gemm_operands(M, N, K, seed=31)
    got, plan = run_gemm(A, B, M, N, K, K, K, out_f32=False, atom=1, tile_n=tile_n, pipe_depth=depth)
    assert (plan["atom"], plan["tile_n"], plan["pipe_depth"]) == (1, tile_n, depth)
    ref, ab = oracle.gemm(A, B, M, N, K, K, K)
    check_against_oracle(got, ref, ab, False, f"atom1 n{tile_n} d{depth}")


def test_gemm_persistent_many_tiles_small_grid():
    # Few CTAs, many tiles: each CTA loops through tiles, the two TMEM
    # accumulators alternate and the stage ring wraps many times.
    M, N, K = 1024, 1024, 320
    A, B = datagen.gemm_operands(M, N, K, seed=41)
    for tile_n in (64, 128, 256):
        got, plan = run_gemm(A, B, M, N, K, K, K, out_f32=True, atom=1, tile_n=tile_n, max_ctas=3, group_m=3)
        assert plan["grid"] == 3
        ref, ab = oracle.gemm(A, B, M, N, K, K, K)
        check_against_oracle(got, ref, ab, True, f"persistent n{tile_n}")


@pytest.mark.parametrize("atom,tile_n", [(1, 64), (1, 128), (1, 256), (2, 128), (2, 256)])
def test_gemm_odd_waves_walk_k_backwards(atom, tile_n):
    # A persistent CTA's odd-numbered units load their K blocks last to first.
    # Two clusters over many tiles give every CTA several odd waves. With a
    # permutation A every output is one product, exact in any order, so a K
    # block loaded from the wrong coordinate shows as a wrong element.
    M = K = 640
    N = 384
    perm = np.random.default_rng(17).permutation(K)
    A = np.zeros((M, K), dtype=np.uint16)
    A[np.arange(M), perm] = ONE
    B = datagen.Stream(18).uniform_bf16((N, K))
    got, plan = run_gemm(A, B, M, N, K, K, K, out_f32=True, atom=atom, tile_n=tile_n, max_ctas=2 * atom,
                         group_m=2, no_tail=1)
    assert plan["grid"] == 2 * atom and plan["m_tiles"] * plan["n_tiles"] >= 6
    assert np.array_equal(got, datagen.bf16_to_f32(B).astype(np.float64)[:, perm].T)
    # Ragged K (the last block partly past K) on random operands, with the
    # narrow tail on where the variant has one.
    M, N, K = 700, 520, 1000
    A, B = datagen.gemm_operands(M, N, K, seed=19)
    got, plan = run_gemm(A, B, M, N, K, K, K, out_f32=True, atom=atom, tile_n=tile_n, max_ctas=4 * atom)
    ref, ab = oracle.gemm(A, B, M, N, K, K, K)
    check_against_oracle(got, ref, ab, True, f"odd waves atom{atom} n{tile_n}")


# ---------------------------------------------- plain-load producer ---

@pytest.mark.parametrize("M,N,K,lda,ldb,ldc,offs", [
    (300, 200, 448, 449, 450, 201, (1, 3, 5)),     # odd pitches, misaligned bases
    (129, 77, 1000, 1003, 1001, 77, (0, 0, 1)),
    (520, 600, 1216, 1216, 1216, 600, (4, 0, 0)),  # only A misaligned (by 8 bytes)
])
@pytest.mark.parametrize("out_f32", [True, False])
def test_gemm_fallback_producer(M, N, K, lda, ldb, ldc, offs, out_f32):
    A, B = datagen.gemm_operands(M, N, K, seed=51, lda=lda, ldb=ldb)
    oa, ob, oc = offs
    a_all = dev_bf16(np.concatenate([np.zeros(oa, np.uint16), A.reshape(-1)]))
    b_all = dev_bf16(np.concatenate([np.zeros(ob, np.uint16), B.reshape(-1)]))
    c_all = new_out(1, M * ldc + oc, out_f32).reshape(-1)
    a, b, c = a_all[oa:], b_all[ob:], c_all[oc:]
    tp.tp_gemm_bf16_ex(a, b, c, M, N, K, lda, ldb, ldc, out_f32=out_f32)
    expect_ok()
    assert tp.tp_last_plan()["path"] == tp.TP_PATH_FALLBACK_MAINLOOP
    full = host_f64(c_all)
    assert np.all(np.isnan(full[:oc]))
    got = full[oc:].reshape(M, ldc)
    assert np.all(np.isnan(got[:, N:]))
    ref, ab = oracle.gemm(A, B, M, N, K, lda, ldb)
    check_against_oracle(got[:, :N], ref, ab, out_f32, "fallback producer")


@pytest.mark.parametrize("M,N,K,lda,ldb,offs", [
    (5, 3, 100, 101, 103, (1, 1)),        # fewer than 8 rows: classes without rows
    (8, 8, 64, 65, 66, (0, 0)),           # one row per class, one K block
    (17, 300, 8, 9, 11, (0, 0)),          # K < 8: the window is mostly zero fill
    (1000, 136, 200, 203, 207, (3, 7)),   # every class offset, ragged M and N tiles
    (256, 384, 2000, 2001, 2005, (0, 2)),  # K tail 16 elements past a window boundary
    (640, 520, 512, 512, 512, (1, 0)),    # aligned pitch, base 2 bytes off: one offset for all classes
])
def test_gemm_row_class_windows(M, N, K, lda, ldb, offs):
    # The plain-load GEMM reads each row class (rows r mod 8) through its own
    # TMA window; cover classes with no rows, every window offset, K and
    # row tails, against the oracle and (fp32 C) bit for bit against the TMA
    # producer on the same values.
    A, B = datagen.gemm_operands(M, N, K, seed=M + K, lda=lda, ldb=ldb)
    oa, ob = offs
    a_all = dev_bf16(np.concatenate([np.zeros(oa, np.uint16), A.reshape(-1)]))
    b_all = dev_bf16(np.concatenate([np.zeros(ob, np.uint16), B.reshape(-1)]))
    c = new_out(M, N, True)
    tp.tp_gemm_bf16_ex(a_all[oa:], b_all[ob:], c, M, N, K, lda, ldb, N, out_f32=True)
    expect_ok()
    assert tp.tp_last_plan()["path"] == tp.TP_PATH_FALLBACK_MAINLOOP
    ref, ab = oracle.gemm(A, B, M, N, K, lda, ldb)
    got = host_f64(c)
    check_against_oracle(got, ref, ab, True, "row-class windows")
    if (K * 2) % 16 == 0:
        # packed copies go through the TMA producer (one wave of tiles: it
        # walks K forwards, as the plain loads do)
        Ap = np.ascontiguousarray(A.reshape(M, lda)[:, :K])
        Bp = np.ascontiguousarray(B.reshape(N, ldb)[:, :K])
        c2 = new_out(M, N, True)
        tp.tp_gemm_bf16_ex(dev_bf16(Ap), dev_bf16(Bp), c2, M, N, K, K, K, N, out_f32=True, atom=1, tile_n=128,
                           pipe_depth=6)
        expect_ok()
        assert tp.tp_last_plan()["path"] == tp.TP_PATH_MAINLOOP
        assert torch.equal(c, c2)


@pytest.mark.parametrize("case", [(2, 9, 7, 3, 20, 3, 3, 1, 1), (1, 12, 11, 70, 66, 3, 3, 2, 1),
                                  (2, 6, 6, 12, 8, 1, 1, 1, 0)])
def test_conv_fallback_producer(case):
    # C or K not a multiple of 8: the im2col tiles are gathered with plain loads.
    N, H, W, C, K, R, S, st, pad = case
    x, w = datagen.conv_operands(N, H, W, C, K, R, S, seed=52)
    P, Q = oracle.conv_out_hw(H, W, R, S, st, pad)
    y = new_out(N * P * Q, K, True)
    tp.tp_conv2d_fprop_bf16_ex(dev_bf16(x), dev_bf16(w), y, N, H, W, C, K, R, S, st, pad, out_f32=True)
    expect_ok()
    assert tp.tp_last_plan()["path"] == tp.TP_PATH_FALLBACK_MAINLOOP
    ref, ab = oracle.conv(x, w, N, H, W, C, K, R, S, st, pad)
    check_against_oracle(host_f64(y), ref, ab, True, f"conv fallback {case}")


@pytest.mark.parametrize("atom,tile_n", [(1, 128), (2, 256)])
@pytest.mark.parametrize("out_f32", [True, False])
def test_gemm_c_without_tma_stores(atom, tile_n, out_f32):
    # A and B suit TMA, C does not (base off by one element, odd pitch): the
    # TMA producer runs and the epilogue writes all of C with plain stores.
    M, N, K, ldc, oc = 300, 203, 448, 205, 1
    A, B = datagen.gemm_operands(M, N, K, seed=54)
    c_all = new_out(1, M * ldc + oc, out_f32).reshape(-1)
    c = c_all[oc:]
    tp.tp_gemm_bf16_ex(dev_bf16(A), dev_bf16(B), c, M, N, K, K, K, ldc, out_f32=out_f32, atom=atom, tile_n=tile_n)
    expect_ok()
    assert tp.tp_last_plan()["path"] == tp.TP_PATH_MAINLOOP
    full = host_f64(c_all)
    assert np.isnan(full[0])
    got = full[oc:].reshape(M, ldc)
    assert np.all(np.isnan(got[:, N:]))
    ref, ab = oracle.gemm(A, B, M, N, K, K, K)
    check_against_oracle(got[:, :N], ref, ab, out_f32, "C by plain stores")


@pytest.mark.parametrize("out_f32", [True, False])
def test_splitk_into_unaligned_c(out_f32):
    # The reduction's scalar stores: C off by one element, odd pitch.
    M, N, K, ldc, oc = 128, 331, 2048, 333, 1
    A, B = datagen.gemm_operands(M, N, K, seed=55)
    ws = torch.empty(tp.tp_gemm_splitk_workspace_bytes(M, N, 4) // 4, dtype=torch.float32, device="cuda")
    c_all = new_out(1, M * ldc + oc, out_f32).reshape(-1)
    tp.tp_gemm_bf16_splitk(dev_bf16(A), dev_bf16(B), c_all[oc:], M, N, K, K, K, ldc, out_f32=out_f32, splits=4,
                           workspace=ws)
    expect_ok()
    assert tp.tp_last_plan()["splits"] == 4
    full = host_f64(c_all)
    got = full[oc:].reshape(M, ldc)
    assert np.isnan(full[0]) and np.all(np.isnan(got[:, N:]))
    ref, ab = oracle.gemm(A, B, M, N, K, K, K)
    check_against_oracle(got[:, :N], ref, ab, out_f32, "split-K unaligned C")


@pytest.mark.parametrize("out_f32", [True, False])
def test_conv_output_channels_not_granular(out_f32):
    # K = 100 output channels: y rows are not whole 16-byte granules, so y is
    # written with plain stores while x and w still load through TMA.
    N, H, W, C, K, R, S = 2, 10, 9, 64, 100, 3, 3
    x, w = datagen.conv_operands(N, H, W, C, K, R, S, seed=56)
    y = new_out(N * H * W, K, out_f32)
    tp.tp_conv2d_fprop_bf16_ex(dev_bf16(x), dev_bf16(w), y, N, H, W, C, K, R, S, 1, 1, out_f32=out_f32)
    expect_ok()
    assert tp.tp_last_plan()["path"] == tp.TP_PATH_MAINLOOP
    ref, ab = oracle.conv(x, w, N, H, W, C, K, R, S, 1, 1)
    check_against_oracle(host_f64(y), ref, ab, out_f32, "conv K=100")


CONV_WIN_CASES = [
    # N, H, W, C, K, R, S, pad, (x offset, w offset) in elements
    (2, 9, 7, 3, 20, 3, 3, 1, (0, 0)),
    (1, 13, 11, 130, 136, 3, 3, 1, (0, 0)),   # three channel blocks, the last 2 wide
    (2, 8, 8, 250, 256, 3, 3, 1, (1, 3)),     # odd channels, misaligned bases
    (1, 10, 12, 64, 72, 5, 5, 2, (1, 0)),     # C a multiple of 8, x 2 bytes off
    (3, 5, 5, 17, 9, 1, 1, 0, (0, 0)),        # 1x1
    (1, 1, 3, 5, 4, 3, 3, 1, (0, 0)),         # fewer than 8 pixels and filters: empty classes
    (4, 20, 18, 36, 140, 3, 3, 1, (2, 1)),    # 1440 pixels: several tiles, ragged last tile
    (1, 30, 30, 19, 300, 3, 3, 1, (0, 5)),    # three filter tiles, the last ragged
    (1, 16, 15, 40, 64, 7, 7, 3, (1, 1)),     # 7x7: 49 taps, offsets across three image rows
]


@pytest.mark.parametrize("case", CONV_WIN_CASES)
@pytest.mark.parametrize("out_f32", [True, False])
def test_conv_row_class_windows(case, out_f32):
    # Stride-1 convolutions whose output is the input's size, on operands TMA
    # cannot describe: the plain-load producer loads each tap's pixels and
    # the filters through row-class windows, masking padding rows and the
    # channels past C.
    N, H, W, C, K, R, S, pad, (ox, ow) = case
    x, w = datagen.conv_operands(N, H, W, C, K, R, S, seed=N * H + C)
    x_all = dev_bf16(np.concatenate([np.zeros(ox, np.uint16), x.reshape(-1)]))
    w_all = dev_bf16(np.concatenate([np.zeros(ow, np.uint16), w.reshape(-1)]))
    y = new_out(N * H * W, K, out_f32)
    tp.tp_conv2d_fprop_bf16_ex(x_all[ox:], w_all[ow:], y, N, H, W, C, K, R, S, 1, pad, out_f32=out_f32)
    expect_ok()
    assert tp.tp_last_plan()["path"] == tp.TP_PATH_FALLBACK_MAINLOOP
    ref, ab = oracle.conv(x, w, N, H, W, C, K, R, S, 1, pad)
    check_against_oracle(host_f64(y), ref, ab, out_f32, f"conv windows {case}")


def test_conv_windows_match_tma_path_bit_for_bit():
    # Only the base's alignment rules TMA out: both producers stage the same
    # swizzled tiles in the same K order, so fp32 outputs agree exactly.
    N, H, W, C, K, R, S = 2, 14, 13, 128, 256, 3, 3
    x, w = datagen.conv_operands(N, H, W, C, K, R, S, seed=88)
    x_off = dev_bf16(np.concatenate([np.zeros(1, np.uint16), x.reshape(-1)]))[1:]
    y1, y2 = new_out(N * H * W, K, True), new_out(N * H * W, K, True)
    tp.tp_conv2d_fprop_bf16_ex(dev_bf16(x), dev_bf16(w), y1, N, H, W, C, K, R, S, 1, 1, out_f32=True, atom=1,
                               tile_n=128)
    assert tp.tp_last_plan()["path"] == tp.TP_PATH_MAINLOOP
    tp.tp_conv2d_fprop_bf16_ex(x_off, dev_bf16(w), y2, N, H, W, C, K, R, S, 1, 1, out_f32=True)
    expect_ok()
    assert tp.tp_last_plan()["path"] == tp.TP_PATH_FALLBACK_MAINLOOP
    assert torch.equal(y1, y2)


def test_fallback_matches_tma_path_bit_for_bit():
    # The same operands through both producers: the tensor core sees the same
    # swizzled stages, so the outputs are identical.
    M, N, K = 384, 256, 640
    A, B = datagen.gemm_operands(M, N, K, seed=53)
    a, b = dev_bf16(A), dev_bf16(B)
    b_off_all = dev_bf16(np.concatenate([np.zeros(1, np.uint16), B.reshape(-1)]))
    c1, c2 = new_out(M, N, True), new_out(M, N, True)
    tp.tp_gemm_bf16_ex(a, b, c1, M, N, K, K, K, N, out_f32=True, atom=1, tile_n=128, pipe_depth=6)
    tp.tp_gemm_bf16_ex(a, b_off_all[1:], c2, M, N, K, K, K, N, out_f32=True)
    expect_ok()
    assert tp.tp_last_plan()["path"] == tp.TP_PATH_FALLBACK_MAINLOOP
    assert torch.equal(c1, c2)


# ------------------------------------------------------------------ conv ---

CONV_CASES = [
    # N, H, W, C, K, R, S, stride, pad
    (2, 9, 7, 64, 64, 3, 3, 1, 1),
    (1, 12, 10, 16, 72, 3, 3, 1, 1),      # C < 64: channel overhang zero-filled
    (2, 11, 9, 128, 200, 3, 3, 2, 1),     # stride 2, ragged N
    (3, 6, 6, 96, 128, 1, 1, 1, 0),       # 1x1
    (1, 10, 13, 32, 64, 3, 5, 1, 2),      # R != S, pad 2
    (2, 7, 7, 8, 8, 3, 3, 1, 0),          # no padding, tiny C
]


@pytest.mark.parametrize("case", CONV_CASES)
@pytest.mark.parametrize("out_f32", [True, False])
def test_conv_small_every_element(case, out_f32):
    N, H, W, C, K, R, S, st, pad = case
    x, w = datagen.conv_operands(N, H, W, C, K, R, S, seed=2)
    P, Q = oracle.conv_out_hw(H, W, R, S, st, pad)
    y = new_out(N * P * Q, K, out_f32)
    tp.tp_conv2d_fprop_bf16_ex(dev_bf16(x), dev_bf16(w), y, N, H, W, C, K, R, S, st, pad, out_f32=out_f32,
                               atom=1)
    expect_ok()
    assert tp.tp_last_plan()["conv"] == 1
    ref, ab = oracle.conv(x, w, N, H, W, C, K, R, S, st, pad)
    check_against_oracle(host_f64(y), ref, ab, out_f32, f"conv {case}")


def test_conv_centre_delta_bit_exact():
    N, H, W, C = 2, 16, 12, 64
    x = datagen.Stream(9).uniform_bf16((N, H, W, C))
    w = np.zeros((C, 3, 3, C), dtype=np.uint16)
    w[np.arange(C), 1, 1, np.arange(C)] = ONE
    y = new_out(N * H * W, C, True)
    tp.tp_conv2d_fprop_bf16_ex(dev_bf16(x), dev_bf16(w), y, N, H, W, C, C, 3, 3, 1, 1, out_f32=True, atom=1)
    expect_ok()
    assert np.array_equal(host_f64(y), datagen.bf16_to_f32(x).astype(np.float64).reshape(-1, C))


# ------------------------------------------------------- latency probe ---

@pytest.mark.parametrize("kind,floor,ceiling", [(0, 4, 16), (1, 8, 512)])
def test_fma_chain_latency_probe(kind, floor, ceiling):
    # The chain's result is exact (seed + chain < 2^24); the cycles per link
    # bound the RAW latency from above. The hazards note measured 4 (fp32)
    # and 8 (fp64) cycles on B200; GB300's fp64 path is far slower (about 64
    # cycles per dependent DFMA), so only plausibility is checked.
    seed, chain = 3.0, 64 * 1024
    result, cpl = tp.tp_probe_fma_latency(kind, chain, seed)
    assert result == seed + chain
    assert 1.0 <= cpl <= ceiling
    print(f"kind {kind}: {cpl:.2f} cycles per dependent fma (B200 note: {floor})")


# ------------------------------------------------ host-buffer end to end ---

def _pinned(arr):
    t = torch.from_numpy(np.ascontiguousarray(arr))
    return t.pin_memory()


@pytest.mark.parametrize("out_f32", [True, False])
def test_gemm_host_buffers_end_to_end(out_f32):
    M, N, K, lda, ldb, ldc = 300, 200, 448, 456, 464, 208    # pitched, ragged tiles
    A, B = datagen.gemm_operands(M, N, K, seed=57, lda=lda, ldb=ldb)
    a_h, b_h = _pinned(A.view(np.int16)), _pinned(B.view(np.int16))
    c_h = torch.full((M, ldc), -1, dtype=torch.int32 if out_f32 else torch.int16).pin_memory()
    dA = torch.empty(M * lda, dtype=torch.int16, device="cuda")
    dB = torch.empty(N * ldb, dtype=torch.int16, device="cuda")
    dC = torch.empty((M, ldc), dtype=torch.float32 if out_f32 else torch.bfloat16, device="cuda")
    tp.tp_gemm_bf16_host(a_h, b_h, c_h, M, N, K, lda, ldb, ldc, dA, dB, dC, out_f32=out_f32)
    torch.cuda.synchronize()
    expect_ok()
    raw = c_h.numpy()
    got = (raw.view(np.float32) if out_f32 else datagen.bf16_to_f32(raw.view(np.uint16))).astype(np.float64)
    assert np.all(raw[:, N:] == -1)                  # the pitch padding is not written
    ref, ab = oracle.gemm(A, B, M, N, K, lda, ldb)
    check_against_oracle(got[:, :N], ref, ab, out_f32, "host buffers")
    # The same kernels as the device-resident call: identical bits.
    c_dev = new_out(M, ldc, out_f32)
    tp.tp_gemm_bf16_ex(dA.view(torch.bfloat16), dB.view(torch.bfloat16), c_dev, M, N, K, lda, ldb, ldc,
                       out_f32=out_f32)
    dev = host_f64(c_dev)
    assert np.array_equal(dev[:, :N], got[:, :N])


def test_gemm_host_buffers_k0_and_errors():
    M, N = 5, 9
    c_h = torch.full((M, N), 7.0, dtype=torch.float32).pin_memory()
    dC = torch.empty((M, N), dtype=torch.float32, device="cuda")
    tp.tp_gemm_bf16_host(None, None, c_h, M, N, 0, 0, 0, N, None, None, dC, out_f32=True)
    torch.cuda.synchronize()
    assert torch.count_nonzero(c_h) == 0
    with pytest.raises(tp.TPError) as e:
        tp.tp_gemm_bf16_host(None, None, c_h, M, N, 4, 4, 4, N, None, None, dC, out_f32=True)
    assert e.value.status == tp.TP_ERR_INVALID_ARG


def test_gemm_host_buffers_pageable():
    # Pageable (not page-locked) host memory: the copies are staged by the
    # driver and block the host, with the same result.
    M, N, K = 200, 136, 256
    A, B = datagen.gemm_operands(M, N, K, seed=58)
    a_h, b_h = np.ascontiguousarray(A), np.ascontiguousarray(B)
    c_h = np.zeros((M, N), dtype=np.float32)
    dA = torch.empty(M * K, dtype=torch.int16, device="cuda")
    dB = torch.empty(N * K, dtype=torch.int16, device="cuda")
    dC = torch.empty((M, N), dtype=torch.float32, device="cuda")
    tp.tp_gemm_bf16_host(a_h.ctypes.data, b_h.ctypes.data, c_h.ctypes.data, M, N, K, K, K, N, dA, dB, dC,
                         out_f32=True)
    torch.cuda.synchronize()
    expect_ok()
    ref, ab = oracle.gemm(A, B, M, N, K, K, K)
    check_against_oracle(c_h.astype(np.float64), ref, ab, True, "pageable host buffers")


# ------------------------------------------------ torch-facing wrappers ---

@pytest.mark.parametrize("out_f32", [True, False])
def test_convenience_wrappers(out_f32):
    # tp.gemm / tp.conv2d_fprop take shapes and pitches from the tensors:
    # a padded-pitch A (a column slice of a wider buffer) and a flat y.
    M, N, K = 300, 200, 448
    A, B = datagen.gemm_operands(M, N, K, seed=91, lda=456)
    a_full = dev_bf16(A)                     # M x 456, the first K columns used
    b = dev_bf16(B)
    c = new_out(M, N, out_f32)
    tp.gemm(a_full[:, :K], b, c)
    expect_ok()
    ref, ab = oracle.gemm(A, B, M, N, K, 456, K)
    check_against_oracle(host_f64(c), ref, ab, out_f32, "tp.gemm")
    Nb, H, W, C, Kc, R, S = 2, 9, 7, 64, 72, 3, 3
    x, w = datagen.conv_operands(Nb, H, W, C, Kc, R, S, seed=92)
    y = new_out(Nb * H * W, Kc, out_f32)
    tp.conv2d_fprop(dev_bf16(x).view(Nb, H, W, C), dev_bf16(w).view(Kc, R, S, C), y, stride=1, pad=1)
    expect_ok()
    ref, ab = oracle.conv(x, w, Nb, H, W, C, Kc, R, S, 1, 1)
    check_against_oracle(host_f64(y), ref, ab, out_f32, "tp.conv2d_fprop")
