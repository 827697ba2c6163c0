"""GPU parity of the 1-SM atom at MMA N = 64 (128 x 64 output tiles, up to 8
stages) against the CPU oracle: every compiled ring depth, ragged tiles,
both output types, the convolution and split-K forms, and the automatic
choice that sends few-tile problems to it. Also the fp32-output conv at a
size where the planner picks an N = 256 variant."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import datagen  # noqa: E402
import oracle  # noqa: E402
import mbarrier_pipelined_tensor_gb300 as tp  # noqa: E402
from gpu_util import check_against_oracle, dev_bf16, expect_ok, host_f64, new_out, run_gemm  # noqa: E402

pytestmark = pytest.mark.gpu

ONE = np.uint16(0x3F80)


@pytest.mark.parametrize("depth", range(2, 9))
def test_n64_every_depth(depth):
    M, N, K = 600, 520, 1216          # N = 8 tiles of 64 + 8 columns
    A, B = datagen.gemm_operands(M, N, K, seed=81)
    got, plan = run_gemm(A, B, M, N, K, K, K, out_f32=False, atom=1, tile_n=64, pipe_depth=depth)
    assert (plan["atom"], plan["tile_n"], plan["pipe_depth"]) == (1, 64, depth)
    assert (plan["m_tiles"], plan["n_tiles"]) == (5, 9)
    ref, ab = oracle.gemm(A, B, M, N, K, K, K)
    check_against_oracle(got, ref, ab, False, f"n64 d{depth}")


@pytest.mark.parametrize("out_f32", [True, False])
def test_n64_ragged_config_padded_c(out_f32):
    M, N, K = 320, 200, 448
    A, B = datagen.gemm_operands(M, N, K, seed=0)
    got, plan = run_gemm(A, B, M, N, K, K, K, ldc=216, out_f32=out_f32, atom=1, tile_n=64)
    assert (plan["tile_n"], plan["grid"]) == (64, 12)
    ref, ab = oracle.gemm(A, B, M, N, K, K, K)
    check_against_oracle(got, ref, ab, out_f32, "n64 320x200x448")


def test_n64_identity_bit_exact():
    M = K = 384
    N = 328
    A = np.where(np.eye(M, K, dtype=bool), ONE, np.uint16(0)).astype(np.uint16)
    B = datagen.Stream(83).uniform_bf16((N, K))
    got, _ = run_gemm(A, B, M, N, K, K, K, out_f32=True, atom=1, tile_n=64)
    assert np.array_equal(got, datagen.bf16_to_f32(B).astype(np.float64).T)


def test_n64_chosen_for_few_tiles():
    M = N = K = 1000
    A, B = datagen.gemm_operands(M, N, K, seed=84, lda=1008, ldb=1008)
    got, plan = run_gemm(A, B, M, N, K, 1008, 1008, out_f32=True)
    assert (plan["atom"], plan["tile_n"], plan["pipe_depth"], plan["grid"]) == (1, 64, 8, 128)
    ref, ab = oracle.gemm(A, B, M, N, K, 1008, 1008)
    check_against_oracle(got, ref, ab, True, "n64 auto 1000^3")


def test_n64_one_tile_row_long_k():
    M, N, K = 128, 4096, 4096
    A, B = datagen.gemm_operands(M, N, K, seed=85)
    got, plan = run_gemm(A, B, M, N, K, K, K, out_f32=False)
    assert (plan["atom"], plan["tile_n"], plan["grid"]) == (1, 64, 64)
    ref, ab = oracle.gemm(A, B, M, N, K, K, K)
    check_against_oracle(got, ref, ab, False, "n64 128x4096x4096")


@pytest.mark.parametrize("K", [64, 100, 200])
@pytest.mark.parametrize("out_f32", [True, False])
def test_n64_conv(K, out_f32):
    # K = 100 bf16: y rows of 200 bytes are not whole 16-byte granules, so the
    # epilogue writes them with plain stores.
    N, H, W, C, R, S, st, pad = 2, 13, 11, 96, 3, 3, 1, 1
    x, w = datagen.conv_operands(N, H, W, C, K, R, S, seed=86)
    P, Q = oracle.conv_out_hw(H, W, R, S, st, pad)
    y = new_out(N * P * Q, K, out_f32)
    tp.tp_conv2d_fprop_bf16_ex(dev_bf16(x), dev_bf16(w), y, N, H, W, C, K, R, S, st, pad, out_f32=out_f32,
                               atom=1, tile_n=64)
    expect_ok()
    plan = tp.tp_last_plan()
    assert (plan["atom"], plan["tile_n"], plan["conv"]) == (1, 64, 1)
    ref, ab = oracle.conv(x, w, N, H, W, C, K, R, S, st, pad)
    check_against_oracle(host_f64(y), ref, ab, out_f32, f"n64 conv K={K}")


@pytest.mark.parametrize("atom", [1, 2])
def test_conv_f32_n256(atom):
    N, H, W, C, K, R, S, st, pad = 2, 13, 11, 96, 256, 3, 3, 1, 1
    x, w = datagen.conv_operands(N, H, W, C, K, R, S, seed=87)
    P, Q = oracle.conv_out_hw(H, W, R, S, st, pad)
    y = new_out(N * P * Q, K, True)
    tp.tp_conv2d_fprop_bf16_ex(dev_bf16(x), dev_bf16(w), y, N, H, W, C, K, R, S, st, pad, out_f32=True,
                               atom=atom, tile_n=256)
    expect_ok()
    assert (tp.tp_last_plan()["atom"], tp.tp_last_plan()["tile_n"]) == (atom, 256)
    ref, ab = oracle.conv(x, w, N, H, W, C, K, R, S, st, pad)
    check_against_oracle(host_f64(y), ref, ab, True, f"conv f32 atom {atom} n256")


def test_conv_f32_auto_where_n256_is_chosen():
    # 32768 output pixels x 256 channels: the planner's pick is an N = 256
    # variant, which must exist in fp32 form (sampled check: two whole images
    # with every padding border, plus random pixels).
    N, H, W, C, K, R, S, st, pad = 8, 64, 64, 64, 256, 3, 3, 1, 1
    x, w = datagen.conv_operands(N, H, W, C, K, R, S, seed=88)
    P, Q = oracle.conv_out_hw(H, W, R, S, st, pad)
    y = new_out(N * P * Q, K, True)
    tp.tp_conv2d_fprop_bf16_ex(dev_bf16(x), dev_bf16(w), y, N, H, W, C, K, R, S, st, pad, out_f32=True)
    expect_ok()
    assert tp.tp_last_plan()["tile_n"] == 256
    rng = np.random.default_rng(88)
    pix = np.unique(np.concatenate([np.arange(P * Q), np.arange((N - 1) * P * Q, N * P * Q),
                                    rng.integers(0, N * P * Q, 1024)]))
    ref, ab = oracle.conv(x, w, N, H, W, C, K, R, S, st, pad, pixels=pix)
    got = host_f64(y)[pix]
    check_against_oracle(got, ref, ab, True, "conv f32 auto 8x64x64x64 -> 256")
