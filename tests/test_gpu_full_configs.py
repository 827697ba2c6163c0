"""Parity at the full benchmark sizes, in the launch configurations the
benchmark times, against the oracle on deterministic samples it can compute
in seconds:

* GEMM 8192^3, N(0,1)*0.02 operands (seed 1): every 32nd row plus the last
  (all 8192 columns) and every 32nd column plus the last (all rows).
* skinny set (seed 3): (128, 8192, 16384) on 64 rows x all columns,
  (4096, 4096, 512) on 128 rows, (1000, 1000, 1000) in full.
* conv 32x56x56x256 * 3x3x256, stride 1, pad 1 (seed 2): every output of
  images 0 and 31 (all padding borders) plus 4096 random pixels.
* 1 GiB copy (seed 4): bit-exact, compared on the device.
* the plain-load producer at the benchmark's fallback row, 4096^3 with
  lda = ldb = 4097 (seed 7): every 128th row plus the last; and the conv
  fallback row, 32x56x56x250 * 3x3x250 (256 filters, seed 9): images 0 and
  31 plus 2048 random pixels.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import datagen  # noqa: E402
import oracle  # noqa: E402
import mbarrier_pipelined_tensor_gb300 as tp  # noqa: E402
from gpu_util import check_against_oracle, dev_bf16, dev_u16, expect_ok, host_f64, new_out  # noqa: E402

pytestmark = pytest.mark.gpu

# Launch configurations the benchmark uses (auto choice plus the explicit
# variants it reports).
GEMM_VARIANTS = [dict(), dict(atom=2, tile_n=256), dict(atom=1, tile_n=256), dict(atom=2, tile_n=128)]


@pytest.fixture(scope="module")
def big_gemm():
    M = N = K = 8192
    A, B = datagen.gemm_operands(M, N, K, seed=1, dist="normal")
    rows = oracle.sample_rows(M, 32)
    cols = oracle.sample_rows(N, 32)
    ref_r, ab_r = oracle.gemm(A, B, M, N, K, K, K, rows=rows)
    ref_c, ab_c = oracle.gemm(A, B, M, N, K, K, K, cols=cols)
    return dict(M=M, N=N, K=K, a=dev_bf16(A), b=dev_bf16(B), rows=rows, cols=cols,
                ref_r=ref_r, ab_r=ab_r, ref_c=ref_c, ab_c=ab_c)


@pytest.mark.parametrize("variant", GEMM_VARIANTS, ids=lambda v: "-".join(f"{k}{x}" for k, x in v.items()) or "auto")
def test_gemm_8192_sampled(big_gemm, variant):
    g = big_gemm
    M, N, K = g["M"], g["N"], g["K"]
    c = new_out(M, N, False)
    tp.tp_gemm_bf16_ex(g["a"], g["b"], c, M, N, K, K, K, N, out_f32=False, **variant)
    expect_ok()
    rows_t = torch.from_numpy(g["rows"]).cuda()
    cols_t = torch.from_numpy(g["cols"]).cuda()
    got_r = host_f64(c.index_select(0, rows_t))
    got_c = host_f64(c.index_select(1, cols_t))
    check_against_oracle(got_r, g["ref_r"], g["ab_r"], False, "8192^3 rows")
    check_against_oracle(got_c, g["ref_c"], g["ab_c"], False, "8192^3 cols")


@pytest.fixture(scope="module")
def skinny():
    return list(zip(datagen.SKINNY_SHAPES, datagen.skinny_operands()))


@pytest.mark.parametrize("idx", [0, 1, 2])
@pytest.mark.parametrize("out_f32", [True, False])
def test_skinny_set_splitk(skinny, idx, out_f32):
    (M, N, K), (A, B) = skinny[idx]
    rows = {0: np.arange(1, 128, 2), 1: oracle.sample_rows(M, 32) + 1, 2: None}[idx]
    if rows is not None:
        rows = np.minimum(rows, M - 1)
    ref, ab = oracle.gemm(A, B, M, N, K, K, K, rows=rows)
    ws = torch.empty(tp.tp_gemm_splitk_workspace_bytes(M, N, 16) // 4, dtype=torch.float32, device="cuda")
    c = new_out(M, N, out_f32)
    tp.tp_gemm_bf16_splitk(dev_bf16(A), dev_bf16(B), c, M, N, K, K, K, N, out_f32=out_f32, splits=0, workspace=ws)
    expect_ok()
    got = host_f64(c if rows is None else c.index_select(0, torch.from_numpy(rows).cuda()))
    check_against_oracle(got, ref, ab, out_f32, f"skinny split-K {M}x{N}x{K}")


@pytest.mark.parametrize("idx", [0, 1, 2])
@pytest.mark.parametrize("out_f32", [True, False])
def test_skinny_set(skinny, idx, out_f32):
    (M, N, K), (A, B) = skinny[idx]
    rows = {0: np.arange(0, 128, 2), 1: oracle.sample_rows(M, 32), 2: None}[idx]
    ref, ab = oracle.gemm(A, B, M, N, K, K, K, rows=rows)
    c = new_out(M, N, out_f32)
    tp.tp_gemm_bf16_ex(dev_bf16(A), dev_bf16(B), c, M, N, K, K, K, N, out_f32=out_f32)
    expect_ok()
    got = host_f64(c if rows is None else c.index_select(0, torch.from_numpy(rows).cuda()))
    check_against_oracle(got, ref, ab, out_f32, f"skinny {M}x{N}x{K}")


@pytest.fixture(scope="module")
def big_conv():
    N, H, W, C, K, R, S = 32, 56, 56, 256, 256, 3, 3
    x, w = datagen.conv_operands(N, H, W, C, K, R, S, seed=2)
    P, Q = oracle.conv_out_hw(H, W, R, S, 1, 1)
    pq = P * Q
    rng = np.random.default_rng(2)
    pix = np.unique(np.concatenate([np.arange(pq), np.arange(31 * pq, 32 * pq),
                                    rng.integers(0, N * pq, 4096)]))
    ref, ab = oracle.conv(x, w, N, H, W, C, K, R, S, 1, 1, pixels=pix)
    return dict(shape=(N, H, W, C, K, R, S), x=dev_bf16(x), w=dev_bf16(w), pix=pix, ref=ref, ab=ab, M=N * pq)


@pytest.mark.parametrize("variant", [dict(), dict(atom=2, tile_n=256), dict(atom=1, tile_n=128),
                                     dict(atom=2, tile_n=128)],
                         ids=lambda v: "-".join(f"{k}{x}" for k, x in v.items()) or "auto")
def test_conv_full_sampled(big_conv, variant):
    g = big_conv
    N, H, W, C, K, R, S = g["shape"]
    y = new_out(g["M"], K, False)
    tp.tp_conv2d_fprop_bf16_ex(g["x"], g["w"], y, N, H, W, C, K, R, S, 1, 1, **variant)
    expect_ok()
    got = host_f64(y.index_select(0, torch.from_numpy(g["pix"]).cuda()))
    check_against_oracle(got, g["ref"], g["ab"], False, "conv 32x56x56x256")


def test_copy_1gib_bit_exact():
    rows, cols = 32768, 16384
    src = dev_u16(datagen.copy_source(rows, cols, seed=4))
    dst = torch.zeros_like(src)
    tp.tp_tma_copy_2d(src, dst, rows, cols, cols)
    expect_ok()
    assert tp.tp_last_plan()["path"] == tp.TP_PATH_TMA_COPY
    assert torch.equal(src, dst)


def test_plain_load_4096_odd_pitch_sampled():
    # The benchmark's fallback row: odd pitches rule TMA out for A and B, so
    # the 1-SM N = 128 mainloop is fed through the row-class windows.
    M = N = K = 4096
    ld = K + 1
    A, B = datagen.gemm_operands(M, N, K, seed=7, dist="normal", lda=ld, ldb=ld)
    rows = oracle.sample_rows(M, 128)
    ref, ab = oracle.gemm(A, B, M, N, K, ld, ld, rows=rows)
    c = new_out(M, N, False)
    tp.tp_gemm_bf16_ex(dev_bf16(A), dev_bf16(B), c, M, N, K, ld, ld, N, atom=1, tile_n=128)
    expect_ok()
    assert tp.tp_last_plan()["path"] == tp.TP_PATH_FALLBACK_MAINLOOP
    got = host_f64(c.index_select(0, torch.from_numpy(rows).cuda()))
    check_against_oracle(got, ref, ab, False, "plain-load 4096^3 odd pitches")


def test_plain_load_conv_c250_sampled():
    # The benchmark's conv fallback row: 250 channels rule TMA out; the
    # stride-1 same-size conv runs on row-class windows.
    N, H, W, C, K, R, S = 32, 56, 56, 250, 256, 3, 3
    x, w = datagen.conv_operands(N, H, W, C, K, R, S, seed=9)
    pq = H * W
    rng = np.random.default_rng(9)
    pix = np.unique(np.concatenate([np.arange(pq), np.arange(31 * pq, 32 * pq), rng.integers(0, N * pq, 2048)]))
    ref, ab = oracle.conv(x, w, N, H, W, C, K, R, S, 1, 1, pixels=pix)
    y = new_out(N * pq, K, False)
    tp.tp_conv2d_fprop_bf16(dev_bf16(x), dev_bf16(w), y, N, H, W, C, K, R, S, 1, 1)
    expect_ok()
    assert tp.tp_last_plan()["path"] == tp.TP_PATH_FALLBACK_MAINLOOP
    got = host_f64(y.index_select(0, torch.from_numpy(pix).cuda()))
    check_against_oracle(got, ref, ab, False, "conv 32x56x56x250 windows")
