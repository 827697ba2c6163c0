"""GPU parity of split-K: (tile, K slice) work units of the mainloop write
fp32 partials into a caller workspace, a reduction kernel sums them into C.
Checked element by element against the oracle (same tolerance: the fp32
accumulator bound holds for any summation order)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import datagen  # noqa: E402
import oracle  # noqa: E402
import mbarrier_pipelined_tensor_gb300 as tp  # noqa: E402
from gpu_util import check_against_oracle, dev_bf16, expect_ok, host_f64, new_out  # noqa: E402

pytestmark = pytest.mark.gpu


def run_splitk(A, B, M, N, K, lda, ldb, ldc, out_f32, splits, ws_splits=None, **opts):
    ws_splits = splits if ws_splits is None else ws_splits
    nbytes = tp.tp_gemm_splitk_workspace_bytes(M, N, max(1, ws_splits))
    ws = torch.full((nbytes // 4,), float("nan"), dtype=torch.float32, device="cuda")
    c = new_out(M, ldc, out_f32)
    tp.tp_gemm_bf16_splitk(dev_bf16(A), dev_bf16(B), c, M, N, K, lda, ldb, ldc, out_f32=out_f32, splits=splits,
                           workspace=ws, **opts)
    expect_ok()
    plan = tp.tp_last_plan()
    full = host_f64(c)
    assert np.all(np.isnan(full[:, N:]))
    return full[:, :N], plan


@pytest.mark.parametrize("splits", [2, 3, 7])
@pytest.mark.parametrize("out_f32", [True, False])
def test_splitk_skinny(splits, out_f32):
    M, N, K = 128, 1024, 4096
    A, B = datagen.gemm_operands(M, N, K, seed=61)
    got, plan = run_splitk(A, B, M, N, K, K, K, N, out_f32, splits)
    assert plan["splits"] == splits
    ref, ab = oracle.gemm(A, B, M, N, K, K, K)
    check_against_oracle(got, ref, ab, out_f32, f"split-K {splits}")


@pytest.mark.parametrize("atom,tile_n", [(1, 64), (1, 128), (1, 256), (2, 128), (2, 256)])
def test_splitk_every_variant_ragged(atom, tile_n):
    M, N, K = 300, 201, 1001
    lda = ldb = 1008
    A, B = datagen.gemm_operands(M, N, K, seed=62, lda=lda, ldb=ldb)
    got, plan = run_splitk(A, B, M, N, K, lda, ldb, 208, True, 4, atom=atom, tile_n=tile_n)
    assert (plan["atom"], plan["tile_n"], plan["splits"]) == (atom, tile_n, 4)
    ref, ab = oracle.gemm(A, B, M, N, K, lda, ldb)
    check_against_oracle(got, ref, ab, True, f"split-K atom{atom} n{tile_n}")


@pytest.mark.parametrize("atom,tile_n", [(1, 128), (2, 256)])
def test_splitk_odd_waves(atom, tile_n):
    # Two clusters over 3 slices of every tile: most (tile, slice) units run
    # in odd waves, whose K blocks are loaded last to first.
    M, N, K = 300, 201, 1001
    lda = ldb = 1008  # split-K feeds the mainloop through TMA: 16-byte pitches
    A, B = datagen.gemm_operands(M, N, K, seed=64, lda=lda, ldb=ldb)
    got, plan = run_splitk(A, B, M, N, K, lda, ldb, N, True, 3, atom=atom, tile_n=tile_n, max_ctas=2 * atom)
    assert plan["splits"] == 3 and plan["grid"] == 2 * atom
    ref, ab = oracle.gemm(A, B, M, N, K, lda, ldb)
    check_against_oracle(got, ref, ab, True, f"split-K odd waves atom{atom} n{tile_n}")


def test_splitk_slices_never_empty():
    # K = 130 is 3 K blocks; 5 slices asked -> 3 used, each non-empty.
    M, N, K = 256, 256, 136
    A, B = datagen.gemm_operands(M, N, K, seed=63)
    got, plan = run_splitk(A, B, M, N, K, K, K, N, True, 5)
    assert plan["splits"] == 3 and plan["k_blocks"] == 3
    ref, ab = oracle.gemm(A, B, M, N, K, K, K)
    check_against_oracle(got, ref, ab, True, "split-K clamp")


def test_splitk_auto_is_capped_by_workspace():
    M, N, K = 128, 2048, 8192
    A, B = datagen.gemm_operands(M, N, K, seed=64)
    got, plan = run_splitk(A, B, M, N, K, K, K, N, False, 0, ws_splits=2)
    assert plan["splits"] <= 2
    ref, ab = oracle.gemm(A, B, M, N, K, K, K)
    check_against_oracle(got, ref, ab, False, "split-K auto")


def test_splitk_identity_is_exact():
    # Every partial sum of an identity product is exact: slices add zeros.
    M = K = 512
    N = 320
    A = np.where(np.eye(M, K, dtype=bool), np.uint16(0x3F80), np.uint16(0)).astype(np.uint16)
    B = datagen.Stream(65).uniform_bf16((N, K))
    got, plan = run_splitk(A, B, M, N, K, K, K, N, True, 4)
    assert plan["splits"] == 4
    assert np.array_equal(got, datagen.bf16_to_f32(B).astype(np.float64).T)


def test_splitk_errors():
    M, N, K = 128, 256, 1024
    a = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    b = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
    c = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    small = torch.zeros(16, dtype=torch.float32, device="cuda")
    with pytest.raises(tp.TPError) as e:
        tp.tp_gemm_bf16_splitk(a, b, c, M, N, K, K, K, N, out_f32=True, splits=4, workspace=small)
    assert e.value.status == tp.TP_ERR_INVALID_ARG
    # One slice needs no workspace: the plain mainloop runs.
    tp.tp_gemm_bf16_splitk(a, b, c, M, N, K, K, K, N, out_f32=True, splits=1, workspace=None)
    expect_ok()
    assert tp.tp_last_plan()["splits"] == 1


@pytest.mark.parametrize("out_f32", [True, False])
def test_splitk_plain_load_producer(out_f32):
    # Odd pitches: the K slices run on the plain-load producer's row-class
    # windows and write their fp32 partials like the TMA producer's.
    M, N, K, ld = 200, 384, 2500, 2503
    A, B = datagen.gemm_operands(M, N, K, seed=71, lda=ld, ldb=ld)
    a, b = dev_bf16(A), dev_bf16(B)
    splits = 4
    ws = torch.empty(tp.tp_gemm_splitk_workspace_bytes(M, N, splits) // 4, dtype=torch.float32, device="cuda")
    c = new_out(M, N, out_f32)
    tp.tp_gemm_bf16_splitk(a, b, c, M, N, K, ld, ld, N, out_f32=out_f32, splits=splits, workspace=ws)
    expect_ok()
    plan = tp.tp_last_plan()
    assert plan["path"] == tp.TP_PATH_FALLBACK_MAINLOOP and plan["splits"] == splits
    ref, ab = oracle.gemm(A, B, M, N, K, ld, ld)
    check_against_oracle(host_f64(c), ref, ab, out_f32, "split-K plain-load")
