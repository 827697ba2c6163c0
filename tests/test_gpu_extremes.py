"""GPU parity at extreme sizes, on outputs the oracle computes one by one.

* An 8.6 GB C (131072 x 32765 bf16, pitch 32768): byte offsets past 4 GiB in
  the TMA stores and in the plain stores of the ragged last columns.
* K = 2^20 (16384 K blocks): the stage ring's phases wrap thousands of
  times within one tile; also through split-K.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import datagen  # noqa: E402
import oracle  # noqa: E402
import mbarrier_pipelined_tensor_gb300 as tp  # noqa: E402
from gpu_util import check_against_oracle, dev_bf16, expect_ok, host_f64  # noqa: E402

pytestmark = pytest.mark.gpu


def test_output_beyond_4gib():
    M, N, K, ldc = 131072, 32765, 64, 32768
    A, B = datagen.gemm_operands(M, N, K, seed=71)
    c = torch.empty((M, ldc), dtype=torch.bfloat16, device="cuda")
    tp.tp_gemm_bf16_ex(dev_bf16(A), dev_bf16(B), c, M, N, K, K, K, ldc)
    expect_ok()
    assert c.numel() * 2 > (1 << 32)
    rows = np.unique(np.concatenate([np.arange(0, M, 4099), np.arange(M - 5, M)]))
    cols = np.unique(np.concatenate([np.arange(0, N, 1021), np.arange(N - 13, N)]))
    ref_r, ab_r = oracle.gemm(A, B, M, N, K, K, K, rows=rows)
    got_r = host_f64(c.index_select(0, torch.from_numpy(rows).cuda()))[:, :N]
    check_against_oracle(got_r, ref_r, ab_r, False, "rows of an 8.6 GB C")
    ref_c, ab_c = oracle.gemm(A, B, M, N, K, K, K, cols=cols)
    got_c = host_f64(c[:, :N].index_select(1, torch.from_numpy(cols).cuda()))
    check_against_oracle(got_c, ref_c, ab_c, False, "columns of an 8.6 GB C")


@pytest.fixture(scope="module")
def long_k():
    M, N, K = 128, 192, 1 << 20
    A, B = datagen.gemm_operands(M, N, K, seed=72)
    rows = np.array([0, 1, 63, 64, 126, 127])
    ref, ab = oracle.gemm(A, B, M, N, K, K, K, rows=rows)
    return dict(M=M, N=N, K=K, a=dev_bf16(A), b=dev_bf16(B), rows=rows, ref=ref, ab=ab)


@pytest.mark.parametrize("opts", [dict(atom=1, tile_n=128), dict(atom=1, tile_n=256)],
                         ids=["1sm-n128-d6", "1sm-n256-d4"])
def test_long_k_ring_wraps(long_k, opts):
    g = long_k
    c = torch.full((g["M"], g["N"]), float("nan"), dtype=torch.float32, device="cuda")
    tp.tp_gemm_bf16_ex(g["a"], g["b"], c, g["M"], g["N"], g["K"], g["K"], g["K"], g["N"], out_f32=True, **opts)
    expect_ok()
    assert tp.tp_last_plan()["k_blocks"] == 16384
    got = host_f64(c.index_select(0, torch.from_numpy(g["rows"]).cuda()))
    check_against_oracle(got, g["ref"], g["ab"], True, f"K = 2^20 {opts}")


def test_long_k_split(long_k):
    g = long_k
    ws = torch.empty(tp.tp_gemm_splitk_workspace_bytes(g["M"], g["N"], 16) // 4, dtype=torch.float32,
                     device="cuda")
    c = torch.full((g["M"], g["N"]), float("nan"), dtype=torch.float32, device="cuda")
    tp.tp_gemm_bf16_splitk(g["a"], g["b"], c, g["M"], g["N"], g["K"], g["K"], g["K"], g["N"], out_f32=True,
                           splits=16, workspace=ws)
    expect_ok()
    assert tp.tp_last_plan()["splits"] == 16
    got = host_f64(c.index_select(0, torch.from_numpy(g["rows"]).cuda()))
    check_against_oracle(got, g["ref"], g["ab"], True, "K = 2^20 split 16")


def _pattern(rows, cols):
    """rows x cols 16-bit patterns (any bits, NaN payloads included), made on
    the device by torch: a copy's expected result is its own source."""
    n = rows * cols
    g = torch.arange(n, dtype=torch.int64, device="cuda")
    return ((g * 2654435761 + (g >> 13)) & 0xFFFF).to(torch.int32).to(torch.int16).view(rows, cols)


@pytest.mark.parametrize("force_vec", [False, True], ids=["tma", "vectorized"])
def test_copy_beyond_2_31_elements(force_vec):
    rows, cols = 131075, 16392                      # 2.149e9 elements, 4.3 GB each way
    src = _pattern(rows, cols)
    assert src.numel() > (1 << 31)
    dst = torch.zeros_like(src)
    tp.tp_tma_copy_2d_ex(src, dst, rows, cols, cols, force_vec=force_vec)
    expect_ok()
    assert torch.equal(src, dst)
    del dst


def test_transpose_beyond_2_31_elements():
    rows, cols = 131075, 16392
    src = _pattern(rows, cols)
    dst = torch.empty((cols, rows), dtype=torch.int16, device="cuda")
    tp.tp_tma_transpose_2d(src, dst, rows, cols, cols, rows)
    expect_ok()
    assert torch.equal(dst, src.t())
