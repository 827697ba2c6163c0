"""The split-K GEMM entry point that allocates nothing.

tp_gemm_bf16_splitk_noalloc exists for callers that may not allocate device
memory while they run (a fixed device-memory budget reserved up front by
another allocator, or code where cudaMalloc's implicit device-wide
synchronization is not allowed): its partial sums live in a fixed array
inside the library. This checks, through the C ABI, that two calls in a row
really split K into the slices asked for (so the fixed array is used), give
bit for bit the output of tp_gemm_bf16_splitk (the same split-K work with a
caller workspace, summed in the same order) and meet the oracle's tolerance;
that a call left to choose its slice count chooses one that fits the array;
and that a request larger than the array is refused. The file sorts last so
that a run stopping at the first failure has already run every other test;
it needs no earlier test.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import datagen  # noqa: E402
import oracle  # noqa: E402
import mbarrier_pipelined_tensor_gb300 as tp  # noqa: E402
from gpu_util import check_against_oracle, dev_bf16, expect_ok, host_f64, new_out  # noqa: E402

pytestmark = pytest.mark.gpu


def _with_workspace(a, b, M, N, K, out_f32, splits):
    ws = torch.empty(tp.tp_gemm_splitk_workspace_bytes(M, N, splits) // 4, dtype=torch.float32, device="cuda")
    c = new_out(M, N, out_f32)
    tp.tp_gemm_bf16_splitk(a, b, c, M, N, K, K, K, N, out_f32=out_f32, splits=splits, workspace=ws)
    expect_ok()
    assert tp.tp_last_plan()["splits"] == splits
    return host_f64(c)


def test_noalloc_matches_caller_workspace_on_two_calls_in_a_row():
    cases = [(128, 2048, 4096, True, 7), (300, 520, 1216, False, 4)]
    data = []
    for i, (M, N, K, out_f32, splits) in enumerate(cases):
        A, B = datagen.gemm_operands(M, N, K, seed=70 + i)
        data.append((A, B, dev_bf16(A), dev_bf16(B)))
    # Two calls in a row on the shared array, each plan read right after its
    # own call (the last-plan record keeps only the latest call), then the
    # checks.
    outs, plans = [], []
    for (M, N, K, out_f32, splits), (_, _, a, b) in zip(cases, data):
        c = new_out(M, N, out_f32)
        tp.tp_gemm_bf16_splitk_noalloc(a, b, c, M, N, K, K, K, N, out_f32=out_f32, splits=splits)
        plans.append(tp.tp_last_plan())
        outs.append(c)
    expect_ok()
    for (M, N, K, out_f32, splits), (A, B, a, b), c, plan in zip(cases, data, outs, plans):
        assert splits > 1 and plan["splits"] == splits, f"{M}x{N}x{K}: ran {plan['splits']} slices"
        got = host_f64(c)
        assert not np.isnan(got).any(), f"{M}x{N}x{K}: elements left unwritten"
        ref, ab = oracle.gemm(A, B, M, N, K, K, K)
        check_against_oracle(got, ref, ab, out_f32, f"no-alloc {M}x{N}x{K}")
        want = _with_workspace(a, b, M, N, K, out_f32, splits)
        assert np.array_equal(got, want), f"{M}x{N}x{K}: differs from the caller-workspace result"


def test_noalloc_chosen_slice_count_fits_the_array():
    # Skinny, deep K: the library splits K by itself (splits = 0) and must
    # pick a count whose partials fit the fixed array.
    M, N, K = 128, 8192, 16384
    A, B = datagen.gemm_operands(M, N, K, seed=72)
    a, b = dev_bf16(A), dev_bf16(B)
    c = new_out(M, N, False)
    tp.tp_gemm_bf16_splitk_noalloc(a, b, c, M, N, K, K, K, N, splits=0)
    plan = tp.tp_last_plan()
    expect_ok()
    sp = plan["splits"]
    assert sp >= 1
    if sp > 1:
        assert tp.tp_gemm_splitk_workspace_bytes(M, N, sp) <= tp.tp_gemm_splitk_noalloc_capacity()
    rows = oracle.sample_rows(M, 16)
    ref, ab = oracle.gemm(A, B, M, N, K, K, K, rows=rows)
    check_against_oracle(host_f64(c)[rows], ref, ab, False, f"no-alloc auto split ({sp} slices)")


def test_noalloc_rejects_requests_beyond_its_array():
    cap = tp.tp_gemm_splitk_noalloc_capacity()
    M, N, K = 1024, 4096, 8192
    splits = 8
    assert tp.tp_gemm_splitk_workspace_bytes(M, N, splits) > cap
    a = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    b = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
    c = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tp.TPError) as e:
        tp.tp_gemm_bf16_splitk_noalloc(a, b, c, M, N, K, K, K, N, splits=splits)
    assert e.value.status == tp.TP_ERR_WORKSPACE_LIMIT
