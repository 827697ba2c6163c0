"""Pins for the CPU oracle, independent of the oracle's own formula.

Each case is fixed by mathematics, not by re-running the oracle: identity and
permutation operands, all-ones and rank-1 closed forms, exact rational
evaluation (``fractions``) on tiny inputs, numpy's matmul as a library
routine, and structural conv cases (delta filters, 1x1 = GEMM, tap counts at
the border). A dropped term, a wrong sign or index, a transposed operand or a
flipped filter fails at least one of them.
"""
from fractions import Fraction

import numpy as np
import pytest

import datagen
import oracle

ONE = np.uint16(0x3F80)  # bf16 1.0
ZERO = np.uint16(0)


def bf16(values) -> np.ndarray:
    """Exact fp32 values -> bf16 bits (values must be bf16-representable)."""
    v = np.asarray(values, dtype=np.float32)
    h = datagen.f32_to_bf16_rne(v)
    assert np.array_equal(datagen.bf16_to_f32(h), v), "value not exact in bf16"
    return h


def frac(h) -> Fraction:
    return Fraction(float(datagen.bf16_to_f32(np.uint16(h))))


def rand_bf16(shape, seed):
    return datagen.Stream(seed).uniform_bf16(shape)


def dyadic(shape, seed, lo=-64, hi=64):
    """Small integers / 64: every sum of a few products is exact in fp64."""
    r = datagen.splitmix64(seed, 0, int(np.prod(shape)))
    ints = (r % np.uint64(hi - lo + 1)).astype(np.int64) + lo
    return bf16(ints.astype(np.float32) / 64.0).reshape(shape)


# ----------------------------------------------------------------- GEMM -----

def test_left_identity_gives_b_transposed_view():
    M = K = 37
    N = 23
    A = np.where(np.eye(M, K, dtype=bool), ONE, ZERO).astype(np.uint16)
    B = rand_bf16((N, K), 11)                      # b(k, j) = B[j, k]
    ref, ab = oracle.gemm(A, B, M, N, K, K, K)
    expect = datagen.bf16_to_f32(B).astype(np.float64).T   # C[i][j] = b(i, j) = B[j, i]
    assert np.array_equal(ref, expect)
    assert np.array_equal(ab, np.abs(expect))


def test_right_identity_gives_a():
    M, N = 19, 41
    K = N
    A = rand_bf16((M, K), 12)
    B = np.where(np.eye(N, K, dtype=bool), ONE, ZERO).astype(np.uint16)
    ref, _ = oracle.gemm(A, B, M, N, K, K, K)
    assert np.array_equal(ref, datagen.bf16_to_f32(A).astype(np.float64))


def test_permutation_rows():
    M = K = 29
    N = 13
    perm = np.random.default_rng(5).permutation(K)
    A = np.zeros((M, K), dtype=np.uint16)
    A[np.arange(M), perm] = ONE                    # a(i, perm[i]) = 1
    B = rand_bf16((N, K), 13)
    ref, _ = oracle.gemm(A, B, M, N, K, K, K)
    expect = datagen.bf16_to_f32(B).astype(np.float64)[:, perm].T  # C[i][j] = b(perm[i], j)
    assert np.array_equal(ref, expect)


@pytest.mark.parametrize("K", [1, 7, 64, 1000, 16384])
def test_all_ones_sums_to_k(K):
    M, N = 5, 7
    A = np.full((M, K), ONE, dtype=np.uint16)
    B = np.full((N, K), ONE, dtype=np.uint16)
    ref, ab = oracle.gemm(A, B, M, N, K, K, K)
    assert np.all(ref == K) and np.all(ab == K)


def test_rank_one_closed_form():
    M, N, K = 9, 6, 448
    u = rand_bf16((M,), 21)
    v = rand_bf16((N,), 22)
    A = np.repeat(u[:, None], K, axis=1)
    B = np.repeat(v[:, None], K, axis=1)
    ref, _ = oracle.gemm(A, B, M, N, K, K, K)
    uf = datagen.bf16_to_f32(u).astype(np.float64)
    vf = datagen.bf16_to_f32(v).astype(np.float64)
    assert np.array_equal(ref, K * np.outer(uf, vf))


def test_signs_cancel():
    # a = [x, -x], b = [y, y]: sum is exactly 0, abs is 2|xy|.
    M, N, K = 3, 4, 2
    x = rand_bf16((M,), 31)
    y = rand_bf16((N,), 32)
    A = np.stack([x, x ^ np.uint16(0x8000)], axis=1)
    B = np.stack([y, y], axis=1)
    ref, ab = oracle.gemm(A, B, M, N, K, K, K)
    assert np.all(ref == 0.0)
    xf = datagen.bf16_to_f32(x).astype(np.float64)
    yf = datagen.bf16_to_f32(y).astype(np.float64)
    assert np.array_equal(ab, 2 * np.abs(np.outer(xf, yf)))


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (9, 2, 9), (4, 9, 8)])
def test_bruteforce_exact_rationals(M, N, K):
    A = dyadic((M, K), 40 + M)
    B = dyadic((N, K), 50 + N)
    ref, ab = oracle.gemm(A, B, M, N, K, K, K)
    for i in range(M):
        for j in range(N):
            terms = [frac(A[i, k]) * frac(B[j, k]) for k in range(K)]
            assert ref[i, j] == float(sum(terms, Fraction(0)))
            assert ab[i, j] == float(sum((abs(t) for t in terms), Fraction(0)))


def test_bruteforce_rationals_uniform_inputs():
    M, N, K = 6, 5, 9
    A = rand_bf16((M, K), 61)
    B = rand_bf16((N, K), 62)
    ref, _ = oracle.gemm(A, B, M, N, K, K, K)
    for i in range(M):
        for j in range(N):
            exact = sum((frac(A[i, k]) * frac(B[j, k]) for k in range(K)), Fraction(0))
            assert abs(Fraction(ref[i, j]) - exact) <= Fraction(1, 2 ** 50)


@pytest.mark.parametrize("M,N,K", [(320, 200, 448), (1, 300, 1000), (130, 7, 65)])
def test_matches_library_matmul(M, N, K):
    A, B = datagen.gemm_operands(M, N, K, seed=7)
    ref, ab = oracle.gemm(A, B, M, N, K, K, K)
    a = datagen.bf16_to_f32(A).astype(np.float64)
    b = datagen.bf16_to_f32(B).astype(np.float64)
    np.testing.assert_allclose(ref, a @ b.T, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ab, np.abs(a) @ np.abs(b).T, rtol=1e-13, atol=0)
    assert np.all(ab >= np.abs(ref))


def test_pitched_operands_ignore_padding():
    M, N, K = 33, 17, 70
    A, B = datagen.gemm_operands(M, N, K, seed=8)
    Ap, Bp = datagen.gemm_operands(M, N, K, seed=8, lda=88, ldb=80)
    ref, ab = oracle.gemm(A, B, M, N, K, K, K)
    refp, abp = oracle.gemm(Ap, Bp, M, N, K, 88, 80)
    assert np.array_equal(ref, refp) and np.array_equal(ab, abp)
    assert np.all(np.isfinite(refp))


def test_sampled_rows_cols_match_full():
    M, N, K = 100, 90, 80
    A, B = datagen.gemm_operands(M, N, K, seed=9)
    ref, ab = oracle.gemm(A, B, M, N, K, K, K)
    rows = np.array([0, 5, 99, 42])
    cols = np.array([89, 0, 3])
    r2, a2 = oracle.gemm(A, B, M, N, K, K, K, rows=rows, cols=cols)
    assert np.array_equal(r2, ref[np.ix_(rows, cols)])
    assert np.array_equal(a2, ab[np.ix_(rows, cols)])


def test_k_zero_is_zero():
    ref, ab = oracle.gemm(np.zeros(4, np.uint16), np.zeros(4, np.uint16), 2, 2, 0, 1, 1)
    assert np.all(ref == 0) and np.all(ab == 0)


def test_acceptance_rule():
    ref = np.array([1.0, -2.0, 0.0])
    ab = np.array([10.0, 2.0, 0.0])
    ok, _, _ = oracle.check(ref + np.array([0.0099, -0.0019, 0.0]), ref, ab, out_bf16=False)
    assert ok
    ok, _, nbad = oracle.check(ref + np.array([0.0102, 0.0, 0.0]), ref, ab, out_bf16=False)
    assert not ok and nbad == 1
    ok, _, _ = oracle.check(np.array([np.nan, -2.0, 0.0]), ref, ab, out_bf16=False)
    assert not ok


# bf16 outputs. ref = +-3 with sum|a*b| = 5: the fp32 bound is
# 1e-3 * 5 + 1e-6 = 0.005001 and half a bf16 ulp of the true value adds
# 2**-8 * 3 = 0.01171875, so the bf16 bound is 0.01671975 on either sign.
# A term of 2**-7 (0.0284385), a signed ref (0.005001 - 0.01171875 < 0 for
# ref = -3) or the term on fp32 outputs (0.01671975) each flips one of the
# accept / reject decisions below.
@pytest.mark.parametrize("ref", [3.0, -3.0])
def test_acceptance_bf16_bound_edges(ref):
    r = np.array([ref])
    ab = np.array([5.0])
    for sign in (1.0, -1.0):
        ok, _, _ = oracle.check(r + sign * 0.01671, r, ab, out_bf16=True)
        assert ok, f"ref {ref}: error 0.01671 is inside the bf16 bound 0.01671975"
        ok, _, nbad = oracle.check(r + sign * 0.01673, r, ab, out_bf16=True)
        assert not ok and nbad == 1, f"ref {ref}: error 0.01673 is outside the bf16 bound"


def test_acceptance_fp32_has_no_bf16_term():
    r = np.array([3.0, -3.0])
    ab = np.array([5.0, 5.0])
    ok, _, _ = oracle.check(r + 0.00500, r, ab, out_bf16=False)
    assert ok
    ok, _, nbad = oracle.check(r + np.array([0.00501, -0.00501]), r, ab, out_bf16=False)
    assert not ok and nbad == 2, "fp32 bound is 0.005001: no half-ulp term"


def test_acceptance_bf16_admits_rounding_of_a_close_fp32_result():
    # True value 1 + 2**-8 + 2**-20 (one product, so sum|a*b| = the value).
    # An fp32 result one ulp (2**-23) above it rounds (RNE) to the bf16
    # value 1 + 2**-7, an error of 2**-8 - 2**-20 - 2**-23 = 0.00390506;
    # the bf16 bound, 1e-3 * v + 1e-6 + 2**-8 * v = 0.00492646, admits it,
    # the fp32 bound (0.00100491) does not.
    v = 1.0 + 2.0 ** -8 + 2.0 ** -20
    near = np.array([v + 2.0 ** -23], dtype=np.float32)
    rounded = datagen.bf16_to_f32(datagen.f32_to_bf16_rne(near)).astype(np.float64)
    assert rounded[0] == 1.0 + 2.0 ** -7
    r, ab = np.array([v]), np.array([v])
    ok, _, _ = oracle.check(rounded, r, ab, out_bf16=True)
    assert ok
    ok, _, _ = oracle.check(rounded, r, ab, out_bf16=False)
    assert not ok


def test_acceptance_bf16_admits_a_tie_rounded_to_even():
    # 1 + 2**-8 lies halfway between the bf16 values 1 and 1 + 2**-7 and
    # rounds to the even one, 1: an error of exactly half an ulp (2**-8).
    # With a quarter-ulp term (2**-9 * v) the bound would be 0.00296794.
    v = 1.0 + 2.0 ** -8
    rounded = datagen.bf16_to_f32(datagen.f32_to_bf16_rne(np.array([v], dtype=np.float32)))
    assert rounded[0] == 1.0
    ok, worst, _ = oracle.check(rounded.astype(np.float64), np.array([v]), np.array([v]), out_bf16=True)
    assert ok and worst > 0.75, "a half-ulp error uses most of the bf16 bound"


# ----------------------------------------------------------------- conv -----

def conv_ref(x, w, N, H, W, C, K, R, S, st, pad):
    P, Q = oracle.conv_out_hw(H, W, R, S, st, pad)
    ref, ab = oracle.conv(x, w, N, H, W, C, K, R, S, st, pad)
    return ref.reshape(N, P, Q, K), ab.reshape(N, P, Q, K)


def test_conv_1x1_equals_gemm():
    N, H, W, C, K = 2, 5, 7, 24, 10
    x, w = datagen.conv_operands(N, H, W, C, K, 1, 1, seed=70)
    ref, _ = conv_ref(x, w, N, H, W, C, K, 1, 1, 1, 0)
    xf = datagen.bf16_to_f32(x).astype(np.float64).reshape(-1, C)
    wf = datagen.bf16_to_f32(w).astype(np.float64).reshape(K, C)
    np.testing.assert_allclose(ref.reshape(-1, K), xf @ wf.T, rtol=0, atol=1e-12)


def _delta_filter(K, R, S, C, r0, s0):
    w = np.zeros((K, R, S, C), dtype=np.uint16)
    for k in range(K):
        w[k, r0, s0, k] = ONE
    return w


def test_conv_centre_delta_is_identity():
    N, H, W, C = 2, 6, 5, 8
    x = rand_bf16((N, H, W, C), 71)
    ref, _ = conv_ref(x, _delta_filter(C, 3, 3, C, 1, 1), N, H, W, C, C, 3, 3, 1, 1)
    assert np.array_equal(ref, datagen.bf16_to_f32(x).astype(np.float64))


def test_conv_offset_delta_is_cross_correlation_shift():
    # Tap (r, s) = (0, 2) with pad 1 reads x[p - 1][q + 1]: catches a flipped
    # filter (true convolution), swapped r/s or a wrong pad sign.
    N, H, W, C = 1, 6, 7, 4
    x = rand_bf16((N, H, W, C), 72)
    ref, _ = conv_ref(x, _delta_filter(C, 3, 3, C, 0, 2), N, H, W, C, C, 3, 3, 1, 1)
    xf = datagen.bf16_to_f32(x).astype(np.float64)
    expect = np.zeros_like(xf)
    expect[:, 1:, :-1, :] = xf[:, :-1, 1:, :]
    assert np.array_equal(ref, expect)


def test_conv_stride_two_subsamples():
    N, H, W, C = 1, 9, 8, 3
    x = rand_bf16((N, H, W, C), 73)
    ref, _ = conv_ref(x, _delta_filter(C, 3, 3, C, 1, 1), N, H, W, C, C, 3, 3, 2, 1)
    xf = datagen.bf16_to_f32(x).astype(np.float64)
    assert ref.shape == (1, 5, 4, C)
    assert np.array_equal(ref, xf[:, 0::2, 0::2, :])


def test_conv_all_ones_counts_taps():
    N, H, W, C, K = 1, 6, 5, 16, 3
    x = np.full((N, H, W, C), ONE, dtype=np.uint16)
    w = np.full((K, 3, 3, C), ONE, dtype=np.uint16)
    ref, ab = conv_ref(x, w, N, H, W, C, K, 3, 3, 1, 1)
    rows = np.array([2] + [3] * (H - 2) + [2])
    cols = np.array([2] + [3] * (W - 2) + [2])
    taps = np.outer(rows, cols)                     # 4 corner, 6 edge, 9 interior
    assert taps[0, 0] == 4 and taps[0, 2] == 6 and taps[2, 2] == 9
    assert np.array_equal(ref[0, :, :, 0], C * taps.astype(np.float64))
    assert np.array_equal(ref, ab)


def test_conv_bruteforce_exact_rationals():
    N, H, W, C, K, R, S, st, pad = 2, 5, 4, 3, 2, 3, 2, 2, 1
    x = dyadic((N, H, W, C), 74)
    w = dyadic((K, R, S, C), 75)
    ref, _ = conv_ref(x, w, N, H, W, C, K, R, S, st, pad)
    P, Q = oracle.conv_out_hw(H, W, R, S, st, pad)
    assert (P, Q) == (3, 3)
    for n in range(N):
        for p in range(P):
            for q in range(Q):
                for k in range(K):
                    s_ = Fraction(0)
                    for r in range(R):
                        for s in range(S):
                            h, ww = p * st - pad + r, q * st - pad + s
                            if 0 <= h < H and 0 <= ww < W:
                                for c in range(C):
                                    s_ += frac(x[n, h, ww, c]) * frac(w[k, r, s, c])
                    assert ref[n, p, q, k] == float(s_)


def test_conv_sampled_pixels_match_full():
    N, H, W, C, K = 2, 7, 6, 8, 5
    x, w = datagen.conv_operands(N, H, W, C, K, 3, 3, seed=76)
    ref, ab = oracle.conv(x, w, N, H, W, C, K, 3, 3, 1, 1)
    pix = np.array([0, 41, 83, 17])
    r2, a2 = oracle.conv(x, w, N, H, W, C, K, 3, 3, 1, 1, pixels=pix)
    assert np.array_equal(r2, ref[pix]) and np.array_equal(a2, ab[pix])


# ------------------------------------------------------------ generators -----

def test_splitmix64_published_vector():
    # First outputs of SplitMix64 seeded with 0 (Vigna's reference code).
    r = datagen.splitmix64(0, 0, 3)
    assert [int(v) for v in r] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_splitmix64_chunked_equals_block():
    n = (1 << 22) + 12345
    a = datagen.splitmix64(9, 100, n)
    assert a[0] == datagen.splitmix64(9, 100, 1)[0]
    assert a[-1] == datagen.splitmix64(9, 100 + n - 1, 1)[0]


def test_bf16_rne_ties_to_even():
    x = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 1.0 + 2 ** -8 + 2 ** -20],
                 dtype=np.float32)
    got = datagen.bf16_to_f32(datagen.f32_to_bf16_rne(x))
    assert list(got) == [1.0, 1.0 + 2 ** -6, -1.0, 1.0 + 2 ** -7]


def test_uniform_range_and_normal_scale():
    s = datagen.Stream(1)
    u = datagen.bf16_to_f32(s.uniform_bf16((100000,)))
    assert u.min() >= -1.0 and u.max() <= 1.0 and abs(u.mean()) < 0.01
    z = datagen.bf16_to_f32(datagen.Stream(2).normal_bf16((100000,)))
    assert abs(z.std() - 0.02) < 0.001 and abs(z.mean()) < 0.001
