"""The stage ring's protocol checked on the device ("B200 Tma Pipeline
Designer", step 8: every ready / free barrier has exactly one producer and
one consumer) and the MMA side of the lost-completion failure (its Failure
modes).

Arrival accounting (tp_gemm_opts.protocol) counts, per CTA, every arrival the
real kernel issues on each barrier in each phase, and the transaction bytes
each full-barrier phase expects and receives. The counts must equal those
of the CPU protocol model (tests/test_pipeline_protocol.py) run over the
same work units: one arrival per full / empty / acc_full phase, one per
epilogue warp of the pair per acc_empty phase, no arrival in a phase the
schedule does not reach, and expected bytes equal to the bytes of the loads
issued into that phase. The skipped-commit self tests make the MMA issuer
drop one tcgen05.commit; the waits behind it must give up with a status and
the next GEMM must match the oracle.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import datagen  # noqa: E402
import oracle  # noqa: E402
import mbarrier_pipelined_tensor_gb300 as tp  # noqa: E402
from gpu_util import check_against_oracle, dev_bf16, expect_ok, host_f64, new_out  # noqa: E402
from test_pipeline_protocol import simulate  # noqa: E402

pytestmark = pytest.mark.gpu

P = tp.PROTO_PHASES
S = tp.PROTO_MAX_STAGES
A_BYTES = 128 * 64 * 2
LDG_WARPS = 8  # producer warps of the plain-load producer


def expected_counts(plan, tma=True):
    """Arrivals and bytes per CTA, barrier and phase, from the CPU model run
    over each cluster's work units (units u = c, c + clusters, ...)."""
    CG, D, grid, KB = plan["cluster"], plan["pipe_depth"], plan["grid"], plan["k_blocks"]
    tiles = plan["m_tiles"] * plan["n_tiles"]
    tail = plan["tail_units"]
    parts = plan["tail_parts"] or 1
    n_full = tiles - tail // parts if tail else tiles
    num_units = n_full + tail if tail else tiles
    clusters = grid // CG
    b_bytes = plan["tile_n"] // CG * 64 * 2
    exp = np.zeros((grid, tp.PROTO_SLOTS), dtype=np.int64)
    for c in range(clusters):
        units = list(range(c, num_units, clusters))
        if not units:
            continue
        assert len(units) * KB < P * D, "case exceeds the counted phases"
        bars = {}
        simulate(CG, D, list(range(len(units))), KB, seed=c, out=bars)
        lead = c * CG
        for s in range(D):
            for k, who in enumerate(bars["full"][0][s].done):
                # the plain-load producer's warps each arrive once per phase
                exp[lead, s * P + k] = len(who) * (1 if tma else LDG_WARPS)
            for r in range(CG):
                for k, who in enumerate(bars["empty"][r][s].done):
                    exp[lead + r, (S + s) * P + k] = len(who)
        for b in range(2):
            for r in range(CG):
                for k, who in enumerate(bars["accf"][r][b].done):
                    exp[lead + r, (2 * S + b) * P + k] = len(who)
            for k, who in enumerate(bars["acce"][0][b].done):
                exp[lead, (2 * S + 2 + b) * P + k] = len(who)
        if tma:
            for it in range(len(units) * KB):
                s, k = it % D, it // D
                narrow = tail > 0 and units[it // KB] >= n_full
                nbytes = CG * (A_BYTES + (b_bytes // parts if narrow else b_bytes))
                exp[lead, tp.PROTO_TX_EXPECT + s * P + k] = nbytes
                exp[lead, tp.PROTO_TX_ISSUED + s * P + k] = nbytes
    return exp


def check_counts(got, exp, plan):
    bad = np.argwhere(got != exp)
    if bad.size:
        cta, slot = bad[0]
        raise AssertionError(f"{bad.shape[0]} counters differ; first: CTA {cta} slot {slot} "
                             f"(barrier {slot // P}, phase {slot % P}): device {got[cta, slot]}, "
                             f"model {exp[cta, slot]}; plan {plan}")


def counted(launch):
    """Runs `launch(protocol=buf)` once uncounted (for the plan), then counted."""
    launch(protocol=None)
    plan = tp.tp_last_plan()
    buf = torch.zeros(plan["grid"] * tp.PROTO_SLOTS, dtype=torch.int32, device="cuda")
    launch(protocol=buf)
    expect_ok()
    assert tp.tp_last_plan() == plan
    return buf.view(plan["grid"], tp.PROTO_SLOTS).cpu().numpy().view(np.uint32).astype(np.int64), plan


GEMM_VARIANTS = [(1, 128, 2, 4), (1, 128, 6, 4), (1, 64, 8, 4), (1, 256, 4, 4), (2, 128, 2, 4), (2, 128, 6, 4),
                 (2, 128, 8, 4), (2, 256, 2, 8), (2, 256, 6, 8), (2, 256, 6, 0)]


@pytest.mark.parametrize("atom,tile_n,depth,ctas", GEMM_VARIANTS)
def test_gemm_arrivals_match_the_model(atom, tile_n, depth, ctas):
    # Ragged M, N and K (16 k-blocks, the last 40 deep); a small grid so that
    # each CTA runs several units and wraps the ring many times. The 2-SM,
    # N = 256 cases end in narrow units: 6 pair tiles on 4 clusters in
    # halves, on the whole GPU in quarters.
    M, N, K = 300, 520, 1000
    A, B = datagen.gemm_operands(M, N, K, seed=110)
    a, b = dev_bf16(A), dev_bf16(B)
    c = new_out(M, N, False)

    def launch(protocol):
        tp.tp_gemm_bf16_ex(a, b, c, M, N, K, K, K, N, atom=atom, tile_n=tile_n, pipe_depth=depth,
                           max_ctas=ctas, protocol=protocol)

    got, plan = counted(launch)
    assert (plan["atom"], plan["tile_n"], plan["pipe_depth"]) == (atom, tile_n, depth)
    if (atom, tile_n) == (2, 256):
        assert plan["tail_units"] > 0
    check_counts(got, expected_counts(plan), plan)
    ref, ab = oracle.gemm(A, B, M, N, K, K, K)
    check_against_oracle(host_f64(c), ref, ab, False, "counted launch")


@pytest.mark.parametrize("atom,tile_n", [(1, 128), (1, 256), (2, 128), (2, 256)])
def test_conv_arrivals_match_the_model(atom, tile_n):
    Nb, H, W, C, K, R, Sf = 2, 12, 12, 128, 256, 3, 3
    x, w = datagen.conv_operands(Nb, H, W, C, K, R, Sf, seed=111)
    xd, wd = dev_bf16(x), dev_bf16(w)
    M = Nb * H * W
    y = new_out(M, K, False)

    def launch(protocol):
        tp.tp_conv2d_fprop_bf16_ex(xd, wd, y, Nb, H, W, C, K, R, Sf, 1, 1, atom=atom, tile_n=tile_n,
                                   max_ctas=2 * atom, protocol=protocol)

    got, plan = counted(launch)
    assert plan["conv"] == 1 and plan["k_blocks"] == 18
    check_counts(got, expected_counts(plan), plan)
    ref, ab = oracle.conv(x, w, Nb, H, W, C, K, R, Sf, 1, 1)
    check_against_oracle(host_f64(y), ref, ab, False, "counted conv")


def test_plain_load_producer_arrivals_match_the_model():
    # Odd pitches rule TMA out: one plain arrival per producer warp and full
    # phase, no bytes.
    M, N, K, ld = 300, 520, 1000, 1001
    A, B = datagen.gemm_operands(M, N, K, seed=112)
    A, B = datagen.pad_rows(A, ld), datagen.pad_rows(B, ld)
    a, b = dev_bf16(A), dev_bf16(B)
    c = new_out(M, N, True)

    def launch(protocol):
        tp.tp_gemm_bf16_ex(a, b, c, M, N, K, ld, ld, N, out_f32=True, max_ctas=4, protocol=protocol)

    got, plan = counted(launch)
    assert plan["path"] == tp.TP_PATH_FALLBACK_MAINLOOP
    check_counts(got, expected_counts(plan, tma=False), plan)
    ref, ab = oracle.gemm(A, B, M, N, K, ld, ld)
    check_against_oracle(host_f64(c), ref, ab, True, "counted plain-load launch")


@pytest.mark.parametrize("which,sites", [(1, (1, 2, 4)), (2, (3, 4))])
@pytest.mark.parametrize("atom", [1, 2])
def test_mainloop_skipped_commit_times_out_and_recovers(which, sites, atom):
    # which 1: no commit to empty[0] after the first k-block, so stage 0 is
    # never handed back (K = 1024: 16 k-blocks, more than any ring's stages).
    # which 2: no commit to acc_full after the first tile.
    M, N, K = 256, 256, 1024
    A, B = datagen.gemm_operands(M, N, K, seed=113)
    a, b = dev_bf16(A), dev_bf16(B)
    c = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    tp.tp_selftest_mainloop_skipped_commit(a, b, c, M, N, K, which, atom, 200)
    st, site, block, thread = tp.tp_device_status_detail()
    assert st == tp.TP_ERR_TIMEOUT and site in sites, (st, site)
    assert tp.tp_device_status() == tp.TP_OK
    c2 = new_out(M, N, True)
    tp.tp_gemm_bf16_ex(a, b, c2, M, N, K, K, K, N, out_f32=True, atom=atom, tile_n=128)
    expect_ok()
    ref, ab = oracle.gemm(A, B, M, N, K, K, K)
    check_against_oracle(host_f64(c2), ref, ab, True, "after the skipped-commit self test")


def test_skipped_commit_rejects_bad_arguments():
    a = torch.zeros(64 * 64, dtype=torch.bfloat16, device="cuda")
    c = torch.zeros(64 * 64, dtype=torch.float32, device="cuda")
    for which, atom in ((0, 1), (3, 1), (1, 3)):
        with pytest.raises(tp.TPError) as e:
            tp.tp_selftest_mainloop_skipped_commit(a, a, c, 64, 64, 64, which, atom, 100)
        assert e.value.status == tp.TP_ERR_INVALID_ARG
