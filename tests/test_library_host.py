"""Host-side checks of libtp that need no GPU: the library loads and exports
every entry point include/tp.h declares, the shared-memory budget reproduces
the stage table of the "two-free-pipeline-stages" note, and the dispatch plan
(TMA suitability, tile counts, variant choice) is right."""
import os
import re

import pytest

import mbarrier_pipelined_tensor_gb300 as tp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tp.h")
GOLDEN = os.path.join(ROOT, "tests", "golden", "stage_budget.txt")
SM_COUNT = 152
SMEM_LIMIT = 232448
AL = 1 << 20  # a 16-byte aligned fake device address (nothing is launched)


def header_functions():
    text = open(HEADER).read()
    return re.findall(r"^TP_API\s+(?:const\s+char\s*\*|int64_t|int)\s+(tp_\w+)\(", text, flags=re.M)


def test_every_declared_symbol_is_exported():
    names = header_functions()
    assert len(names) >= 16
    for n in names:
        assert hasattr(tp._lib, n), n
    assert sorted(names) == sorted(tp.EXPORTED)


def test_status_strings():
    assert tp.tp_status_string(tp.TP_OK) == "TP_OK"
    assert tp.tp_status_string(tp.TP_ERR_SMEM_BUDGET) == "TP_ERR_SMEM_BUDGET"
    assert tp.tp_status_string(99) == "TP_ERR_UNKNOWN"


# ------------------------------------------------------ stage budget -----

def golden_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if line:
            atom, stages, val = line.split()
            rows.append((int(atom), int(stages), None if val == "FAIL" else int(val)))
    return rows


def page_stage_bytes(atom):
    # Tile 256x128x64 on a 2x1x1 cluster: a CTA's A fragment is 128x64 bf16;
    # the 1-SM atom holds the whole 128-row N-side tile, the 2-SM atom half.
    return 128 * 64 * 2 + (128 // atom) * 64 * 2


def test_golden_budget_table_is_consistent_arithmetic():
    rows = golden_rows()
    (a0, s0, b0) = rows[0]
    other = b0 - s0 * page_stage_bytes(a0)          # the other smem tenants
    assert other == 34816
    for atom, stages, val in rows:
        total = stages * page_stage_bytes(atom) + other
        if val is None:
            assert total > SMEM_LIMIT, (atom, stages, total)
        else:
            assert total == val and total <= SMEM_LIMIT


def test_library_budget_reproduces_page_depths():
    # Our kernel's other tenants differ from the page's, but the deepest ring
    # per atom, the failing depths and the identical budget at the deepest
    # ring come out the same.
    rows = golden_rows()
    fits = {}
    for atom in (1, 2):
        fits[atom] = [d for d in range(2, 12) if tp.tp_query_smem_bytes(atom, d, 128)[0] == tp.TP_OK]
    deepest = {a: max(fits[a]) for a in fits}
    for atom, stages, val in rows:
        if val is None:
            st, b = tp.tp_query_smem_bytes(atom, stages, 128)
            assert st == tp.TP_ERR_SMEM_BUDGET and b > SMEM_LIMIT
        else:
            assert deepest[atom] == stages
    b1 = tp.tp_query_smem_bytes(1, deepest[1], 128)[1]
    b2 = tp.tp_query_smem_bytes(2, deepest[2], 128)[1]
    assert b1 == b2 <= SMEM_LIMIT


def test_query_rejects_impossible():
    assert tp.tp_query_smem_bytes(3, 4, 128)[0] == tp.TP_ERR_INVALID_ARG
    assert tp.tp_query_smem_bytes(1, 4, 96)[0] == tp.TP_ERR_INVALID_ARG
    # 1-SM, N = 64: stages of 16 KiB A + 8 KiB B; 8 fit, 9 do not.
    assert tp.tp_query_smem_bytes(1, 8, 64) == (tp.TP_OK, 230656)
    assert tp.tp_query_smem_bytes(1, 9, 64)[0] == tp.TP_ERR_SMEM_BUDGET


def test_compiled_variants_match_budget():
    ks = tp.tp_list_kernels()
    assert len(ks) >= 20
    for k in ks:
        st, b = tp.tp_query_smem_bytes(k["atom"], k["pipe_depth"], k["tile_n"], k["out_f32"])
        # The plain-load producer adds staging buffers of a stage's rows
        # as 144-byte windows: the conv's with a 4-byte code per row, the
        # GEMM's (row-class windows by TMA) followed by their four barriers.
        rows = 128 + k["tile_n"] // k["atom"]
        if not k["ldg"]:
            staging = 0
        elif k["ldg"] == 2:        # the conv's row-class windows: 160-byte rows, a 16-byte record each
            staging = 3 * (rows * 160 + 16) + 64
        else:
            staging = 2 * rows * (144 + 4) if k["conv"] else 3 * rows * 144 + 64
        assert st == tp.TP_OK and b + staging == k["smem_bytes"], k
        assert k["smem_bytes"] <= SMEM_LIMIT
    sweep = {(k["atom"], k["pipe_depth"]) for k in ks if k["tile_n"] == 128 and not k["conv"] and not k["out_f32"]}
    assert {(1, d) for d in range(2, 7)} <= sweep
    assert {(2, d) for d in range(2, 9)} <= sweep
    n64 = {k["pipe_depth"] for k in ks if k["tile_n"] == 64 and not k["conv"] and not k["out_f32"]}
    assert set(range(2, 9)) <= n64
    # Every variant the planner may pick by itself has all four output forms
    # (bf16 / fp32 GEMM, bf16 / fp32 conv) and split-K at its deepest ring.
    have = {(k["atom"], k["tile_n"], k["pipe_depth"], k["out_f32"], k["conv"], k["splitk"]) for k in ks
            if not k["ldg"]}
    for atom, tile_n, d in ((2, 256, 6), (1, 256, 4), (2, 128, 8), (1, 128, 6), (1, 64, 8)):
        for form in ((0, 0, 0), (1, 0, 0), (0, 1, 0), (1, 1, 0), (1, 0, 1)):
            assert (atom, tile_n, d) + form in have, (atom, tile_n, d, form)


# ------------------------------------------------------------- plans -----

def plan(M, N, K, lda=None, ldb=None, ldc=None, A=AL, B=AL, C=AL, out_f32=False, **opts):
    lda = K if lda is None else lda
    ldb = K if ldb is None else ldb
    ldc = N if ldc is None else ldc
    return tp.tp_gemm_plan(A, B, C, M, N, K, lda, ldb, ldc, out_f32=out_f32, sm_count=SM_COUNT, **opts)


def test_plan_ragged_small_config():
    st, p = plan(320, 200, 448, atom=1, tile_n=128)
    assert st == tp.TP_OK and p["path"] == tp.TP_PATH_MAINLOOP
    assert (p["m_tiles"], p["n_tiles"], p["k_blocks"]) == (3, 2, 7)
    assert p["grid"] == 6 and p["smem_bytes"] <= SMEM_LIMIT
    st, p = plan(320, 200, 448, atom=2, tile_n=128)
    assert (p["m_tiles"], p["n_tiles"], p["grid"], p["cluster"]) == (2, 2, 8, 2)


def test_auto_variant_choice():
    # Large square: the 2-SM atom at MMA N = 256 (fewest waves x widest tile).
    st, p = plan(8192, 8192, 8192)
    assert (p["atom"], p["tile_n"], p["pipe_depth"]) == (2, 256, 6)
    # Few output tiles: 128 x 64 tiles spread the operand streams over twice
    # as many SMs (1000^3: 128 CTAs instead of 64), and a single wave of 1-SM
    # tiles avoids the cluster's fixed cost.
    st, p = plan(1000, 1000, 1000, lda=1008, ldb=1008, ldc=1000, out_f32=True)
    assert (p["atom"], p["tile_n"], p["pipe_depth"]) == (1, 64, 8) and p["grid"] == 128
    st, p = plan(128, 128, 64)
    assert (p["atom"], p["tile_n"], p["grid"]) == (1, 64, 2)
    # One row of tiles over a long K: 128 x 64 tiles give 128 CTAs (the
    # 2-SM atom would leave half of each pair's rows empty at M = 128).
    st, p = plan(128, 8192, 16384)
    assert (p["atom"], p["tile_n"], p["grid"]) == (1, 64, 128)
    # Mid-size: 1-SM, N = 256 tiles fill one wave.
    st, p = plan(2048, 2048, 2048)
    assert (p["atom"], p["tile_n"]) == (1, 256)
    # Several waves: the 2-SM atom's deeper ring wins.
    st, p = plan(2560, 2560, 2560)
    assert (p["atom"], p["tile_n"]) == (2, 256)
    # A fixed field restricts the choice.
    st, p = plan(8192, 8192, 8192, atom=1)
    assert (p["atom"], p["tile_n"], p["pipe_depth"]) == (1, 256, 4)
    st, p = plan(8192, 8192, 8192, tile_n=128)
    assert (p["atom"], p["tile_n"], p["pipe_depth"]) == (2, 128, 8)


def test_plan_big_square_grid_is_persistent():
    st, p = plan(8192, 8192, 8192)
    assert st == tp.TP_OK and p["grid"] == SM_COUNT
    st, p = plan(8192, 8192, 8192, atom=2, tile_n=256)
    assert st == tp.TP_OK and p["cluster"] == 2 and p["grid"] == SM_COUNT
    assert (p["m_tiles"], p["n_tiles"], p["k_blocks"]) == (32, 32, 128)


def test_plan_k_tiles_ragged():
    for K, kt in [(16, 1), (40, 1), (64, 1), (65, 2), (1000, 16), (1001, 16), (16384, 256)]:
        st, p = plan(128, 128, K, lda=(K + 7) // 8 * 8, ldb=(K + 7) // 8 * 8)
        assert st == tp.TP_OK and p["k_blocks"] == kt, K


def test_plan_edge_cases():
    assert plan(0, 5, 7)[0] == tp.TP_OK and plan(0, 5, 7)[1]["path"] == tp.TP_PATH_NONE
    st, p = plan(5, 7, 0, lda=8, ldb=8, ldc=8)
    assert st == tp.TP_OK and p["path"] == tp.TP_PATH_ZERO_FILL
    assert plan(-1, 5, 7)[0] == tp.TP_ERR_INVALID_ARG
    assert plan(4, 4, 16, lda=8)[0] == tp.TP_ERR_INVALID_ARG          # lda < K
    assert plan(4, 4, 16, ldc=2)[0] == tp.TP_ERR_INVALID_ARG          # ldc < N
    assert plan(4, 4, 16, A=0)[0] == tp.TP_ERR_INVALID_ARG            # NULL A


def test_plan_tma_suitability():
    FB, ML = tp.TP_PATH_FALLBACK_MAINLOOP, tp.TP_PATH_MAINLOOP
    assert plan(64, 64, 64, A=AL + 2)[1]["path"] == FB                # base not 16-B aligned
    assert plan(64, 64, 60, lda=60)[1]["path"] == FB                  # lda*2 = 120 not a multiple of 16
    assert plan(64, 60, 64, ldc=60, out_f32=True)[1]["path"] == ML    # 60*4 = 240 = 15*16
    assert plan(64, 60, 64, ldc=60)[1]["path"] == ML                  # 60*2 = 120: C by plain stores
    assert plan(64, 64, 64, C=AL + 2)[1]["path"] == ML                # C base: plain stores, TMA loads
    assert plan(64, 64, 64, B=AL + 2)[1]["path"] == FB
    st, p = plan(64, 64, 64, A=AL + 2)
    # the GEMM's three window staging buffers leave 2 ring stages
    assert st == tp.TP_OK and (p["atom"], p["tile_n"], p["pipe_depth"]) == (1, 128, 2)
    assert plan(64, 64, 64, A=AL + 1)[0] == tp.TP_ERR_INVALID_ARG     # a bf16 must be 2-byte aligned
    assert plan(64, 64, 64, C=AL + 2, out_f32=True)[0] == tp.TP_ERR_INVALID_ARG
    assert plan(64, 64, 64, A=AL + 2, atom=2)[0] == tp.TP_ERR_UNSUPPORTED


def test_plan_budget_errors():
    assert plan(256, 256, 256, atom=2, pipe_depth=9)[0] == tp.TP_ERR_SMEM_BUDGET
    assert plan(256, 256, 256, atom=1, tile_n=128, pipe_depth=7)[0] == tp.TP_ERR_SMEM_BUDGET
    assert plan(256, 256, 256, atom=1, tile_n=64, pipe_depth=9)[0] == tp.TP_ERR_SMEM_BUDGET
    st, p = plan(256, 256, 256, atom=1, tile_n=64, pipe_depth=8)
    assert st == tp.TP_OK and p["pipe_depth"] == 8
    assert plan(256, 256, 256, atom=1, tile_n=256, pipe_depth=5)[0] == tp.TP_ERR_SMEM_BUDGET
    assert plan(256, 256, 256, atom=3)[0] == tp.TP_ERR_INVALID_ARG
    st, p = plan(256, 256, 256, atom=2, pipe_depth=8)
    assert st == tp.TP_OK and p["pipe_depth"] == 8


def test_splitk_workspace_arithmetic():
    assert tp.tp_gemm_splitk_workspace_bytes(128, 8192, 4) == 4 * 128 * 8192 * 4
    assert tp.tp_gemm_splitk_workspace_bytes(300, 201, 3) == 3 * 300 * 204 * 4   # rows padded to 16 bytes
    with pytest.raises(tp.TPError):
        tp.tp_gemm_splitk_workspace_bytes(10, 10, 0)
    ks = [k for k in tp.tp_list_kernels() if k["splitk"]]
    assert {(k["atom"], k["tile_n"]) for k in ks} == {(1, 64), (1, 128), (1, 256), (2, 128), (2, 256)}
    assert all(k["out_f32"] == 1 and k["conv"] == 0 for k in ks)


def test_narrow_tail_plan():
    # 8192^3 on 152 SMs: 1024 pair tiles, 76 clusters, 36 left for the last
    # wave -> 72 half-width units (144 quarters would not fit one wave).
    st, p = plan(8192, 8192, 8192)
    assert (p["atom"], p["tile_n"], p["tail_units"], p["tail_parts"], p["grid"]) == (2, 256, 72, 2, 152)
    st, p = plan(8192, 8192, 8192, no_tail=1)
    assert p["tail_units"] == 0
    # A grid cap above the machine (non-persistent launch): the wave is still
    # the 76 clusters that run at once, so only the 36 leftover tiles split,
    # and each of the 988 + 72 units gets a cluster of its own.
    st, p = plan(8192, 8192, 8192, atom=2, tile_n=256, max_ctas=100000)
    assert (p["tail_units"], p["grid"]) == (72, 2 * 1060)
    # The conv's GEMM view, 392 tiles: 5 waves + 12, and 4 x 12 <= 76 -> 48
    # quarter-width units.
    st, p = plan(100352, 256, 2304, atom=2, tile_n=256, max_ctas=100000)
    assert (p["tail_units"], p["tail_parts"], p["grid"]) == (48, 4, 2 * 428)
    st, p = plan(100352, 256, 2304, atom=2, tile_n=256)
    assert (p["tail_units"], p["tail_parts"], p["grid"]) == (48, 4, 152)
    # 10 tiles on 4 clusters: 8 whole, 2 left -> 4 halves (8 quarters would not fit).
    st, p = plan(1280, 512, 640, atom=2, tile_n=256, max_ctas=8)
    assert (p["tail_units"], p["tail_parts"], p["grid"]) == (4, 2, 8)
    # No tail when the leftover does not fit twice into a wave, or for N = 128.
    st, p = plan(2048 * 5, 256 * 16, 512, atom=2, tile_n=256)     # 40 x 16 = 640 tiles: 640 % 76 = 32 fits
    assert p["tail_units"] == 64
    st, p = plan(256 * 70, 256, 512, atom=2, tile_n=256)          # 70 tiles < 76 clusters: all halves, 140 > 76
    assert p["tail_units"] == 0
    st, p = plan(8192, 8192, 8192, atom=2, tile_n=128)
    assert p["tail_units"] == 0


def test_no_tma_multicast_in_kernels():
    """The 2-SM atom feeds each CTA of the pair from its own TMA loads, which
    complete on the leader's barrier ("SM100_TMA_2SM_LOAD" semantics: each
    CTA loads its half, no multicast). No bulk-copy instruction in the kernel
    sources carries a cluster multicast; the one multicast token allowed is
    the tensor-core commit that signals both CTAs of the pair."""
    csrc = os.path.join(ROOT, "mbarrier_pipelined_tensor_gb300", "csrc")
    offenders = []
    for name in sorted(os.listdir(csrc)):
        if not name.endswith((".cu", ".cuh", ".cpp", ".h")):
            continue
        with open(os.path.join(csrc, name)) as f:
            for n, line in enumerate(f, 1):
                if "multicast" not in line:
                    continue
                if re.search(r"cp\.async\.bulk|\.tile::|im2col", line) or "tcgen05.commit" not in line:
                    offenders.append(f"{name}:{n}: {line.strip()}")
    assert not offenders, offenders


def test_l2_priority_choice():
    """Automatic L2 priorities: an operand read by at most two tile rows
    streams (evict-first) while the small, widely re-read one stays
    (evict-last); square problems keep normal priority."""
    def mode(M, N, K, **o):
        st, p = plan(M, N, K, **o)
        assert st == tp.TP_OK
        return p["l2_hint"]
    assert mode(128, 8192, 16384) == 2      # B streams, A (4 MB) stays
    assert mode(8192, 128, 16384) == 5      # mirrored
    assert mode(8192, 8192, 8192) == 1
    assert mode(4096, 4096, 512) == 1
    assert mode(128, 256, 64) == 1          # B not much bigger than A
    assert mode(128, 8192, 16384, l2_hint=1) == 1
    assert mode(8192, 8192, 8192, l2_hint=4) == 4
    assert mode(8192, 8192, 8192, l2_hint=7) == 7   # explicit evict_normal policy
    assert plan(128, 128, 128, l2_hint=8)[0] == tp.TP_ERR_INVALID_ARG


def test_convenience_wrappers_reject_bad_views():
    # The torch-facing wrappers take pitches from strides; views they cannot
    # describe are refused before anything reaches the library.
    torch = pytest.importorskip("torch")
    bf = torch.bfloat16
    A = torch.zeros(64, 32, dtype=bf)
    B = torch.zeros(48, 32, dtype=bf)
    C = torch.zeros(64, 48, dtype=bf)
    with pytest.raises(ValueError):
        tp.gemm(torch.zeros(32, 64, dtype=bf).t(), B, C)            # transposed A
    with pytest.raises(ValueError):
        tp.gemm(A, torch.zeros(48, 16, dtype=bf), C)                 # B of the wrong K
    with pytest.raises(ValueError):
        tp.gemm(A, B, torch.zeros(64, 40, dtype=bf))                 # C of the wrong N
    with pytest.raises(ValueError):
        tp.gemm(A.float(), B, C)                                     # fp32 operand
    x = torch.zeros(2, 8, 8, 16, dtype=bf)
    w = torch.zeros(32, 3, 3, 16, dtype=bf)
    with pytest.raises(ValueError):
        tp.conv2d_fprop(x, torch.zeros(32, 3, 3, 8, dtype=bf), torch.zeros(2, 8, 8, 32, dtype=bf), pad=1)
    with pytest.raises(ValueError):
        tp.conv2d_fprop(x.permute(0, 2, 1, 3), w, torch.zeros(2, 8, 8, 32, dtype=bf), pad=1)   # not NHWC-packed
    with pytest.raises(ValueError):
        tp.conv2d_fprop(x, w, torch.zeros(2, 6, 6, 32, dtype=bf), pad=1)                       # wrong P, Q


C_CONSUMER = r"""
#include <stdio.h>
#include "tp.h"
int main(void)
{
    tp_gemm_opts o = {0};
    tp_plan pl;
    int64_t b = 0;
    int st = tp_query_smem_bytes(2, 6, 256, 0, &b);
    printf("%d %lld %s\n", st, (long long)b, tp_status_string(st));
    st = tp_gemm_plan((void*)0x100000, (void*)0x100000, (void*)0x100000, 8192, 8192, 8192, 8192, 8192, 8192, 0,
                      &o, 152, &pl);
    printf("%d %d %d %d %d\n", st, pl.atom, pl.tile_n, pl.pipe_depth, pl.grid);
    return 0;
}
"""


def test_header_is_plain_c_and_links(tmp_path):
    # include/tp.h is a C header: a C99 program compiles against it without
    # warnings (-pedantic -Werror), links libtp.so and plans the 8192^3 GEMM
    # without a GPU.
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(tp.LIB_PATH)
    src = tmp_path / "consumer.c"
    src.write_text(C_CONSUMER)
    exe = tmp_path / "consumer"
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", f"-I{ROOT}/include", str(src),
                        f"-L{libdir}", "-ltp", f"-Wl,-rpath,{libdir}", "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    assert out.stdout.split("\n")[:2] == ["0 230656 TP_OK", "0 2 256 6 152"]
