#!/usr/bin/env python3
"""Benchmark of the TMA-pipelined tcgen05 BF16 mainloop (libtp) on GB300.

A step is one BF16 GEMM C = A.B at M = N = K = 8192 (A row-major, B
column-major, N(0,1)*0.02 operands from seed 1, fp32 accumulation, bf16 C)
through the C ABI. `value` is TFLOP/s over exactly --steps steps timed with
CUDA events on the launching stream (inputs, 256 MiB, exceed the 129 MB L2).
The same run also measures the other rows of the path, each against its
roofline: the implicit-GEMM conv (32x56x56x256, 3x3, K 256), the 1 GiB TMA
copy (GB/s vs HBM), the skinny GEMM set and the small ragged GEMM.

Two JSON lines on stdout (rank 0): the full per-row record
({"bench_detail": ...}), then the bench line, which ends with a compact
per-row "summary". Multi-GPU (torchrun): every rank runs the
same problem on its own GPU (replicas: the path has no cross-GPU exchange);
value = all ranks' FLOPs / the slowest rank's time.

--impl reference times the CPU fp64 oracle (the only reference this path
has) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "BF16 GEMM/conv TFLOP/s and % of tensor peak; TMA copy GB/s vs HBM (1×GB300)"
WORKLOAD = "bf16 GEMM M=N=K={n}, A row-major / B col-major, N(0,1)*0.02 seed 1, fp32 accumulate, bf16 out"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1000 * 1000


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["tp", "reference"], default="tp")
    ap.add_argument("--no-rows", action="store_true", help="only the headline GEMM")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--sweep", action="store_true", help="(kept for old command lines: the PIPE_DEPTH x atom sweep "
                    "runs with the rows)")
    ap.add_argument("--atom", type=int, default=0)
    ap.add_argument("--tile-n", type=int, default=0)
    ap.add_argument("--depth", type=int, default=0)
    ap.add_argument("--size", type=int, default=8192, help="M = N = K of the timed GEMM")
    ap.add_argument("--group-m", type=int, default=0, help="tile raster group (0 = library default)")
    ap.add_argument("--l2-hint", type=int, default=0, help="operand L2 priorities (tp_gemm_opts.l2_hint)")
    ap.add_argument("--only", choices=["gemm", "conv", "copy", "transpose"], default=None,
                    help="time only this workload for --steps launches (for profiling)")
    ap.add_argument("--shape", type=str, default="", help="M,N,K for --only gemm (default: --size cubed)")
    ap.add_argument("--pitch", type=int, default=0,
                    help="row pitch of A and B in elements for --only gemm (0 = K, the packed layout)")
    ap.add_argument("--conv-n", type=int, default=32, help="conv batch for --only conv")
    ap.add_argument("--conv-c", type=int, default=256,
                    help="input channels for --only conv (not a multiple of 8: the plain-load producer)")
    ap.add_argument("--copy-rows", type=int, default=32768, help="rows (x 16384) for --only copy/transpose")
    ap.add_argument("--gsweep", type=str, default="",
                    help="comma-separated group_m[:l2_hint] values: time a --steps loop of each")
    ap.add_argument("--record-traffic", metavar="NCU_CSV", default=None,
                    help="no GPU: write profiles/traffic.json from an ncu --csv capture of the headline launch")
    ap.add_argument("--traffic-command", default="", help="the ncu command line recorded with --record-traffic")
    ap.add_argument("--launch-table", metavar="NCU_CSV", default=None,
                    help="no GPU: print per-kernel launches, total time and share of an ncu --csv launch list")
    return ap.parse_args()


# ------------------------------------------------------------ distributed --

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(backend: str):
    import torch.distributed as dist
    world, rank, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return dist


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def reduce_max(x: float, device=None) -> float:
    """Max of a float over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ misc ---

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash() -> str:
    """Hash of every library source (kernels and the dispatch that picks them)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mbarrier_pipelined_tensor_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from a committed ncu capture, if the kernel
    sources are unchanged since it was taken (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    e = rec.get(kernel)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- timing ---

def time_loop(torch, stream, fn, n):
    """Total ms of n back-to-back calls, CUDA events on `stream`."""
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(n):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def time_each_flushed(torch, stream, fn, n, flush_buf):
    """ms of one call after writing a buffer larger than L2: the trimmed
    mean (middle 80%) of max(n, 40) calls, and the fastest call.

    CUDA event timestamps on the GB300 machine advance in steps of ~2.05 us, so
    one call reads as one of the two multiples of the step around its true
    time, the nearer one more often. A median therefore snaps to the step
    lattice; the mean over many calls (whose start falls anywhere between
    two steps) recovers the value in between."""
    out = []
    for _ in range(max(n, 40)):
        flush_buf.fill_(1)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        out.append(e0.elapsed_time(e1))
    out.sort()
    k = len(out) // 10
    mid = out[k:len(out) - k]
    return sum(mid) / len(mid), out[0]


# -------------------------------------------------------------- workloads --

def gemm_inputs(torch, M, N, K, seed, dist_name):
    import numpy as np
    import datagen
    A, B = datagen.gemm_operands(M, N, K, seed=seed, dist=dist_name)
    a = torch.from_numpy(A.view(np.int16)).cuda().view(torch.bfloat16)
    b = torch.from_numpy(B.view(np.int16)).cuda().view(torch.bfloat16)
    return A, B, a, b


def e2e_pipelined(torch, tp, a_h, b_h, M, N, K, opts, steps, depth=3):
    """ms per step of `steps` end-to-end GEMMs through tp_gemm_bf16_host:
    every step uploads A and B from pinned host memory, runs the GEMM and
    downloads C. Steps go round-robin over `depth` streams, each with its
    own device buffers and host C, so that a step's download overlaps the
    next steps' uploads and GEMMs."""
    streams = [torch.cuda.Stream() for _ in range(depth)]
    dA = [torch.empty_like(a_h, device="cuda") for _ in range(depth)]
    dB = [torch.empty_like(b_h, device="cuda") for _ in range(depth)]
    dC = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(depth)]
    c_h = [torch.empty((M, N), dtype=torch.bfloat16).pin_memory() for _ in range(depth)]

    def run(n):
        for i in range(n):
            j = i % depth
            tp.tp_gemm_bf16_host(a_h, b_h, c_h[j], M, N, K, K, K, N, dA[j], dB[j], dC[j],
                                 stream=streams[j].cuda_stream, **opts)

    run(depth)
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    for st in streams:
        st.wait_stream(cur)
    run(steps)
    for st in streams:
        cur.wait_stream(st)
    e1.record(cur)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def role_timeline(torch, tp, launch):
    """One traced launch: per-role waiting shares averaged over CTAs (the
    MMA issuer's over pair leaders)."""
    launch(None)
    plan = tp.tp_last_plan()
    buf = torch.zeros(tp.TRACE_SLOTS * plan["grid"], dtype=torch.int64, device="cuda")
    launch(buf)
    torch.cuda.synchronize()
    t = buf.view(plan["grid"], tp.TRACE_SLOTS).double().cpu()
    mma = t[::plan["cluster"]]
    return {
        "producer_wait_empty_share": round(float((t[:, 1] / t[:, 0]).mean()), 3),
        "mma_wait_full_share": round(float((mma[:, 3] / mma[:, 2]).mean()), 3),
        "mma_wait_acc_empty_share": round(float((mma[:, 4] / mma[:, 2]).mean()), 3),
        "epilogue_wait_acc_full_share": round(float((t[:, 6] / t[:, 5]).mean()), 3),
        "mma_span_us": round(float(mma[:, 2].mean()) / 1e3, 2),
    }


def small_gemm_latency(torch, tp, stream, reps=50):
    """us per launch of small GEMMs issued back to back, eagerly and as
    one replayed CUDA graph of `reps` launches."""
    import numpy as np
    import datagen
    out = {"unit": "us per launch", "launches": reps}
    for (M, N, K, f32) in ((320, 200, 448, True), (1000, 1000, 1000, False), (4096, 4096, 512, False)):
        A, B = datagen.gemm_operands(M, N, K, seed=0)
        lda = (K + 7) // 8 * 8
        if lda != K:
            A, B = datagen.pad_rows(A, lda), datagen.pad_rows(B, lda)
        a = torch.from_numpy(A.view(np.int16)).cuda().view(torch.bfloat16)
        b = torch.from_numpy(B.view(np.int16)).cuda().view(torch.bfloat16)
        c = torch.empty((M, N), dtype=torch.float32 if f32 else torch.bfloat16, device="cuda")
        side = torch.cuda.Stream()

        def launch(st):
            tp.tp_gemm_bf16_ex(a, b, c, M, N, K, lda, lda, N, out_f32=f32, stream=st.cuda_stream)

        for _ in range(3):
            launch(side)
        side.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for _ in range(reps):
                launch(side)
        g.replay()
        torch.cuda.synchronize()
        eager_ms = time_loop(torch, stream, lambda: launch(stream), reps) / reps
        graph_ms = time_loop(torch, stream, g.replay, 5) / (5 * reps)
        out[f"{M}x{N}x{K}"] = {"eager_us": round(eager_ms * 1e3, 2), "graph_us": round(graph_ms * 1e3, 2)}
        del g
    return out


def measure_rows(torch, tp, stream, peaks, flush_buf):
    """The path's other rows, each with its own roofline."""
    import numpy as np
    import datagen
    rows = {}
    s = stream.cuda_stream
    # conv 32x56x56x256, 3x3, K 256 (x 51 MB fits L2: flushed between calls)
    N, H, W, C, K, R, S = 32, 56, 56, 256, 256, 3, 3
    x, w = datagen.conv_operands(N, H, W, C, K, R, S, seed=2)
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    wd = torch.from_numpy(w.view(np.int16)).cuda().view(torch.bfloat16)
    M = N * H * W
    y = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    flops = 2.0 * M * K * R * S * C

    def conv(**o):
        tp.tp_conv2d_fprop_bf16_ex(xd, wd, y, N, H, W, C, K, R, S, 1, 1, stream=s, **o)

    conv_res = {}
    for name, o in (("auto", {}), ("atom1_n128", dict(atom=1, tile_n=128)), ("atom2_n256", dict(atom=2, tile_n=256)),
                    ("atom2_n128", dict(atom=2, tile_n=128))):
        for _ in range(3):
            conv(**o)
        med, best = time_each_flushed(torch, stream, lambda: conv(**o), 20, flush_buf)
        plan = tp.tp_last_plan()
        conv_res[name] = {"us": round(med * 1e3, 2), "tflops": round(flops / (med * 1e-3) / 1e12, 1),
                          "frac_of_peak": round(flops / (med * 1e-3) / 1e12 / peaks["bf16_tflops"], 3),
                          "atom": plan["atom"], "tile_n": plan["tile_n"], "pipe_depth": plan["pipe_depth"]}
    conv_res["role_timeline"] = role_timeline(
        torch, tp, lambda tr: tp.tp_conv2d_fprop_bf16_ex(xd, wd, y, N, H, W, C, K, R, S, 1, 1, stream=s, trace=tr))
    rows["conv_32x56x56x256_3x3"] = {"unit": "TFLOP/s", "l2": "flushed between calls (trimmed mean of 40)", **conv_res}
    del xd, wd, y

    # TMA read stream of a 256 MiB operand (the skinny GEMM's B, 8192 x 16384):
    # the measured bound of a GEMM that streams B once, with the same write
    # flush before each timed call as the GEMM rows.
    rr, cc = 8192, 16384
    rbuf = torch.zeros((rr, cc), dtype=torch.int16, device="cuda")
    rd = lambda: tp.tp_tma_read_2d(rbuf, rr, cc, cc, stream=s)  # noqa: E731
    for _ in range(3):
        rd()
    med_r, _ = time_each_flushed(torch, stream, rd, 20, flush_buf)
    b2b_r = time_loop(torch, stream, rd, 20) / 20
    read_gbs = rr * cc * 2 / (med_r * 1e-3) / 1e9
    rows["tma_read_stream_256MiB"] = {"unit": "GB/s", "flushed_gbs": round(read_gbs, 1), "us_flushed": round(med_r * 1e3, 2),
                                      "b2b_gbs": round(rr * cc * 2 / (b2b_r * 1e-3) / 1e9, 1),
                                      "frac_of_hbm_copy": round(read_gbs / peaks["hbm_gbs"], 3),
                                      "plan": {k: tp.tp_last_plan()[k] for k in ("pipe_depth", "grid")}}
    del rbuf

    # skinny set (uniform seed 3)
    sk = {}
    for (Ms, Ns, Ks), (A, B) in zip(datagen.SKINNY_SHAPES, datagen.skinny_operands()):
        a = torch.from_numpy(A.view(np.int16)).cuda().view(torch.bfloat16)
        b = torch.from_numpy(B.view(np.int16)).cuda().view(torch.bfloat16)
        c = torch.empty((Ms, Ns), dtype=torch.bfloat16, device="cuda")

        def g():
            tp.tp_gemm_bf16(a, b, c, Ms, Ns, Ks, Ks, Ks, Ns, stream=s)

        for _ in range(3):
            g()
        med, best = time_each_flushed(torch, stream, g, 20, flush_buf)
        f = 2.0 * Ms * Ns * Ks
        byts = 2.0 * (Ms * Ks + Ns * Ks + Ms * Ns)
        tfl = f / (med * 1e-3) / 1e12
        bound = min(peaks["bf16_tflops"], f / byts * peaks["hbm_gbs"] * 1e9 / 1e12)
        # the same bound with the measured read stream in place of the copy peak
        read_bound = min(peaks["bf16_tflops"], f / byts * read_gbs * 1e9 / 1e12)
        row = {"us": round(med * 1e3, 2), "tflops": round(tfl, 1), "roofline_tflops": round(bound, 1),
               "frac": round(tfl / bound, 3), "read_bound_tflops": round(read_bound, 1),
               "read_frac": round(tfl / read_bound, 3), "grid": tp.tp_last_plan()["grid"]}
        row["role_timeline"] = role_timeline(
            torch, tp, lambda tr: tp.tp_gemm_bf16_ex(a, b, c, Ms, Ns, Ks, Ks, Ks, Ns, stream=s, trace=tr))
        # split-K with a caller workspace (slices chosen by the library)
        ws = torch.empty(tp.tp_gemm_splitk_workspace_bytes(Ms, Ns, 16) // 4, dtype=torch.float32, device="cuda")

        def gs():
            tp.tp_gemm_bf16_splitk(a, b, c, Ms, Ns, Ks, Ks, Ks, Ns, splits=0, workspace=ws, stream=s)

        for _ in range(3):
            gs()
        med_s, _ = time_each_flushed(torch, stream, gs, 20, flush_buf)
        pl = tp.tp_last_plan()
        tfl_s = f / (med_s * 1e-3) / 1e12
        row["splitk"] = {"us": round(med_s * 1e3, 2), "tflops": round(tfl_s, 1), "frac": round(tfl_s / bound, 3),
                         "read_frac": round(tfl_s / read_bound, 3),
                         "splits": pl["splits"], "grid": pl["grid"], "atom": pl["atom"], "tile_n": pl["tile_n"]}
        sk[f"{Ms}x{Ns}x{Ks}"] = row
        del a, b, c, ws
    rows["skinny_gemm_set"] = {"unit": "TFLOP/s", "l2": "flushed between calls (trimmed mean of 40)", **sk}

    # small ragged GEMM 320x200x448 (latency)
    A, B = datagen.gemm_operands(320, 200, 448, seed=0)
    a = torch.from_numpy(A.view(np.int16)).cuda().view(torch.bfloat16)
    b = torch.from_numpy(B.view(np.int16)).cuda().view(torch.bfloat16)
    c = torch.empty((320, 200), dtype=torch.float32, device="cuda")
    g = lambda: tp.tp_gemm_bf16_f32(a, b, c, 320, 200, 448, 448, 448, 200, stream=s)  # noqa: E731
    for _ in range(3):
        g()
    med, best = time_each_flushed(torch, stream, g, 50, flush_buf)
    rows["gemm_320x200x448_f32"] = {"unit": "us", "mean_us": round(med * 1e3, 2), "min_us": round(best * 1e3, 2)}
    # The floor of the flushed timing itself: a one-element kernel timed the
    # same way (events around the call, right after the L2 flush). Every
    # flushed row carries about this much that is not the measured kernel.
    tiny = torch.zeros(1, device="cuda")
    med, best = time_each_flushed(torch, stream, lambda: tiny.add_(1), 50, flush_buf)
    rows["flush_floor"] = {"unit": "us", "mean_us": round(med * 1e3, 2), "min_us": round(best * 1e3, 2),
                           "what": "a one-element torch kernel timed like the flushed rows"}

    # The same small GEMMs back to back: eager launches from Python against a
    # CUDA graph of the same launches (no host cost per call; consecutive
    # launches overlap their set-up through programmatic dependent launch).
    rows["small_gemm_launch_latency"] = small_gemm_latency(torch, tp, stream)

    # 1 GiB TMA copy (input 1 GiB >> L2: back to back)
    rr, cc = 32768, 16384
    src = torch.from_numpy(datagen.copy_source(rr, cc, seed=4).view(np.int16)).cuda()
    dst = torch.empty_like(src)
    cp = lambda: tp.tp_tma_copy_2d(src, dst, rr, cc, cc, stream=s)  # noqa: E731
    for _ in range(3):
        cp()
    n = 20
    ms = time_loop(torch, stream, cp, n) / n
    moved = 2.0 * rr * cc * 2
    gbs = moved / (ms * 1e-3) / 1e9
    rows["tma_copy_1GiB"] = {"unit": "GB/s", "gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 3),
                             "ms": round(ms, 4), "bit_exact": bool(torch.equal(src, dst))}
    del dst
    # 1 GiB TMA transpose of the same matrix (dst 16384 x 32768)
    dst = torch.empty((cc, rr), dtype=torch.int16, device="cuda")
    tr = lambda: tp.tp_tma_transpose_2d(src, dst, rr, cc, cc, rr, stream=s)  # noqa: E731
    for _ in range(3):
        tr()
    ms = time_loop(torch, stream, tr, n) / n
    gbs = moved / (ms * 1e-3) / 1e9
    rows["tma_transpose_1GiB"] = {"unit": "GB/s", "gbs": round(gbs, 1),
                                  "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 3), "ms": round(ms, 4),
                                  "bit_exact": bool(torch.equal(dst, src.t()))}
    del dst
    rows["fallback_paths"] = fallback_paths(torch, tp, stream, src, peaks)
    del src

    # dependent fma chains (RAW latency upper bound, SM cycles per link)
    probe = {}
    for kind, name in ((0, "ffma_f32"), (1, "dfma_f64")):
        res, cpl = tp.tp_probe_fma_latency(kind, 64 * 4096, 3.0, stream=s)
        probe[name] = {"cycles_per_link": round(cpl, 3), "exact": res == 3.0 + 64 * 4096}
    probe["pages_b200"] = {"ffma_f32": 4, "dfma_f64": 8}
    rows["fma_chain_latency"] = probe
    return rows


def fallback_paths(torch, tp, stream, src, peaks):
    """The paths taken where TMA cannot describe the operands: the
    vectorized copy and tile transpose (forced on the same 1 GiB matrix), and
    the plain-load producer feeding the tcgen05 mainloop (a 4096^3 GEMM whose
    odd pitches rule TMA out), next to the TMA producer on the same shape."""
    s = stream.cuda_stream
    rr, cc = src.shape
    moved = 2.0 * rr * cc * 2
    out = {}
    dst = torch.empty_like(src)
    cp = lambda: tp.tp_tma_copy_2d_ex(src, dst, rr, cc, cc, stream=s, force_vec=True)  # noqa: E731
    for _ in range(3):
        cp()
    ms = time_loop(torch, stream, cp, 20) / 20
    out["vec_copy_1GiB"] = {"unit": "GB/s", "gbs": round(moved / (ms * 1e-3) / 1e9, 1),
                            "vectorized_path": tp.tp_last_plan()["path"] == tp.TP_PATH_VEC_COPY,
                            "frac_of_hbm": round(moved / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 3),
                            "bit_exact": bool(torch.equal(src, dst))}
    del dst
    dst = torch.empty((cc, rr), dtype=torch.int16, device="cuda")
    tr = lambda: tp.tp_tma_transpose_2d_ex(src, dst, rr, cc, cc, rr, stream=s, force_vec=True)  # noqa: E731
    for _ in range(3):
        tr()
    ms = time_loop(torch, stream, tr, 20) / 20
    out["vec_transpose_1GiB"] = {"unit": "GB/s", "gbs": round(moved / (ms * 1e-3) / 1e9, 1),
                                 "tile_path": tp.tp_last_plan()["path"] == tp.TP_PATH_VEC_TRANSPOSE,
                                 "frac_of_hbm": round(moved / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 3),
                                 "bit_exact": bool(torch.equal(dst, src.t()))}
    del dst
    # The tile transpose where it is needed: odd pitches on both sides (rows
    # only 2-byte aligned), the same 32768 x 16384 elements.
    lds, ldd = cc + 1, rr + 1
    so = torch.empty((rr, lds), dtype=torch.int16, device="cuda")
    so[:, :cc].copy_(src)
    do = torch.empty((cc, ldd), dtype=torch.int16, device="cuda")
    tro = lambda: tp.tp_tma_transpose_2d(so, do, rr, cc, lds, ldd, stream=s)  # noqa: E731
    for _ in range(3):
        tro()
    ms = time_loop(torch, stream, tro, 20) / 20
    out["vec_transpose_1GiB_odd_pitches"] = {
        "unit": "GB/s", "gbs": round(moved / (ms * 1e-3) / 1e9, 1), "ld_src": lds, "ld_dst": ldd,
        "tile_path": tp.tp_last_plan()["path"] == tp.TP_PATH_VEC_TRANSPOSE,
        "frac_of_hbm": round(moved / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 3),
        "bit_exact": bool(torch.equal(do[:, :rr], src.t()))}
    del so, do
    M = N = K = 4096
    flops = 2.0 * M * N * K
    gen = torch.Generator(device="cuda").manual_seed(7)
    for name, ld in (("plain_load_producer_4096", K + 1), ("tma_producer_4096_same_variant", K)):
        a = (torch.randn(M * ld, device="cuda", generator=gen) * 0.02).bfloat16()
        b = (torch.randn(N * ld, device="cuda", generator=gen) * 0.02).bfloat16()
        c = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
        g = lambda: tp.tp_gemm_bf16_ex(a, b, c, M, N, K, ld, ld, N, stream=s, atom=1, tile_n=128)  # noqa: E731
        for _ in range(3):
            g()
        ms = time_loop(torch, stream, g, 20) / 20
        plan = tp.tp_last_plan()
        out[name] = {"unit": "TFLOP/s", "tflops": round(flops / (ms * 1e-3) / 1e12, 1), "lda": ld,
                     "path": "plain-load" if plan["path"] == tp.TP_PATH_FALLBACK_MAINLOOP else "tma",
                     "atom": plan["atom"], "tile_n": plan["tile_n"], "pipe_depth": plan["pipe_depth"]}
        del a, b, c
    # The conv where channels are not a multiple of 8: the plain-load
    # producer's row-class windows (stride 1, output the input's size).
    Nc, H, W, K = 32, 56, 56, 256
    for name, C in (("plain_load_conv_c250", 250), ("tma_conv_c256", 256)):
        x = (torch.randn(Nc * H * W * C, device="cuda", generator=gen) * 0.02).bfloat16()
        w = (torch.randn(K * 9 * C, device="cuda", generator=gen) * 0.02).bfloat16()
        y = torch.empty((Nc * H * W, K), device="cuda", dtype=torch.bfloat16)
        cv = lambda: tp.tp_conv2d_fprop_bf16(x, w, y, Nc, H, W, C, K, 3, 3, 1, 1, stream=s)  # noqa: E731
        for _ in range(3):
            cv()
        ms = time_loop(torch, stream, cv, 10) / 10
        plan = tp.tp_last_plan()
        out[name] = {"unit": "TFLOP/s", "tflops": round(2.0 * Nc * H * W * K * 9 * C / (ms * 1e-3) / 1e12, 1),
                     "C": C, "path": "plain-load" if plan["path"] == tp.TP_PATH_FALLBACK_MAINLOOP else "tma"}
        del x, w, y
    return out


def library_comparison(torch, stream, flush_buf, headline_step):
    """The same workloads through PyTorch's vendor-library kernels (cuBLAS for
    the GEMMs, cuDNN for the conv, PyTorch's own copy kernels), timed the same
    way as the rows above. Context only: none of it is on the library's path."""
    import numpy as np
    import datagen
    out = {"note": "torch.mm (cuBLAS), torch conv2d channels_last (cuDNN, benchmark mode), torch copy_; "
                   "same timing as the rows: flushed medians for GEMMs/conv, back-to-back for 1 GiB copies"}
    with torch.cuda.stream(stream):
        N, H, W, C, K, R, S = 32, 56, 56, 256, 256, 3, 3
        x, w = datagen.conv_operands(N, H, W, C, K, R, S, seed=2)
        # NHWC / KRSC bytes viewed as channels_last NCHW / KCRS tensors
        xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16).view(N, H, W, C).permute(0, 3, 1, 2)
        wd = torch.from_numpy(w.view(np.int16)).cuda().view(torch.bfloat16).view(K, R, S, C).permute(0, 3, 1, 2)
        flops = 2.0 * N * H * W * K * R * S * C
        prev = torch.backends.cudnn.benchmark
        torch.backends.cudnn.benchmark = True
        try:
            cv = lambda: torch.nn.functional.conv2d(xd, wd, padding=1)  # noqa: E731
            for _ in range(5):
                cv()
            med, _ = time_each_flushed(torch, stream, cv, 20, flush_buf)
        finally:
            torch.backends.cudnn.benchmark = prev
        out["conv_32x56x56x256_3x3"] = {"us": round(med * 1e3, 2), "tflops": round(flops / (med * 1e-3) / 1e12, 1)}
        del xd, wd
        for (Ms, Ns, Ks) in ((8192, 8192, 8192), (128, 8192, 16384), (4096, 4096, 512), (1000, 1000, 1000),
                             (320, 200, 448)):
            a = torch.randn(Ms, Ks, device="cuda").bfloat16()
            b = torch.randn(Ns, Ks, device="cuda").bfloat16()
            mm = lambda: torch.mm(a, b.t())  # noqa: E731
            for _ in range(5):
                mm()
            med, _ = time_each_flushed(torch, stream, mm, 20, flush_buf)
            f = 2.0 * Ms * Ns * Ks
            out[f"gemm_{Ms}x{Ns}x{Ks}"] = {"us": round(med * 1e3, 2), "tflops": round(f / (med * 1e-3) / 1e12, 1)}
            del a, b
        # this library's headline launch under the same flushed timing
        med, _ = time_each_flushed(torch, stream, headline_step, 20, flush_buf)
        out["gemm_8192x8192x8192_this_library"] = {"us": round(med * 1e3, 2),
                                                   "tflops": round(2.0 * 8192 ** 3 / (med * 1e-3) / 1e12, 1)}
        rr, cc = 32768, 16384
        src = torch.empty((rr, cc), dtype=torch.int16, device="cuda").random_(-32768, 32767)
        moved = 2.0 * rr * cc * 2
        for name, dst, fn in (("copy_1GiB", torch.empty_like(src), lambda d: d.copy_(src)),
                              ("transpose_1GiB", torch.empty((cc, rr), dtype=torch.int16, device="cuda"),
                               lambda d: d.copy_(src.t()))):
            for _ in range(3):
                fn(dst)
            ms = time_loop(torch, stream, lambda: fn(dst), 20) / 20
            out[name] = {"gbs": round(moved / (ms * 1e-3) / 1e9, 1), "ms": round(ms, 4)}
            del dst
        del src
    return out


def run_sweep(torch, tp, stream, a, b, c, M, N, K, peaks):
    out = []
    s = stream.cuda_stream
    for atom, tile_n, depths in ((1, 64, range(2, 10)), (1, 128, range(2, 8)), (2, 128, range(2, 10)),
                                 (1, 256, range(2, 6)), (2, 256, range(2, 8))):
        for d in depths:
            st, byts = tp.tp_query_smem_bytes(atom, d, tile_n)
            row = {"atom": atom, "tile_n": tile_n, "pipe_depth": d, "smem_bytes": byts}
            if st != tp.TP_OK:
                row["result"] = tp.tp_status_string(st)
                out.append(row)
                continue
            g = lambda: tp.tp_gemm_bf16_ex(a, b, c, M, N, K, K, K, N, stream=s, atom=atom, tile_n=tile_n,  # noqa
                                           pipe_depth=d)
            for _ in range(3):
                g()
            ms = time_loop(torch, stream, g, 20) / 20
            tfl = 2.0 * M * N * K / (ms * 1e-3) / 1e12
            row.update({"ms": round(ms, 4), "tflops": round(tfl, 1), "frac": round(tfl / peaks["bf16_tflops"], 3)})
            out.append(row)
    return out


def cpu_baseline(M, N, K, A, B, target_s=12.0):
    """The oracle as it stands, on a bounded sample of C's rows."""
    import numpy as np
    import oracle
    thr = max(1, oracle.threads())
    t0 = time.perf_counter()
    oracle.gemm(A, B, M, N, K, K, K, rows=np.arange(thr))   # one row per thread: calibrate
    dt = max(time.perf_counter() - t0, 1e-3)
    nrows = int(max(thr, min(M, thr * target_s / dt)))
    rows = np.linspace(0, M - 1, nrows).astype(np.int64)
    t0 = time.perf_counter()
    oracle.gemm(A, B, M, N, K, K, K, rows=rows)
    dt = time.perf_counter() - t0
    flops = 2.0 * nrows * N * K
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.threads(), "kind": "oracle",
            "sample": f"{nrows} of {M} rows of C (all {N} columns, K={K}), fp64 triple loop with sum|a*b|",
            "seconds": round(dt, 2)}


def row_oracle_timings(rows):
    """The oracle timed per row: the small configurations in full, the
    others on a sample of C's rows (conv: output pixels), reported as sampled
    MAC/s and the full problem's time extrapolated from it (labelled)."""
    import numpy as np
    import datagen
    import oracle

    def timed(fn):
        t0 = time.perf_counter()
        fn()
        return max(time.perf_counter() - t0, 1e-6)

    def entry(macs, full_macs, dt, sample):
        e = {"sample": sample, "macs": int(macs), "seconds": round(dt, 4),
             "gmac_per_s": round(macs / dt / 1e9, 3), "cores": oracle.threads()}
        if macs < full_macs:
            e["extrapolated_full_s"] = round(full_macs / (macs / dt), 2)
        return e

    thr = max(1, oracle.threads())
    out = {}
    if "gemm_320x200x448_f32" in rows:
        A, B = datagen.gemm_operands(320, 200, 448, seed=0)
        dt = timed(lambda: oracle.gemm(A, B, 320, 200, 448, 448, 448))
        out["gemm_320x200x448_f32"] = entry(320 * 200 * 448, 320 * 200 * 448, dt, "full")
    for (M, N, K), (A, B) in zip(datagen.SKINNY_SHAPES, datagen.skinny_operands()):
        key = f"{M}x{N}x{K}"
        full = M * N * K
        if full <= 2_000_000_000:
            dt = timed(lambda: oracle.gemm(A, B, M, N, K, K, K))
            out[key] = entry(full, full, dt, "full")
        else:
            r = np.linspace(0, M - 1, min(M, thr * 2)).astype(np.int64)
            dt = timed(lambda: oracle.gemm(A, B, M, N, K, K, K, rows=r))
            out[key] = entry(r.size * N * K, full, dt, f"{r.size} of {M} rows of C")
    Nb, H, W, C, K, R, S = 32, 56, 56, 256, 256, 3, 3
    x, w = datagen.conv_operands(Nb, H, W, C, K, R, S, seed=2)
    pix = np.linspace(0, Nb * H * W - 1, thr * 16).astype(np.int64)
    dt = timed(lambda: oracle.conv(x, w, Nb, H, W, C, K, R, S, 1, 1, pixels=pix))
    out["conv_32x56x56x256_3x3"] = entry(pix.size * K * R * S * C, Nb * H * W * K * R * S * C, dt,
                                         f"{pix.size} of {Nb * H * W} output pixels")
    return out


def summarize(value, achieved, peak, rows, sweep, peaks):
    """Compact per-row results for the end of the bench line: value, unit,
    fraction of its bound and the same-run vendor-library figure."""
    out = {"gemm_8192x8192x8192": {"tflops": round(value, 1), "frac": round(achieved / peak, 3)}}
    lib = (rows or {}).get("library_comparison", {})
    if "gemm_8192x8192x8192" in lib:
        out["gemm_8192x8192x8192"]["cublas_tflops"] = lib["gemm_8192x8192x8192"]["tflops"]
    if "gemm_8192x8192x8192_this_library" in lib:
        # the same launch timed as cuBLAS is (flushed, one call at a time)
        out["gemm_8192x8192x8192"]["flushed_tflops"] = lib["gemm_8192x8192x8192_this_library"]["tflops"]
    if rows:
        cv = rows.get("conv_32x56x56x256_3x3", {})
        if "auto" in cv:
            a = cv["auto"]
            out["conv_32x56x56x256_3x3"] = {
                "tflops": a["tflops"], "us": a["us"], "frac": a["frac_of_peak"],
                "variant": f"{a['atom']}/{a['tile_n']}/{a['pipe_depth']}",
                "cudnn_tflops": lib.get("conv_32x56x56x256_3x3", {}).get("tflops")}
        for key, r in rows.get("skinny_gemm_set", {}).items():
            if not isinstance(r, dict) or "tflops" not in r:
                continue
            e = {"tflops": r["tflops"], "us": r["us"], "frac": r["frac"], "bound_tflops": r["roofline_tflops"],
                 "cublas_tflops": lib.get(f"gemm_{key}", {}).get("tflops")}
            if r.get("read_bound_tflops", 0) < r["roofline_tflops"] and "read_frac" in r:
                e["read_bound_tflops"] = r["read_bound_tflops"]
                e["read_frac"] = r["read_frac"]
            sk = r.get("splitk")
            if sk and sk.get("splits", 1) > 1:
                e["splitk_tflops"] = sk["tflops"]
                e["splitk_frac"] = sk["frac"]
                if "read_frac" in e and "read_frac" in sk:
                    e["splitk_read_frac"] = sk["read_frac"]
                e["splits"] = sk["splits"]
            out[f"gemm_{key}"] = e
        sm = rows.get("gemm_320x200x448_f32")
        if sm:
            out["gemm_320x200x448_f32"] = {"us": sm["mean_us"],
                                           "cublas_us": lib.get("gemm_320x200x448", {}).get("us")}
        if "flush_floor" in rows:
            out["flush_floor_us"] = rows["flush_floor"]["mean_us"]
        for key, lk in (("tma_copy_1GiB", "copy_1GiB"), ("tma_transpose_1GiB", "transpose_1GiB")):
            r = rows.get(key)
            if r:
                out[key] = {"gbs": r["gbs"], "frac": r["frac_of_hbm"], "bit_exact": r["bit_exact"],
                            "torch_gbs": lib.get(lk, {}).get("gbs")}
        rs = rows.get("tma_read_stream_256MiB")
        if rs:
            out["tma_read_stream_256MiB"] = {"flushed_gbs": rs["flushed_gbs"], "b2b_gbs": rs["b2b_gbs"]}
        fb = rows.get("fallback_paths", {})
        if "vec_transpose_1GiB" in fb:
            out["tile_transpose_1GiB"] = {"gbs": fb["vec_transpose_1GiB"]["gbs"],
                                          "odd_pitches_gbs": fb.get("vec_transpose_1GiB_odd_pitches", {}).get("gbs")}
        if "plain_load_producer_4096" in fb:
            out["plain_load_producer_4096"] = {"tflops": fb["plain_load_producer_4096"]["tflops"],
                                               "tma_tflops": fb["tma_producer_4096_same_variant"]["tflops"]}
        if "plain_load_conv_c250" in fb:
            out["plain_load_conv_c250"] = {"tflops": fb["plain_load_conv_c250"]["tflops"],
                                           "tma_c256_tflops": fb.get("tma_conv_c256", {}).get("tflops")}
    if sweep:
        sw = {}
        for r in sweep:
            sw.setdefault(f"{r['atom']}/{r['tile_n']}", []).append(r.get("tflops"))
        out["depth_sweep_tflops"] = {"depths_from": 2, **sw}
    out["peaks"] = {"bf16_tflops": peaks["bf16_tflops"], "hbm_gbs": peaks["hbm_gbs"]}
    return out


# ----------------------------------------------------------------- arms ---

def reference_arm(args):
    import numpy as np
    import datagen
    world, rank, _ = dist_env()
    if world > 1 and rank != 0:
        return 0
    M = N = K = 8192
    # A bounded sample: the rows one step computes; B is drawn in full.
    A, B = datagen.gemm_operands(M, N, K, seed=1, dist="normal")
    import oracle
    per_step_rows = max(1, oracle.threads())  # one row of C per oracle thread
    # Each step is the same bounded sample: per_step_rows rows of C over
    # `ncols` columns spread across N, sized from one timed full-width step
    # so that --steps of them take about 100 s of CPU work.
    t0 = time.perf_counter()
    oracle.gemm(A, B, M, N, K, K, K, rows=np.arange(per_step_rows))
    t_full = time.perf_counter() - t0
    budget_s = 100.0
    ncols = N if args.steps * t_full <= budget_s else max(64, int(N * budget_s / (args.steps * t_full)) // 64 * 64)
    cols = np.arange(ncols) * (N // ncols)
    for _ in range(max(0, args.warmup)):
        oracle.gemm(A, B, M, N, K, K, K, rows=np.arange(per_step_rows), cols=cols)
    t0 = time.perf_counter()
    for i in range(args.steps):
        rows = (np.arange(per_step_rows) * 1021 + i * 7) % M
        oracle.gemm(A, B, M, N, K, K, K, rows=rows, cols=cols)
    dt = time.perf_counter() - t0
    flops = 2.0 * per_step_rows * ncols * K * args.steps
    v = flops / dt / 1e12
    sample = f"{per_step_rows} rows x {ncols} of {N} columns of C per step (K={K})"
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD.format(n=M), "M": M, "N": N, "K": K, "sample": sample,
                       "parallelism": f"cpu oracle, {oracle.threads()} threads"},
            "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": oracle.threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def only_arm(args):
    """One workload alone: --warmup then --steps launches, one short JSON line."""
    import numpy as np
    import torch
    import datagen
    import mbarrier_pipelined_tensor_gb300 as tp
    stream = torch.cuda.current_stream()
    s = stream.cuda_stream
    if args.only == "gemm":
        M, N, K = (int(v) for v in args.shape.split(",")) if args.shape else (args.size,) * 3
        ld = args.pitch or K
        if ld < K:
            raise SystemExit("--pitch must be at least K")
        A, B = datagen.gemm_operands(M, N, K, seed=3, lda=ld, ldb=ld)
        a = torch.from_numpy(A.view(np.int16)).cuda().view(torch.bfloat16)
        b = torch.from_numpy(B.view(np.int16)).cuda().view(torch.bfloat16)
        c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        o = {k: v for k, v in (("atom", args.atom), ("tile_n", args.tile_n), ("pipe_depth", args.depth)) if v}
        gemm = lambda: tp.tp_gemm_bf16_ex(a, b, c, M, N, K, ld, ld, N, stream=s, **o)  # noqa: E731
        flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")

        def fn():
            flush.fill_(1)     # every launch starts from operands in HBM, as in the bench rows
            gemm()
        work, unit = 2.0 * M * N * K / 1e12, "TFLOP/s (flush included)"
        workload = f"gemm {M}x{N}x{K} lda=ldb={ld}"
    elif args.only == "conv":
        N, H, W, C, K, R, S = args.conv_n, 56, 56, args.conv_c, 256, 3, 3
        x, w = datagen.conv_operands(N, H, W, C, K, R, S, seed=2)
        xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
        wd = torch.from_numpy(w.view(np.int16)).cuda().view(torch.bfloat16)
        y = torch.empty((N * H * W, K), dtype=torch.bfloat16, device="cuda")
        fn = lambda: tp.tp_conv2d_fprop_bf16(xd, wd, y, N, H, W, C, K, R, S, 1, 1, stream=s)  # noqa: E731
        work, unit = 2.0 * N * H * W * K * R * S * C / 1e12, "TFLOP/s"
        workload = f"conv {N}x56x56x{C} * 3x3x{C}, 256 filters, stride 1 pad 1"
    else:
        rr, cc = args.copy_rows, 16384
        src = torch.from_numpy(datagen.copy_source(rr, cc, seed=4).view(np.int16)).cuda()
        if args.only == "copy":
            dst = torch.empty_like(src)
            fn = lambda: tp.tp_tma_copy_2d(src, dst, rr, cc, cc, stream=s)  # noqa: E731
        else:
            dst = torch.empty((cc, rr), dtype=torch.int16, device="cuda")
            fn = lambda: tp.tp_tma_transpose_2d(src, dst, rr, cc, cc, rr, stream=s)  # noqa: E731
        work, unit = 2.0 * rr * cc * 2 / 1e9, "GB/s"
        workload = f"{args.only} {rr}x{cc} 2-byte elements"
    for _ in range(max(1, args.warmup)):
        fn()
    ms = time_loop(torch, stream, fn, args.steps) / args.steps
    st = tp.tp_device_status()
    print(json.dumps({"workload": workload, "value": round(work / (ms * 1e-3), 1), "unit": unit,
                      "ms_per_launch": round(ms, 4), "steps": args.steps, "status": st,
                      "plan": tp.tp_last_plan()}), flush=True)
    return 0 if st == tp.TP_OK else 1


def tp_arm(args):
    import numpy as np
    import torch
    if args.only:
        return only_arm(args)
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = dist_init("nccl")
    import mbarrier_pipelined_tensor_gb300 as tp
    peaks, peak_src = load_peaks()
    M = N = K = args.size
    A, B, a, b = gemm_inputs(torch, M, N, K, seed=1, dist_name="normal")
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    s = stream.cuda_stream
    opts = {k: v for k, v in (("atom", args.atom), ("tile_n", args.tile_n), ("pipe_depth", args.depth),
                              ("group_m", args.group_m), ("l2_hint", args.l2_hint)) if v}
    if args.gsweep:
        out = []
        for item in args.gsweep.split(","):
            g, _, h = item.partition(":")
            g, h = int(g), int(h or 0)
            o = dict(opts, group_m=g, l2_hint=h)
            fn = lambda: tp.tp_gemm_bf16_ex(a, b, c, M, N, K, K, K, N, stream=s, **o)  # noqa: E731
            for _ in range(5):
                fn()
            sampler = ClockSampler(local).start()
            ms = time_loop(torch, stream, fn, args.steps)
            clk = sampler.stop()
            out.append({"group_m": g, "l2_hint": h, "tflops": round(2.0 * M * N * K * args.steps / (ms * 1e-3) / 1e12, 1),
                        "ms_per_launch": round(ms / args.steps, 4), "sm_mhz": clk["sm_mhz"],
                        "reasons": clk["reasons"]})
        print(json.dumps({"gsweep": out, "size": M, "steps": args.steps}), flush=True)
        return 0

    def step():
        tp.tp_gemm_bf16_ex(a, b, c, M, N, K, K, K, N, stream=s, **opts)

    for _ in range(max(3, args.warmup)):
        step()
    st = tp.tp_device_status()
    if st != tp.TP_OK:
        raise RuntimeError(f"device status {tp.tp_status_string(st)} after warm-up")
    plan = tp.tp_last_plan()

    # ---- timed region: exactly --steps GEMMs
    sampler = ClockSampler(local).start() if rank == 0 else None
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop() if sampler else None
    ms_local = e0.elapsed_time(e1)
    ms = reduce_max(ms_local, device="cuda")
    st = tp.tp_device_status()
    if st != tp.TP_OK:
        raise RuntimeError(f"device status {tp.tp_status_string(st)} in the timed region")
    flop = 2.0 * M * N * K
    value = flop * args.steps * world / (ms * 1e-3) / 1e12
    per_launch_ms = ms_local / args.steps
    achieved = flop / (per_launch_ms * 1e-3) / 1e12
    # A seconds-long loop of launches runs under the power cap: its
    # denominator is the sustained cuBLAS figure; a short region uses burst.
    peak_kind = "bf16_tflops_sustained" if ms_local > 1000.0 else "bf16_tflops"
    peak = peaks[peak_kind]

    # ---- end to end through the C ABI with host buffers (tp_gemm_bf16_host)
    a_h = torch.from_numpy(A.view(np.int16)).view(torch.bfloat16).pin_memory()
    b_h = torch.from_numpy(B.view(np.int16)).view(torch.bfloat16).pin_memory()
    c_h = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))

    def e2e_step():
        tp.tp_gemm_bf16_host(a_h, b_h, c_h, M, N, K, K, K, N, a, b, c, stream=s, **opts)

    e2e_step()
    barrier()
    serial_ms = reduce_max(time_loop(torch, stream, e2e_step, e2e_steps) / e2e_steps, device="cuda")
    e2e_ms = reduce_max(e2e_pipelined(torch, tp, a_h, b_h, M, N, K, opts, e2e_steps), device="cuda")
    e2e_val = flop * world / (e2e_ms * 1e-3) / 1e12

    rows = sweep = None
    cpu = None
    timeline = role_timeline(torch, tp, lambda tr: tp.tp_gemm_bf16_ex(a, b, c, M, N, K, K, K, N, stream=s,
                                                                       trace=tr, **opts))
    if rank == 0 and not args.no_rows:
        flush_buf = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
        rows = measure_rows(torch, tp, stream, peaks, flush_buf)
        rows["library_comparison"] = library_comparison(torch, stream, flush_buf, step)
        del flush_buf
    if rank == 0 and not args.no_rows and args.size == 8192:
        sweep = run_sweep(torch, tp, stream, a, b, c, M, N, K, peaks)
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(M, N, K, A, B)
        if rows:
            for key, e in row_oracle_timings(rows).items():
                if key in rows:
                    rows[key]["cpu_oracle"] = e
                elif key in rows.get("skinny_gemm_set", {}):
                    rows["skinny_gemm_set"][key]["cpu_oracle"] = e

    if rank == 0:
        kname = "mainloop_kernel"
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD.format(n=M), "M": M, "N": N, "K": K, "inputs_exceed_l2": True,
                       "l2": "inputs (256 MiB) exceed L2; back-to-back launches",
                       "parallelism": f"replicas x{world}", "atom": plan["atom"], "tile_n": plan["tile_n"],
                       "pipe_depth": plan["pipe_depth"], "grid": plan["grid"]},
            "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                         "traffic": recorded_traffic(kname), "kernel": kname,
                         "peak_source": f"{peak_kind} of {peak_src} (timed region {ms_local / 1e3:.2f} s)",
                         "frac_of_burst": round(achieved / peaks["bf16_tflops"], 4),
                         "algorithmic_flop_per_launch": flop},
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_val, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": 2 * M * K * 2,
                    "d2h_bytes_per_step": M * N * 2, "steps": e2e_steps,
                    "how": "tp_gemm_bf16_host per step: upload of A and B from pinned host memory, GEMM, "
                           "download of C; steps round-robin over 3 streams with their own buffers, so "
                           "transfers of neighbouring steps overlap; the host link (measured 280 GB/s both "
                           "ways together) bounds it",
                    "serial_value": round(flop * world / (serial_ms * 1e-3) / 1e12, 2)},
            "clocks": clocks,
            "gpu_launches": args.steps,
            "role_timeline": timeline,
            # Last, so that the tail of stdout always shows every row.
            "summary": summarize(value, achieved, peak, rows, sweep, peaks),
        }
        # The full per-row record (role timelines, oracle timings, library
        # figures, the fallback paths) on a line of its own before the
        # bench line.
        print(json.dumps({"bench_detail": {"rows": rows, "sweep": sweep}}), flush=True)
        print(json.dumps(line), flush=True)
    if dist.is_initialized():
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------- ncu summaries --

_NCU_UNITS = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "Tbyte": 1e12,
              "nsecond": 1e-9, "ns": 1e-9, "usecond": 1e-6, "us": 1e-6, "msecond": 1e-3, "ms": 1e-3,
              "second": 1.0, "s": 1.0}


def ncu_csv_rows(path):
    """(launch id, kernel name, metric, value in bytes or seconds) for every
    metric row of an `ncu --csv` log."""
    import csv
    rows, hdr = [], None
    with open(path, newline="") as f:
        for r in csv.reader(f):
            if not r:
                continue
            if r[0] == "ID":
                hdr = r
                continue
            if hdr is None or len(r) != len(hdr):
                continue
            d = dict(zip(hdr, r))
            try:
                v = float(d["Metric Value"].replace(",", ""))
            except ValueError:
                continue
            rows.append((int(d["ID"]), d["Kernel Name"], d["Metric Name"],
                         v * _NCU_UNITS.get(d.get("Metric Unit", ""), 1.0)))
    return rows


def record_traffic(csv_path, command):
    """profiles/traffic.json from the last captured mainloop launch."""
    per = {}
    for lid, name, metric, v in ncu_csv_rows(csv_path):
        if "mainloop_kernel" in name:
            per.setdefault(lid, {"name": name})[metric] = v
    if not per:
        raise SystemExit(f"no mainloop_kernel launch in {csv_path}")
    e = per[max(per)]
    rd, wr = e["dram__bytes_read.sum"], e["dram__bytes_write.sum"]
    rec = {"mainloop_kernel": {
        "source_hash": kernel_source_hash(),
        "dram_bytes_per_launch": int(round(rd + wr)),
        "dram_bytes_read": int(round(rd)),
        "dram_bytes_write": int(round(wr)),
        "duration_us": round(e.get("gpu__time_duration.sum", 0.0) * 1e6, 2),
        "variant": e["name"].split("(")[0].replace("void ", ""),
        "workload": "bf16 GEMM 8192^3 (bench.py default headline)",
        "command": command,
        "passes": 1}}
    path = os.path.join(ROOT, "profiles", "traffic.json")
    with open(path, "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")
    print(json.dumps(rec))


def launch_table(csv_path):
    """Markdown table: launches, total device time and share per kernel."""
    tot = {}
    cnt = {}
    for _, name, metric, v in ncu_csv_rows(csv_path):
        if metric != "gpu__time_duration.sum":
            continue
        k = name.split("(")[0].replace("void ", "")
        tot[k] = tot.get(k, 0.0) + v
        cnt[k] = cnt.get(k, 0) + 1
    total = sum(tot.values()) or 1.0
    print("| launches | total ms | share | kernel |")
    print("|---:|---:|---:|---|")
    for k in sorted(tot, key=lambda x: -tot[x]):
        print(f"| {cnt[k]} | {tot[k] * 1e3:.3f} | {100.0 * tot[k] / total:.2f}% | `{k}` |")


def main():
    args = parse_args()
    if args.record_traffic:
        record_traffic(args.record_traffic, args.traffic_command)
        return 0
    if args.launch_table:
        launch_table(args.launch_table)
        return 0
    if args.impl == "reference":
        return reference_arm(args)
    return tp_arm(args)


if __name__ == "__main__":
    sys.exit(main())
