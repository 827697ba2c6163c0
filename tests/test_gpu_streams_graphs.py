"""The library under CUDA stream capture and on concurrent streams.

Every launch is asynchronous on the caller's stream and allocates nothing,
so a sequence of calls can be captured into a CUDA graph and replayed, and
calls on different streams run side by side. Checked bit for bit against
the same calls made eagerly on one stream (the same kernels in the same
order give identical bits)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import datagen  # noqa: E402
import mbarrier_pipelined_tensor_gb300 as tp  # noqa: E402
from gpu_util import dev_bf16, dev_u16, expect_ok  # noqa: E402

pytestmark = pytest.mark.gpu


def _problem(seed):
    M, N, K = 1000, 600, 1216
    A, B = datagen.gemm_operands(M, N, K, seed=seed)
    x, w = datagen.conv_operands(2, 20, 18, 64, 128, 3, 3, seed=seed + 1)
    src = datagen.copy_source(300, 1000, seed=seed + 2)
    # odd pitches: the plain-load producer's row-class windows
    Ao, Bo = datagen.gemm_operands(M, N, K, seed=seed + 3, lda=K + 1, ldb=K + 1)
    # 30 channels: the conv's row-class windows
    xo, wo = datagen.conv_operands(2, 20, 18, 30, 64, 3, 3, seed=seed + 4)
    return dict(M=M, N=N, K=K, a=dev_bf16(A), b=dev_bf16(B), x=dev_bf16(x), w=dev_bf16(w), src=dev_u16(src),
                ao=dev_bf16(Ao), bo=dev_bf16(Bo), xo=dev_bf16(xo), wo=dev_bf16(wo))


def _outputs(p):
    ws = torch.empty(tp.tp_gemm_splitk_workspace_bytes(128, p["N"], 4) // 4, dtype=torch.float32, device="cuda")
    return dict(c=torch.empty((p["M"], p["N"]), dtype=torch.float32, device="cuda"),
                c3=torch.empty((p["M"], p["N"]), dtype=torch.bfloat16, device="cuda"),
                c2=torch.empty((128, p["N"]), dtype=torch.bfloat16, device="cuda"),
                y=torch.empty((2 * 20 * 18, 128), dtype=torch.bfloat16, device="cuda"),
                yo=torch.empty((2 * 20 * 18, 64), dtype=torch.bfloat16, device="cuda"),
                dst=torch.empty_like(p["src"]), t=torch.empty((1000, 300), dtype=torch.int16, device="cuda"), ws=ws)


def _enqueue(p, o, stream):
    s = stream.cuda_stream
    M, N, K = p["M"], p["N"], p["K"]
    tp.tp_gemm_bf16_ex(p["a"], p["b"], o["c"], M, N, K, K, K, N, out_f32=True, stream=s)
    tp.tp_gemm_bf16_splitk(p["a"], p["b"], o["c2"], 128, N, K, K, K, N, splits=4, workspace=o["ws"], stream=s)
    tp.tp_gemm_bf16_ex(p["ao"], p["bo"], o["c3"], M, N, K, K + 1, K + 1, N, stream=s)
    tp.tp_conv2d_fprop_bf16_ex(p["x"], p["w"], o["y"], 2, 20, 18, 64, 128, 3, 3, 1, 1, stream=s)
    tp.tp_conv2d_fprop_bf16(p["xo"], p["wo"], o["yo"], 2, 20, 18, 30, 64, 3, 3, 1, 1, stream=s)
    tp.tp_tma_copy_2d(p["src"], o["dst"], 300, 1000, 1000, stream=s)
    tp.tp_tma_transpose_2d(p["src"], o["t"], 300, 1000, 1000, 300, stream=s)


def _same(o1, o2):
    for k in ("c", "c2", "c3", "y", "yo", "dst", "t"):
        assert torch.equal(o1[k], o2[k]), k


def test_graph_capture_and_replay_match_eager():
    p = _problem(101)
    eager = _outputs(p)
    s = torch.cuda.Stream()
    _enqueue(p, eager, s)                       # also loads every kernel before the capture
    s.synchronize()
    expect_ok()
    captured = _outputs(p)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _enqueue(p, captured, s)
    for _ in range(3):
        for v in captured.values():
            v.zero_()
        g.replay()
        torch.cuda.synchronize()
        expect_ok()
        _same(eager, captured)


def test_concurrent_streams_match_serial():
    probs = [_problem(200 + 10 * i) for i in range(3)]
    serial = [_outputs(p) for p in probs]
    s0 = torch.cuda.Stream()
    for p, o in zip(probs, serial):
        _enqueue(p, o, s0)
    s0.synchronize()
    streams = [torch.cuda.Stream() for _ in probs]
    conc = [_outputs(p) for p in probs]
    for _ in range(4):                          # all three streams in flight at once
        for p, o, st in zip(probs, conc, streams):
            _enqueue(p, o, st)
    torch.cuda.synchronize()
    expect_ok()
    for o1, o2 in zip(serial, conc):
        _same(o1, o2)


def test_concurrent_host_threads():
    # Four host threads call the library at once, each on its own stream
    # (ctypes releases the GIL, so planning, descriptor encoding and launches
    # really overlap). Every result equals the single-threaded one bit for bit.
    import threading
    cases = [(320, 200, 448, {}), (1000, 1000, 1000, {}), (512, 768, 640, dict(atom=2, tile_n=256)),
             (256, 512, 1024, dict(atom=1, tile_n=64))]
    data = []
    for i, (M, N, K, o) in enumerate(cases):
        A, B = datagen.gemm_operands(M, N, K, seed=300 + i)
        a, b = dev_bf16(A), dev_bf16(B)
        ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        tp.tp_gemm_bf16_ex(a, b, ref, M, N, K, K, K, N, **o)
        data.append((a, b, ref))
    torch.cuda.synchronize()
    expect_ok()
    errors = []

    def worker(i):
        try:
            M, N, K, o = cases[i]
            a, b, ref = data[i]
            c = torch.empty_like(ref)
            # The first call comes from a thread that has made no CUDA call
            # yet (no current context): encoding C's new tensor map must
            # still work.
            tp.tp_gemm_bf16_ex(a, b, c, M, N, K, K, K, N, **o)
            torch.cuda.current_stream().synchronize()
            st = torch.cuda.Stream()
            for _ in range(25):
                tp.tp_gemm_bf16_ex(a, b, c, M, N, K, K, K, N, stream=st, **o)
                plan = tp.tp_last_plan()   # this thread's own call
                assert (plan["m_tiles"], plan["k_blocks"]) == (-(-M // (128 * plan["atom"])), -(-K // 64))
            st.synchronize()
            if not torch.equal(c, ref):
                errors.append(f"case {i}: result differs from the single-threaded run")
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append(f"case {i}: {e!r}")

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    expect_ok()
