"""Python binding of libtp, the TMA-pipelined tcgen05 BF16 mainloop library.

Argument marshalling only: every entry point passes raw device pointers,
sizes and a CUDA stream handle to the C ABI declared in include/tp.h, and
raises TPError on a non-zero status. Tensors (anything with ``data_ptr()``)
or plain integers are accepted as pointers. PyTorch, when present, only
supplies device memory and the current stream.

There is no fallback: if libtp.so has not been built, importing the package
raises. Build it with ``mbarrier_pipelined_tensor_gb300.build.build()`` (or
``__graft_entry__.build()`` at the repository root).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtp.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libtp.so is not built ({LIB_PATH}); run mbarrier_pipelined_tensor_gb300.build.build() first")

_lib = ctypes.CDLL(LIB_PATH)

TP_OK = 0
TP_ERR_INVALID_ARG = 1
TP_ERR_UNSUPPORTED = 2
TP_ERR_CUDA = 3
TP_ERR_DRIVER_ENCODE = 4
TP_ERR_TIMEOUT = 5
TP_ERR_SMEM_BUDGET = 6
TP_ERR_WORKSPACE_LIMIT = 7

TP_PATH_NONE = 0
TP_PATH_MAINLOOP = 1
TP_PATH_ZERO_FILL = 2
TP_PATH_TMA_COPY = 3
TP_PATH_VEC_COPY = 4
TP_PATH_FALLBACK_MAINLOOP = 5
TP_PATH_TMA_TRANSPOSE = 6
TP_PATH_VEC_TRANSPOSE = 7
TP_PATH_TMA_READ = 8


class tp_gemm_opts(ctypes.Structure):
    _fields_ = [("atom", ctypes.c_int), ("pipe_depth", ctypes.c_int), ("tile_n", ctypes.c_int),
                ("group_m", ctypes.c_int), ("max_ctas", ctypes.c_int), ("l2_hint", ctypes.c_int),
                ("no_tail", ctypes.c_int), ("trace", ctypes.c_void_p), ("events", ctypes.c_void_p),
                ("protocol", ctypes.c_void_p)]


class tp_copy_opts(ctypes.Structure):
    _fields_ = [("box_cols", ctypes.c_int), ("box_rows", ctypes.c_int), ("stages", ctypes.c_int),
                ("ctas_per_sm", ctypes.c_int), ("force_vec", ctypes.c_int)]


class tp_plan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("atom", ctypes.c_int), ("pipe_depth", ctypes.c_int),
                ("tile_n", ctypes.c_int), ("out_f32", ctypes.c_int), ("conv", ctypes.c_int),
                ("grid", ctypes.c_int), ("cluster", ctypes.c_int), ("smem_bytes", ctypes.c_int),
                ("m_tiles", ctypes.c_int64), ("n_tiles", ctypes.c_int64), ("k_blocks", ctypes.c_int64),
                ("splits", ctypes.c_int), ("tail_units", ctypes.c_int),
                ("l2_hint", ctypes.c_int), ("tail_parts", ctypes.c_int)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class tp_kernel_desc(ctypes.Structure):
    _fields_ = [("atom", ctypes.c_int), ("pipe_depth", ctypes.c_int), ("tile_n", ctypes.c_int),
                ("out_f32", ctypes.c_int), ("conv", ctypes.c_int), ("smem_bytes", ctypes.c_int),
                ("ldg", ctypes.c_int), ("splitk", ctypes.c_int)]


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int

_SIGS = {
    "tp_gemm_bf16": ([_P, _P, _P] + [_I64] * 6 + [_P], _I),
    "tp_gemm_bf16_f32": ([_P, _P, _P] + [_I64] * 6 + [_P], _I),
    "tp_gemm_bf16_ex": ([_P, _P, _P] + [_I64] * 6 + [_I, ctypes.POINTER(tp_gemm_opts), _P], _I),
    "tp_gemm_bf16_host": ([_P, _P, _P] + [_I64] * 6 + [_I, _P, _P, _P, ctypes.POINTER(tp_gemm_opts), _P], _I),
    "tp_gemm_bf16_splitk": ([_P, _P, _P] + [_I64] * 6 + [_I, _I, _P, _I64, ctypes.POINTER(tp_gemm_opts), _P], _I),
    "tp_gemm_splitk_workspace_bytes": ([_I64, _I64, _I, ctypes.POINTER(_I64)], _I),
    "tp_gemm_bf16_splitk_noalloc": ([_P, _P, _P] + [_I64] * 6 + [_I, _I, _P], _I),
    "tp_gemm_splitk_noalloc_capacity": ([], _I64),
    "tp_conv2d_fprop_bf16": ([_P, _P, _P] + [_I64] * 9 + [_P], _I),
    "tp_conv2d_fprop_bf16_ex": ([_P, _P, _P] + [_I64] * 9 + [_I, ctypes.POINTER(tp_gemm_opts), _P], _I),
    "tp_tma_copy_2d": ([_P, _P, _I64, _I64, _I64, _P], _I),
    "tp_tma_copy_2d_ex": ([_P, _P, _I64, _I64, _I64, ctypes.POINTER(tp_copy_opts), _P], _I),
    "tp_tma_transpose_2d": ([_P, _P, _I64, _I64, _I64, _I64, _P], _I),
    "tp_tma_transpose_2d_ex": ([_P, _P, _I64, _I64, _I64, _I64, ctypes.POINTER(tp_copy_opts), _P], _I),
    "tp_tma_read_2d": ([_P, _I64, _I64, _I64, ctypes.POINTER(tp_copy_opts), _P], _I),
    "tp_device_status": ([_P], _I),
    "tp_device_status_detail": ([_P, ctypes.POINTER(_I), ctypes.POINTER(_I), ctypes.POINTER(_I)], _I),
    "tp_status_string": ([_I], ctypes.c_char_p),
    "tp_last_cuda_error": ([], _I),
    "tp_query_smem_bytes": ([_I, _I, _I, _I, ctypes.POINTER(_I64)], _I),
    "tp_gemm_plan": ([_P, _P, _P] + [_I64] * 6 + [_I, ctypes.POINTER(tp_gemm_opts), _I,
                                                     ctypes.POINTER(tp_plan)], _I),
    "tp_last_plan": ([ctypes.POINTER(tp_plan)], _I),
    "tp_list_kernels": ([ctypes.POINTER(tp_kernel_desc), _I], _I),
    "tp_selftest_wait_timeout": ([ctypes.c_uint32, _P], _I),
    "tp_selftest_mainloop_withheld_arrival": ([_P, _P, _P, _I64, _I64, _I64, ctypes.c_uint32, _P], _I),
    "tp_selftest_mainloop_skipped_commit": ([_P, _P, _P, _I64, _I64, _I64, _I, _I, ctypes.c_uint32, _P], _I),
    "tp_probe_fma_latency": ([_I, _I, ctypes.c_double, ctypes.POINTER(ctypes.c_double),
                              ctypes.POINTER(ctypes.c_double), _P], _I),
}
for _name, (_args, _res) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = _res

EXPORTED = tuple(_SIGS)


class TPError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {tp_status_string(status)}"
        if status == TP_ERR_CUDA:
            msg += f" (cudaError {_lib.tp_last_cuda_error()})"
        super().__init__(msg)


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


_current_stream = None


def _stream(s):
    """A stream argument as a cudaStream_t integer: an int is passed through,
    an object with .cuda_stream gives its handle, None means torch's current
    stream (or the legacy default stream without torch)."""
    global _current_stream
    if s is None:
        if _current_stream is None:
            try:
                import torch
                _current_stream = (lambda: torch.cuda.current_stream().cuda_stream) \
                    if torch.cuda.is_available() else (lambda: 0)
            except ImportError:
                _current_stream = lambda: 0  # noqa: E731
        return _current_stream()
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(st: int, where: str) -> None:
    if st != TP_OK:
        raise TPError(st, where)


def tp_status_string(status: int) -> str:
    """Name of a TP_* status code."""
    return _lib.tp_status_string(status).decode()


def tp_gemm_bf16(A, B, C, M, N, K, lda, ldb, ldc, stream=None):
    """C (bf16, M x N, pitch ldc) = A (M x K, pitch lda) . B (stored N x K, pitch ldb); pitches in
    elements. Asynchronous on `stream`; raises TPError on a host-visible error."""
    _check(_lib.tp_gemm_bf16(_ptr(A), _ptr(B), _ptr(C), M, N, K, lda, ldb, ldc, _stream(stream)),
           "tp_gemm_bf16")


def tp_gemm_bf16_f32(A, B, C, M, N, K, lda, ldb, ldc, stream=None):
    """tp_gemm_bf16 with the fp32 accumulator written to a float C."""
    _check(_lib.tp_gemm_bf16_f32(_ptr(A), _ptr(B), _ptr(C), M, N, K, lda, ldb, ldc, _stream(stream)),
           "tp_gemm_bf16_f32")


TRACE_SLOTS = 8
TRACE_NAMES = ("producer_span", "producer_wait_empty", "mma_span", "mma_wait_full", "mma_wait_acc_empty",
               "epilogue_span", "epilogue_wait_acc_full", "units")
PROTO_MAX_STAGES = 9
PROTO_PHASES = 64
PROTO_BARS = 2 * PROTO_MAX_STAGES + 4
PROTO_TX_EXPECT = PROTO_BARS * PROTO_PHASES
PROTO_TX_ISSUED = PROTO_TX_EXPECT + PROTO_MAX_STAGES * PROTO_PHASES
PROTO_SLOTS = PROTO_TX_ISSUED + PROTO_MAX_STAGES * PROTO_PHASES
EVENTS_PER_UNIT = 8
EVENT_UNITS = 8
EVENT_SLOTS = EVENTS_PER_UNIT * EVENT_UNITS
EVENT_NAMES = ("producer_start", "producer_end", "mma_start", "mma_end", "epilogue_ready", "epilogue_released",
               "epilogue_stored", "unit")


def _opts(atom=0, pipe_depth=0, tile_n=0, group_m=0, max_ctas=0, l2_hint=0, no_tail=0, trace=None, events=None,
          protocol=None):
    return tp_gemm_opts(atom, pipe_depth, tile_n, group_m, max_ctas, l2_hint, int(bool(no_tail)), _ptr(trace),
                        _ptr(events), _ptr(protocol))


def tp_gemm_bf16_ex(A, B, C, M, N, K, lda, ldb, ldc, out_f32=False, stream=None, **opts):
    """tp_gemm_bf16 / tp_gemm_bf16_f32 with explicit mainloop choices (atom, pipe_depth, tile_n,
    group_m, max_ctas, l2_hint, no_tail, trace, events; all optional, 0 = choose)."""
    o = _opts(**opts)
    _check(_lib.tp_gemm_bf16_ex(_ptr(A), _ptr(B), _ptr(C), M, N, K, lda, ldb, ldc, int(bool(out_f32)),
                                ctypes.byref(o), _stream(stream)), "tp_gemm_bf16_ex")


def tp_gemm_bf16_splitk(A, B, C, M, N, K, lda, ldb, ldc, out_f32=False, splits=0, workspace=None,
                        workspace_bytes=0, stream=None, **opts):
    """The GEMM with K split into `splits` slices (0 = choose) whose fp32 partials go to the
    caller's `workspace` (tp_gemm_splitk_workspace_bytes) and are summed into C by a second kernel."""
    o = _opts(**opts)
    if workspace is not None and not isinstance(workspace, int) and not workspace_bytes:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(_lib.tp_gemm_bf16_splitk(_ptr(A), _ptr(B), _ptr(C), M, N, K, lda, ldb, ldc, int(bool(out_f32)),
                                    splits, _ptr(workspace), workspace_bytes, ctypes.byref(o), _stream(stream)),
           "tp_gemm_bf16_splitk")


def tp_gemm_splitk_workspace_bytes(M, N, splits) -> int:
    """Workspace bytes tp_gemm_bf16_splitk needs for M x N with `splits` slices."""
    b = _I64()
    _check(_lib.tp_gemm_splitk_workspace_bytes(M, N, splits, ctypes.byref(b)), "tp_gemm_splitk_workspace_bytes")
    return int(b.value)


def tp_gemm_bf16_host(A_host, B_host, C_host, M, N, K, lda, ldb, ldc, dA, dB, dC, out_f32=False, stream=None,
                      **opts):
    """End-to-end GEMM on host operands: upload into the device buffers dA,
    dB, GEMM into dC, download into C_host, all enqueued on `stream`. Host
    arguments are pinned torch tensors or raw addresses."""
    o = _opts(**opts)
    _check(_lib.tp_gemm_bf16_host(_ptr(A_host), _ptr(B_host), _ptr(C_host), M, N, K, lda, ldb, ldc,
                                  int(bool(out_f32)), _ptr(dA), _ptr(dB), _ptr(dC), ctypes.byref(o),
                                  _stream(stream)), "tp_gemm_bf16_host")


def tp_gemm_bf16_splitk_noalloc(A, B, C, M, N, K, lda, ldb, ldc, out_f32=False, splits=0, stream=None):
    """Split-K GEMM whose workspace is the library's fixed array (no allocation)."""
    _check(_lib.tp_gemm_bf16_splitk_noalloc(_ptr(A), _ptr(B), _ptr(C), M, N, K, lda, ldb, ldc,
                                            int(bool(out_f32)), splits, _stream(stream)),
           "tp_gemm_bf16_splitk_noalloc")


def tp_gemm_splitk_noalloc_capacity() -> int:
    """Bytes of the in-library split-K workspace of each GPU."""
    return int(_lib.tp_gemm_splitk_noalloc_capacity())


def tp_conv2d_fprop_bf16(x, w, y, N, H, W, C, K, R, S, stride, pad, stream=None):
    """y (N x P x Q x K, bf16) = conv(x (N x H x W x C), w (K x R x S x C)): cross-correlation,
    zero padding `pad`, `stride`; all three tensors packed NHWC / KRSC / NPQK."""
    _check(_lib.tp_conv2d_fprop_bf16(_ptr(x), _ptr(w), _ptr(y), N, H, W, C, K, R, S, stride, pad,
                                     _stream(stream)), "tp_conv2d_fprop_bf16")


def tp_conv2d_fprop_bf16_ex(x, w, y, N, H, W, C, K, R, S, stride, pad, out_f32=False, stream=None, **opts):
    """tp_conv2d_fprop_bf16 with an fp32 output option and the same mainloop choices as
    tp_gemm_bf16_ex."""
    o = _opts(**opts)
    _check(_lib.tp_conv2d_fprop_bf16_ex(_ptr(x), _ptr(w), _ptr(y), N, H, W, C, K, R, S, stride, pad,
                                        int(bool(out_f32)), ctypes.byref(o), _stream(stream)),
           "tp_conv2d_fprop_bf16_ex")


def tp_tma_copy_2d(src, dst, rows, cols, ld, stream=None):
    """dst = src, bit for bit: rows x cols 2-byte elements, both with row pitch `ld` elements."""
    _check(_lib.tp_tma_copy_2d(_ptr(src), _ptr(dst), rows, cols, ld, _stream(stream)), "tp_tma_copy_2d")


def tp_tma_copy_2d_ex(src, dst, rows, cols, ld, stream=None, box_cols=0, box_rows=0, stages=0,
                      ctas_per_sm=0, force_vec=False):
    """tp_tma_copy_2d with explicit ring choices (TMA box, stages, CTAs per SM, or the
    vectorized copy)."""
    o = tp_copy_opts(box_cols, box_rows, stages, ctas_per_sm, int(bool(force_vec)))
    _check(_lib.tp_tma_copy_2d_ex(_ptr(src), _ptr(dst), rows, cols, ld, ctypes.byref(o), _stream(stream)),
           "tp_tma_copy_2d_ex")


def tp_tma_transpose_2d(src, dst, rows, cols, ld_src, ld_dst, stream=None):
    """dst[c][r] = src[r][c], bit for bit: src rows x cols (pitch ld_src), dst cols x rows
    (pitch ld_dst), 2-byte elements."""
    _check(_lib.tp_tma_transpose_2d(_ptr(src), _ptr(dst), rows, cols, ld_src, ld_dst, _stream(stream)),
           "tp_tma_transpose_2d")


def tp_tma_transpose_2d_ex(src, dst, rows, cols, ld_src, ld_dst, stream=None, stages=0, ctas_per_sm=0,
                           force_vec=False):
    """tp_tma_transpose_2d with explicit ring choices (stages, CTAs per SM, or the
    shared-memory tile fallback)."""
    o = tp_copy_opts(0, 0, stages, ctas_per_sm, int(bool(force_vec)))
    _check(_lib.tp_tma_transpose_2d_ex(_ptr(src), _ptr(dst), rows, cols, ld_src, ld_dst, ctypes.byref(o),
                                       _stream(stream)), "tp_tma_transpose_2d_ex")


def tp_tma_read_2d(src, rows, cols, ld, stream=None, box_cols=0, box_rows=0, stages=0, ctas_per_sm=0):
    """Streams rows x cols 2-byte elements (pitch `ld`) through the TMA load ring and discards
    them: how fast the GPU pulls an operand. Options 0 = library default."""
    o = tp_copy_opts(box_cols, box_rows, stages, ctas_per_sm, 0)
    _check(_lib.tp_tma_read_2d(_ptr(src), rows, cols, ld, ctypes.byref(o), _stream(stream)), "tp_tma_read_2d")


def tp_device_status(stream=None) -> int:
    """Synchronizes the stream; returns (and clears) the device status code."""
    return int(_lib.tp_device_status(_stream(stream)))


def tp_device_status_detail(stream=None):
    """Like tp_device_status, plus where the failure was recorded: (status, site, block,
    thread)."""
    site, block, thread = _I(), _I(), _I()
    st = _lib.tp_device_status_detail(_stream(stream), ctypes.byref(site), ctypes.byref(block),
                                      ctypes.byref(thread))
    return int(st), site.value, block.value, thread.value


def tp_query_smem_bytes(atom, pipe_depth, tile_n, out_f32=False):
    """Returns (status, bytes): TP_OK when it fits, TP_ERR_SMEM_BUDGET when not."""
    b = _I64()
    st = _lib.tp_query_smem_bytes(atom, pipe_depth, tile_n, int(bool(out_f32)), ctypes.byref(b))
    return int(st), int(b.value)


def tp_gemm_plan(A, B, C, M, N, K, lda, ldb, ldc, out_f32=False, sm_count=0, **opts):
    """Returns (status, plan dict) without launching anything."""
    o = _opts(**opts)
    p = tp_plan()
    st = _lib.tp_gemm_plan(_ptr(A), _ptr(B), _ptr(C), M, N, K, lda, ldb, ldc, int(bool(out_f32)),
                           ctypes.byref(o), sm_count, ctypes.byref(p))
    return int(st), p.as_dict()


def tp_last_plan() -> dict:
    """The plan (path, variant, launch shape) of this thread's last GEMM / conv / copy call."""
    p = tp_plan()
    _check(_lib.tp_last_plan(ctypes.byref(p)), "tp_last_plan")
    return p.as_dict()


def tp_list_kernels():
    """Every compiled mainloop variant, as dicts (atom, pipe_depth, tile_n, out_f32, conv,
    smem_bytes, ldg, splitk)."""
    n = _lib.tp_list_kernels(None, 0)
    arr = (tp_kernel_desc * n)()
    _lib.tp_list_kernels(arr, n)
    return [{f: getattr(a, f) for f, _ in tp_kernel_desc._fields_} for a in arr]


def tp_probe_fma_latency(kind: int, chain: int = 65536, seed: float = 0.0, stream=None):
    """Returns (chain result, SM cycles per dependent fma link); kind 0 fp32, 1 fp64."""
    r, c = ctypes.c_double(), ctypes.c_double()
    _check(_lib.tp_probe_fma_latency(kind, chain, seed, ctypes.byref(r), ctypes.byref(c), _stream(stream)),
           "tp_probe_fma_latency")
    return r.value, c.value


def tp_selftest_mainloop_withheld_arrival(A, B, C, M, N, K, limit_ms, stream=None):
    """Runs the 1-SM mainloop with its first stage's arrival withheld, so that
    its bounded waits must give up after `limit_ms`; the device status then reads TP_ERR_TIMEOUT."""
    _check(_lib.tp_selftest_mainloop_withheld_arrival(_ptr(A), _ptr(B), _ptr(C), M, N, K, limit_ms, _stream(stream)),
           "tp_selftest_mainloop_withheld_arrival")


def tp_selftest_mainloop_skipped_commit(A, B, C, M, N, K, which, atom, limit_ms, stream=None):
    """Runs the mainloop (atom 1 or 2, MMA N 128) with the MMA issuer skipping its first commit
    to empty[s] (which = 1) or to acc_full[b] (which = 2), so that the waits behind it must give
    up after `limit_ms`; the device status then reads TP_ERR_TIMEOUT."""
    _check(_lib.tp_selftest_mainloop_skipped_commit(_ptr(A), _ptr(B), _ptr(C), M, N, K, which, atom, limit_ms,
                                                    _stream(stream)),
           "tp_selftest_mainloop_skipped_commit")


def tp_selftest_wait_timeout(limit_us: int, stream=None):
    """Launches one bounded wait that nothing satisfies (`limit_us`); returns the device
    status it leaves."""
    _check(_lib.tp_selftest_wait_timeout(limit_us, _stream(stream)), "tp_selftest_wait_timeout")


# --------------------------------------------------------------------------
# Tensor conveniences (still marshalling only: shapes -> sizes and pitches).
# --------------------------------------------------------------------------

def _require(cond, msg):
    if not cond:
        raise ValueError(msg)


def _rows_packed(t, name):
    """A 2-D view whose rows are packed (unit stride along the last axis)."""
    _require(t.dim() == 2, f"{name} must be 2-D, got shape {tuple(t.shape)}")
    _require(t.shape[1] <= 1 or t.stride(1) == 1, f"{name} must have unit stride along its last axis")


def gemm(A, B_nk, C, stream=None, **opts):
    """C (M x N, bf16 or fp32) = A (M x K) . B, B given as an N x K tensor
    (i.e. K x N column-major). Row pitches come from the tensors' strides;
    each row must be packed (a transposed view is rejected, not copied)."""
    for t, name in ((A, "A"), (B_nk, "B_nk"), (C, "C")):
        _rows_packed(t, name)
    M, K = A.shape
    N = B_nk.shape[0]
    _require(B_nk.shape[1] == K, f"B_nk is {tuple(B_nk.shape)}, expected ({N}, {K})")
    _require(tuple(C.shape) == (M, N), f"C is {tuple(C.shape)}, expected ({M}, {N})")
    _require(str(A.dtype).endswith("bfloat16") and str(B_nk.dtype).endswith("bfloat16"), "A and B_nk must be bf16")
    _require(str(C.dtype).endswith("bfloat16") or str(C.dtype).endswith("float32"), "C must be bf16 or fp32")
    out_f32 = str(C.dtype).endswith("float32")
    tp_gemm_bf16_ex(A, B_nk, C, M, N, K, max(A.stride(0), K), max(B_nk.stride(0), K), max(C.stride(0), N),
                    out_f32=out_f32, stream=stream, **opts)
    return C


def conv2d_fprop(x, w, y, stride=1, pad=0, stream=None, **opts):
    """y (N x P x Q x K) = conv(x (N x H x W x C), w (K x R x S x C)), all
    three contiguous (NHWC / KRSC / NPQK); y may also be (N*P*Q) x K."""
    _require(x.dim() == 4 and w.dim() == 4, "x and w must be 4-D (NHWC, KRSC)")
    N, H, W, C = x.shape
    K, R, S, Cw = w.shape
    _require(Cw == C, f"w has {Cw} input channels, x has {C}")
    P = (H + 2 * pad - R) // stride + 1
    Q = (W + 2 * pad - S) // stride + 1
    _require(y.numel() == N * P * Q * K and y.shape[-1] == K, f"y must hold {N}x{P}x{Q}x{K} outputs")
    for t, name in ((x, "x"), (w, "w"), (y, "y")):
        _require(t.is_contiguous(), f"{name} must be contiguous")
    _require(str(x.dtype).endswith("bfloat16") and str(w.dtype).endswith("bfloat16"), "x and w must be bf16")
    _require(str(y.dtype).endswith("bfloat16") or str(y.dtype).endswith("float32"), "y must be bf16 or fp32")
    out_f32 = str(y.dtype).endswith("float32")
    tp_conv2d_fprop_bf16_ex(x, w, y, N, H, W, C, K, R, S, stride, pad, out_f32=out_f32, stream=stream, **opts)
    return y
