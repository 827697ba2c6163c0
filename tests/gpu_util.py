"""Helpers shared by the GPU parity tests: move the generators' bf16 bit
arrays to the device and back, run the library, compare with the oracle."""
import numpy as np
import torch

import datagen
import oracle
import mbarrier_pipelined_tensor_gb300 as tp

BF16_NAN = 0x7FC0


def dev_u16(arr):
    return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.uint16).view(np.int16)).cuda()


def dev_bf16(arr):
    return dev_u16(arr).view(torch.bfloat16)


def host_u16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_f64(t):
    if t.dtype == torch.float32:
        return t.cpu().numpy().astype(np.float64)
    return datagen.bf16_to_f32(host_u16(t)).astype(np.float64)


def new_out(M, ldc, out_f32):
    if out_f32:
        return torch.full((M, ldc), float("nan"), dtype=torch.float32, device="cuda")
    return torch.full((M, ldc), BF16_NAN, dtype=torch.int16, device="cuda").view(torch.bfloat16)


def expect_ok():
    st, site, block, thread = tp.tp_device_status_detail()
    assert st == tp.TP_OK, f"device status {tp.tp_status_string(st)} site {site} block {block} thread {thread}"


def run_gemm(A, B, M, N, K, lda, ldb, ldc=None, out_f32=False, **opts):
    ldc = N if ldc is None else ldc
    a, b = dev_bf16(A), dev_bf16(B)
    c = new_out(M, ldc, out_f32)
    tp.tp_gemm_bf16_ex(a, b, c, M, N, K, lda, ldb, ldc, out_f32=out_f32, **opts)
    expect_ok()
    plan = tp.tp_last_plan()
    full = host_f64(c)
    if ldc > N:  # columns past N must be untouched
        assert np.all(np.isnan(full[:, N:])), "wrote past N"
    return full[:, :N], plan


def check_against_oracle(got, ref, ab, out_f32, what=""):
    ok, worst, nbad = oracle.check(got, ref, ab, out_bf16=not out_f32)
    assert ok, f"{what}: {nbad} elements out of tolerance (worst {worst:.3g}x)"
    return worst
