// Split-K variants of the mainloop: every (tile, K slice) work unit writes
// its fp32 partial into a slice of a caller-provided workspace; a reduction
// kernel sums the slices into C. Both atoms, both MMA N, deepest rings.
#include "gemm_kernel.cuh"

namespace tp {

static const KernelEntry k_table[] = {
    mainloop_entry<1, 128, 6, true, false, false, true>(),
    mainloop_entry<1, 256, 4, true, false, false, true>(),
    mainloop_entry<2, 128, 8, true, false, false, true>(),
    mainloop_entry<2, 256, 6, true, false, false, true>(),
};

const KernelEntry* table_mainloop_splitk(int* n)
{
    *n = static_cast<int>(sizeof(k_table) / sizeof(k_table[0]));
    return k_table;
}

// C[m][n] = sum over slices s of ws[s][m][n], summed in slice order in fp32,
// then rounded to nearest even for a bf16 C. ws rows hold ldw floats (a
// multiple of 4, 16-byte aligned); each thread handles 4 adjacent columns,
// loading the slices four at a time before adding them in order. VEC: C's
// rows allow one 16-byte (fp32) or 8-byte (bf16) store per 4 columns.
//
// Launched as a programmatic dependent of the mainloop that wrote ws: it
// may be scheduled while that grid runs and waits for its completion (and
// the visibility of its writes) before the first load.
template <bool OUT_F32, bool VEC>
__global__ void __launch_bounds__(256)
    splitk_reduce_kernel(const float* __restrict__ ws, void* __restrict__ C, int M, int N, int64_t ldw,
                         int64_t ldc, int splits)
{
    griddep_wait();
    const int64_t quads = (N + 3) / 4;
    const int64_t total = static_cast<int64_t>(M) * quads;
    const int64_t slice = static_cast<int64_t>(M) * ldw;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t m = i / quads;
        const int n = static_cast<int>(i - m * quads) * 4;
        const float* src = ws + m * ldw + n;
        float4 acc = __ldg(reinterpret_cast<const float4*>(src));
        int s = 1;
        for (; s + 4 <= splits; s += 4) {
            float4 v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = __ldg(reinterpret_cast<const float4*>(src + (s + j) * slice));
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                acc.x += v[j].x;
                acc.y += v[j].y;
                acc.z += v[j].z;
                acc.w += v[j].w;
            }
        }
        for (; s < splits; ++s) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(src + s * slice));
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        const int cnt = N - n < 4 ? N - n : 4;
        if constexpr (OUT_F32) {
            float* row = static_cast<float*>(C) + m * ldc + n;
            if (VEC && cnt == 4) {
                *reinterpret_cast<float4*>(row) = acc;
            } else {
                const float a[4] = {acc.x, acc.y, acc.z, acc.w};
                for (int j = 0; j < cnt; ++j) row[j] = a[j];
            }
        } else {
            __nv_bfloat16* row = static_cast<__nv_bfloat16*>(C) + m * ldc + n;
            const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
            const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
            if (VEC && cnt == 4) {
                uint2 u;
                u.x = *reinterpret_cast<const uint32_t*>(&lo);
                u.y = *reinterpret_cast<const uint32_t*>(&hi);
                *reinterpret_cast<uint2*>(row) = u;
            } else {
                const __nv_bfloat16 a[4] = {lo.x, lo.y, hi.x, hi.y};
                for (int j = 0; j < cnt; ++j) row[j] = a[j];
            }
        }
    }
}

template <bool OUT_F32, bool VEC>
cudaError_t launch_reduce_t(const float* ws, void* C, int M, int N, int64_t ldw, int64_t ldc, int splits,
                            unsigned blocks, cudaStream_t st)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<OUT_F32, VEC>, ws, C, M, N, ldw, ldc, splits);
}

cudaError_t launch_splitk_reduce(const float* ws, void* C, int M, int N, int64_t ldw, int64_t ldc, int splits,
                                 int out_f32, int sm_count, cudaStream_t st)
{
    const int64_t total = static_cast<int64_t>(M) * ((N + 3) / 4);
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sm_count) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    const unsigned b = static_cast<unsigned>(blocks);
    const uintptr_t addr = reinterpret_cast<uintptr_t>(C);
    if (out_f32) {
        const bool vec = addr % 16 == 0 && ldc % 4 == 0;
        return vec ? launch_reduce_t<true, true>(ws, C, M, N, ldw, ldc, splits, b, st)
                   : launch_reduce_t<true, false>(ws, C, M, N, ldw, ldc, splits, b, st);
    }
    const bool vec = addr % 8 == 0 && ldc % 4 == 0;
    return vec ? launch_reduce_t<false, true>(ws, C, M, N, ldw, ldc, splits, b, st)
               : launch_reduce_t<false, false>(ws, C, M, N, ldw, ldc, splits, b, st);
}

}  // namespace tp
