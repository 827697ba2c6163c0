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
// multiple of 4, 16-byte aligned); each thread handles 4 adjacent columns.
template <bool OUT_F32>
__global__ void __launch_bounds__(256)
    splitk_reduce_kernel(const float* __restrict__ ws, void* __restrict__ C, int M, int N, int64_t ldw,
                         int64_t ldc, int splits)
{
    const int64_t quads = (N + 3) / 4;
    const int64_t total = static_cast<int64_t>(M) * quads;
    const int64_t slice = static_cast<int64_t>(M) * ldw;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t m = i / quads;
        const int n = static_cast<int>(i - m * quads) * 4;
        const float4* src = reinterpret_cast<const float4*>(ws + m * ldw + n);
        float4 acc = __ldg(src);
        for (int s = 1; s < splits; ++s) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(src) + s * slice));
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        const float a[4] = {acc.x, acc.y, acc.z, acc.w};
        const int cnt = N - n < 4 ? N - n : 4;
        if constexpr (OUT_F32) {
            float* row = static_cast<float*>(C) + m * ldc + n;
            for (int j = 0; j < cnt; ++j) row[j] = a[j];
        } else {
            __nv_bfloat16* row = static_cast<__nv_bfloat16*>(C) + m * ldc + n;
            for (int j = 0; j < cnt; ++j) row[j] = __float2bfloat16_rn(a[j]);
        }
    }
}

cudaError_t launch_splitk_reduce(const float* ws, void* C, int M, int N, int64_t ldw, int64_t ldc, int splits,
                                 int out_f32, int sm_count, cudaStream_t st)
{
    const int64_t total = static_cast<int64_t>(M) * ((N + 3) / 4);
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sm_count) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (out_f32)
        splitk_reduce_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, st>>>(ws, C, M, N, ldw, ldc, splits);
    else
        splitk_reduce_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, st>>>(ws, C, M, N, ldw, ldc, splits);
    return cudaGetLastError();
}

}  // namespace tp
