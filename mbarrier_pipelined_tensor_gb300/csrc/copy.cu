// TMA-only 2D copy (no MMA) and the vectorized thread-copy fallback.
//
// TMA path ("B200 Tma Pipeline Designer", steps 4-7): a persistent CTA of one
// warp; its elected lane runs a ring of STAGES tiles. Load protocol: per-stage
// barrier, arrive.expect_tx(tile bytes) by the issuing lane, the store waits
// for the stage's phase. Store protocol: each TMA store is its own bulk group
// (commit_group); a stage is refilled only after wait_group.read guarantees
// the store issued LAG tiles earlier has finished reading it -- the load-side
// byte count is never used to drain stores.
//
// Fallback ("Do not use when": irregular or misaligned): a grid-stride
// coalesced copy, 16-byte vectors where source and destination share their
// alignment, 2-byte elements otherwise.
#include <cstdint>

#include "common.cuh"

namespace tp {

template <int STAGES, int LAG>
__global__ void __launch_bounds__(32, 1)
    tma_copy_kernel(const __grid_constant__ CUtensorMap src, const __grid_constant__ CUtensorMap dst,
                    const CopyParams p)
{
    static_assert(LAG >= 1 && LAG < STAGES, "refill lag");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t stride = (p.tile_bytes + 1023u) & ~1023u;
    const uint32_t sBar = base + STAGES * stride;
    volatile int* const abort_flag =
        reinterpret_cast<volatile int*>(smem_raw + (sBar - raw) + 8 * STAGES);
    auto full_bar = [&](int s) { return sBar + 8u * s; };

    if (elect_one()) {
        for (int s = 0; s < STAGES; ++s) mbar_init(full_bar(s), 1);
        *abort_flag = 0;
        fence_mbarrier_init();
        prefetch_tensormap(&src);
        prefetch_tensormap(&dst);

        const int total = p.tiles_x * p.tiles_y;
        const int first = static_cast<int>(blockIdx.x);
        const int step = static_cast<int>(gridDim.x);
        const int n_my = first < total ? (total - first + step - 1) / step : 0;
        auto tile_xy = [&](int i, int& x, int& y) {
            const int t = first + i * step;
            const int ty = t / p.tiles_x;
            x = (t - ty * p.tiles_x) * p.box_cols;
            y = ty * p.box_rows;
        };
        auto issue_load = [&](int i) {
            const int s = i % STAGES;
            int x, y;
            tile_xy(i, x, y);
            mbar_arrive_expect_tx(full_bar(s), p.tile_bytes);
            tma_load_2d(base + s * stride, &src, full_bar(s), x, y);
        };

        // Prologue: fill the ring.
        const int pro = n_my < STAGES ? n_my : STAGES;
        for (int i = 0; i < pro; ++i) issue_load(i);
        int loaded = pro;

        // Steady state: store tile i, refill the stage of tile i - LAG.
        int i = 0;
        for (; i < n_my; ++i) {
            const int s = i % STAGES;
            const uint32_t ph = static_cast<uint32_t>(i / STAGES) & 1u;
            if (!wait_bounded(full_bar(s), ph, p.wait, abort_flag, SITE_COPY_FULL)) break;
            int x, y;
            tile_xy(i, x, y);
            tma_store_2d(&dst, base + s * stride, x, y);
            bulk_commit_group();
            const int j = i - LAG + STAGES;  // tile that reuses the stage of tile i - LAG
            if (i >= LAG && j < n_my) {
                bulk_wait_group_read<LAG>();
                issue_load(j);
                loaded = j + 1;
            }
        }
        if (i < n_my) {
            // Gave up: let every load still in flight land (bounded) before exit.
            volatile int no_abort = 0;
            for (int k = i; k < loaded; ++k)
                wait_bounded(full_bar(k % STAGES), static_cast<uint32_t>(k / STAGES) & 1u, p.wait,
                                    &no_abort, SITE_DRAIN);
        }
        // Epilogue: drain every outstanding store.
        bulk_wait_group<0>();
    }
    __syncwarp();
}

template <int STAGES, int LAG>
cudaError_t launch_tma_copy(const CUtensorMap& s, const CUtensorMap& d, const CopyParams& p, int grid,
                            cudaStream_t st)
{
    const uint32_t stride = (p.tile_bytes + 1023u) & ~1023u;
    const int smem = 1024 + STAGES * static_cast<int>(stride) + 8 * STAGES + 16;
    auto kern = tma_copy_kernel<STAGES, LAG>;
    static std::atomic<uint64_t> smem_set{0};
    cudaError_t e = smem_limit_once(kern, 232448, smem_set);  // the limit, not this launch's size
    if (e != cudaSuccess) return e;
    kern<<<grid, 32, smem, st>>>(s, d, p);
    return cudaGetLastError();
}

int copy_smem_bytes(int stages, uint32_t tile_bytes)
{
    const uint32_t stride = (tile_bytes + 1023u) & ~1023u;
    return 1024 + stages * static_cast<int>(stride) + 8 * stages + 16;
}

cudaError_t launch_tma_copy_any(int stages, const CUtensorMap& s, const CUtensorMap& d, const CopyParams& p,
                                int grid, cudaStream_t st)
{
    switch (stages) {
    case 2: return launch_tma_copy<2, 1>(s, d, p, grid, st);
    case 3: return launch_tma_copy<3, 1>(s, d, p, grid, st);
    case 4: return launch_tma_copy<4, 1>(s, d, p, grid, st);
    case 6: return launch_tma_copy<6, 2>(s, d, p, grid, st);
    case 8: return launch_tma_copy<8, 2>(s, d, p, grid, st);
    case 12: return launch_tma_copy<12, 3>(s, d, p, grid, st);
    default: return cudaErrorInvalidValue;
    }
}

// ---------------------------------------------------------- read stream ---
//
// The load half of the copy ring on its own: each CTA streams a contiguous
// run of tiles through its STAGES-deep ring and discards them. It measures
// how fast TMA can pull an operand out of memory -- the bound of a GEMM that
// only streams its B (a skinny M) -- with no store traffic beside it. The
// loop steps tile coordinates incrementally: one thread issues every load.
template <int STAGES>
__global__ void __launch_bounds__(32, 1)
    tma_read_kernel(const __grid_constant__ CUtensorMap src, const CopyParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t stride = (p.tile_bytes + 1023u) & ~1023u;
    const uint32_t sBar = base + STAGES * stride;
    volatile int* const abort_flag =
        reinterpret_cast<volatile int*>(smem_raw + (sBar - raw) + 8 * STAGES);
    auto full_bar = [&](int s) { return sBar + 8u * s; };

    if (elect_one()) {
        for (int s = 0; s < STAGES; ++s) mbar_init(full_bar(s), 1);
        *abort_flag = 0;
        fence_mbarrier_init();
        prefetch_tensormap(&src);
        const int total = p.tiles_x * p.tiles_y;
        const int chunk = (total + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);
        const int first = static_cast<int>(blockIdx.x) * chunk;
        const int count = min(chunk, total - first);
        int tx = first % p.tiles_x, ty = first / p.tiles_x;
        int s = 0;
        uint32_t ph = 0;
        int issued = 0;
        bool ok = true;
        for (int c = 0; c < count; ++c) {
            // stage s was last filled STAGES tiles ago, in the ring pass of parity ph ^ 1
            if (issued >= STAGES && !wait_bounded(full_bar(s), ph ^ 1u, p.wait, abort_flag, SITE_COPY_FULL)) {
                ok = false;
                break;
            }
            mbar_arrive_expect_tx(full_bar(s), p.tile_bytes);
            tma_load_2d(base + s * stride, &src, full_bar(s), tx * p.box_cols, ty * p.box_rows);
            ++issued;
            if (++s == STAGES) {
                s = 0;
                ph ^= 1u;
            }
            if (++tx == p.tiles_x) {
                tx = 0;
                ++ty;
            }
        }
        // Every load still in flight lands before the CTA exits (bounded).
        volatile int no_abort = 0;
        const int n = issued < STAGES ? issued : STAGES;
        for (int k = 0; k < n; ++k) {
            if (--s < 0) {
                s = STAGES - 1;
                ph ^= 1u;
            }
            wait_bounded(full_bar(s), ph, p.wait, ok ? abort_flag : &no_abort, SITE_DRAIN);
        }
    }
    __syncwarp();
}

template <int STAGES>
cudaError_t launch_tma_read(const CUtensorMap& s, const CopyParams& p, int grid, cudaStream_t st)
{
    const uint32_t stride = (p.tile_bytes + 1023u) & ~1023u;
    const int smem = 1024 + STAGES * static_cast<int>(stride) + 8 * STAGES + 16;
    auto kern = tma_read_kernel<STAGES>;
    static std::atomic<uint64_t> smem_set{0};
    cudaError_t e = smem_limit_once(kern, 232448, smem_set);
    if (e != cudaSuccess) return e;
    kern<<<grid, 32, smem, st>>>(s, p);
    return cudaGetLastError();
}

cudaError_t launch_tma_read_any(int stages, const CUtensorMap& s, const CopyParams& p, int grid, cudaStream_t st)
{
    switch (stages) {
    case 2: return launch_tma_read<2>(s, p, grid, st);
    case 4: return launch_tma_read<4>(s, p, grid, st);
    case 8: return launch_tma_read<8>(s, p, grid, st);
    case 12: return launch_tma_read<12>(s, p, grid, st);
    default: return cudaErrorInvalidValue;
    }
}

// ------------------------------------------------------------ fallback ---

// Bytes sh .. sh + 15 of the 32 bytes lo:hi (sh even, 2..14): whole words
// dropped with selects, then a 16-bit funnel shift.
__device__ __forceinline__ uint4 shift_window16(const uint4& lo, const uint4& hi, uint32_t sh)
{
    uint32_t c[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    if (sh & 8u) {
#pragma unroll
        for (int i = 0; i < 6; ++i) c[i] = c[i + 2];
    }
    if (sh & 4u) {
#pragma unroll
        for (int i = 0; i < 5; ++i) c[i] = c[i + 1];
    }
    const uint32_t b = (sh & 2u) << 3;  // 0 or 16 bits
    return make_uint4(__funnelshift_r(c[0], c[1], b), __funnelshift_r(c[1], c[2], b), __funnelshift_r(c[2], c[3], b),
                      __funnelshift_r(c[3], c[4], b));
}

// rows x row_elems 2-byte elements, both buffers with pitch `pitch` elements.
// Per row: 2-byte copies up to dst's first 16-byte boundary, then aligned
// 16-byte stores. Where src has the same alignment the loads are aligned
// 16-byte loads too; otherwise each store's 16 bytes are cut from the two
// aligned source chunks around them (both hold bytes of the row, so neither
// read can leave its page). The last partial chunk is copied by elements.
__global__ void __launch_bounds__(256)
    vec_copy_kernel(const uint16_t* __restrict__ src, uint16_t* __restrict__ dst, int64_t rows,
                    int64_t row_elems, int64_t pitch)
{
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
        const uint16_t* s = src + r * pitch;
        uint16_t* d = dst + r * pitch;
        const uintptr_t sa = reinterpret_cast<uintptr_t>(s);
        const uintptr_t da = reinterpret_cast<uintptr_t>(d);
        int64_t head = static_cast<int64_t>(((16u - (da & 15u)) & 15u) / 2u);
        if (head > row_elems) head = row_elems;
        const int64_t nvec = (row_elems - head) / 8;
        const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
        const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;
        for (int64_t i = tid; i < head; i += nthr) d[i] = s[i];
        uint4* dv = reinterpret_cast<uint4*>(d + head);
        const uintptr_t x = sa + 2u * static_cast<uintptr_t>(head);  // source of dst's first aligned chunk
        const uint32_t sh = static_cast<uint32_t>(x & 15u);
        const uint4* sv = reinterpret_cast<const uint4*>(x - sh);
        if (sh == 0) {
            for (int64_t i = tid; i < nvec; i += nthr) dv[i] = __ldg(sv + i);
        } else {
            for (int64_t i = tid; i < nvec; i += nthr) dv[i] = shift_window16(__ldg(sv + i), __ldg(sv + i + 1), sh);
        }
        for (int64_t i = head + nvec * 8 + tid; i < row_elems; i += nthr) d[i] = s[i];
    }
}

cudaError_t launch_vec_copy(const void* src, void* dst, int64_t rows, int64_t cols, int64_t ld, int sm_count,
                            cudaStream_t st)
{
    const int64_t vec_per_row = (cols + 7) / 8;
    int gx = static_cast<int>((vec_per_row + 255) / 256);
    if (gx < 1) gx = 1;
    if (gx > 64) gx = 64;
    int64_t gy = (static_cast<int64_t>(sm_count) * 8 + gx - 1) / gx;
    if (gy > rows) gy = rows;
    if (gy > 65535) gy = 65535;
    if (gy < 1) gy = 1;
    vec_copy_kernel<<<dim3(gx, static_cast<unsigned>(gy)), 256, 0, st>>>(
        static_cast<const uint16_t*>(src), static_cast<uint16_t*>(dst), rows, cols, ld);
    return cudaGetLastError();
}

// C[m*ldc + n] = 0 for m < M, n < N (K == 0 GEMM: the empty sum).
__global__ void __launch_bounds__(256)
    zero_fill_kernel(uint8_t* __restrict__ c, int64_t M, int64_t row_bytes, int64_t pitch_bytes)
{
    for (int64_t m = blockIdx.y; m < M; m += gridDim.y) {
        uint8_t* row = c + m * pitch_bytes;
        for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < row_bytes / 2;
             i += static_cast<int64_t>(gridDim.x) * blockDim.x)
            reinterpret_cast<uint16_t*>(row)[i] = 0;
    }
}

cudaError_t launch_zero_fill(void* c, int64_t M, int64_t N, int64_t ldc, int elem_bytes, cudaStream_t st)
{
    const int64_t row_bytes = N * elem_bytes;
    int gx = static_cast<int>((row_bytes / 2 + 255) / 256);
    if (gx > 64) gx = 64;
    if (gx < 1) gx = 1;
    int64_t gy = M < 4096 ? M : 4096;
    zero_fill_kernel<<<dim3(gx, static_cast<unsigned>(gy)), 256, 0, st>>>(static_cast<uint8_t*>(c), M, row_bytes,
                                                                           ldc * elem_bytes);
    return cudaGetLastError();
}

// ----------------------------------------------------------- self test ---

// Waits on a barrier that nothing ever arrives on, with a short limit: the
// wait must give up, record ST_TIMEOUT and return. Exercises the bounded-wait
// path without stalling anything else.
__global__ void wait_timeout_selftest_kernel(WaitCtl w)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbarrier_init();
        wait_bounded(smem_u32(&bar), 0, w, reinterpret_cast<volatile int*>(&abort_flag), SITE_SELFTEST);
    }
}

cudaError_t launch_wait_selftest(const WaitCtl& w, cudaStream_t st)
{
    wait_timeout_selftest_kernel<<<1, 32, 0, st>>>(w);
    return cudaGetLastError();
}

}  // namespace tp
