// TMA 2D transpose of 2-byte elements: dst[c][r] = src[r][c], bit for bit.
//
// The copy ring of "B200 Tma Pipeline Designer" (steps 4-7) with a transpose
// between load and store: a persistent one-warp CTA keeps STAGES 64x64 tiles
// in flight (TMA loads with 128-byte swizzle, one expect_tx arrival each by
// the issuing lane); the warp turns each landed tile around in 8x8 blocks
// with ldmatrix / stmatrix.trans (both conflict-free on the swizzled
// layout) into one of two staging tiles, fences the generic proxy and stores
// the staging tile with TMA at the swapped coordinates. A staging tile is
// rewritten only after wait_group.read says its previous store has read it.
//
// Fallback: a 32x32 shared-memory tile transpose with plain loads/stores for
// buffers TMA cannot describe and for the destination's ragged last columns.
#include <cstdint>

#include "common.cuh"

namespace tp {

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void stmatrix_x4_trans(uint32_t addr, const uint32_t (&r)[4])
{
    asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3])
                 : "memory");
}

struct TransposeParams {
    int tiles_x, tiles_y;  // 64-wide tiles along src columns / src rows
    WaitCtl wait;
};

constexpr int kTT = 64;                         // tile edge (elements)
constexpr uint32_t kTileBytes = kTT * kTT * 2;  // 8 KiB

template <int STAGES>
__global__ void __launch_bounds__(32)
    tma_transpose_kernel(const __grid_constant__ CUtensorMap src, const __grid_constant__ CUtensorMap dst,
                         const TransposeParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // swizzle atoms: 1024-B alignment
    const uint32_t sIn = base;
    const uint32_t sOut = base + STAGES * kTileBytes;
    const uint32_t sBar = sOut + 2 * kTileBytes;
    volatile int* const abort_flag = reinterpret_cast<volatile int*>(smem_raw + (sBar - raw) + 8 * STAGES);
    auto full_bar = [&](int s) { return sBar + 8u * s; };
    const uint32_t lane = threadIdx.x & 31u;

    const int total = p.tiles_x * p.tiles_y;
    const int first = static_cast<int>(blockIdx.x);
    const int step = static_cast<int>(gridDim.x);
    const int n_my = first < total ? (total - first + step - 1) / step : 0;
    auto tile_xy = [&](int i, int& tx, int& ty) {
        const int t = first + i * step;
        ty = t / p.tiles_x;
        tx = t - ty * p.tiles_x;
    };
    auto issue_load = [&](int i) {
        const int s = i % STAGES;
        int tx, ty;
        tile_xy(i, tx, ty);
        mbar_arrive_expect_tx(full_bar(s), kTileBytes);
        tma_load_2d(sIn + s * kTileBytes, &src, full_bar(s), tx * kTT, ty * kTT);
    };

    const bool leader = elect_one();
    if (leader) {
        for (int s = 0; s < STAGES; ++s) mbar_init(full_bar(s), 1);
        *abort_flag = 0;
        fence_mbarrier_init();
        prefetch_tensormap(&src);
        prefetch_tensormap(&dst);
        const int pro = n_my < STAGES ? n_my : STAGES;
        for (int i = 0; i < pro; ++i) issue_load(i);
    }
    __syncwarp();

    int i = 0;
    for (; i < n_my; ++i) {
        const int s = i % STAGES;
        int ok = 1;
        if (leader)
            ok = wait_bounded(full_bar(s), static_cast<uint32_t>(i / STAGES) & 1u, p.wait, abort_flag,
                                     SITE_COPY_FULL);
        // The leader lane's result decides for the warp (elect_one's lane).
        ok = __any_sync(0xffffffffu, leader && ok) ? 1 : 0;
        if (!ok) break;
        const uint32_t ob = sOut + static_cast<uint32_t>(i & 1) * kTileBytes;
        if (leader) bulk_wait_group_read<1>();  // the store that last used `ob` has read it
        __syncwarp();
        const uint32_t ib = sIn + s * kTileBytes;
        const uint32_t q8 = lane >> 3, r8 = lane & 7u;
#pragma unroll 4
        for (int it = 0; it < 16; ++it) {
            const uint32_t q = static_cast<uint32_t>(it) * 4u + q8;  // 8x8 block index
            const uint32_t bi = q >> 3, bj = q & 7u;                 // block row / column in the tile
            const uint32_t srow = bi * 8u + r8;                      // src row this lane addresses
            uint32_t v[4];
            ldmatrix_x4(ib + srow * 128u + ((bj ^ (srow & 7u)) << 4), v);
            const uint32_t drow = bj * 8u + r8;                      // dst row (= src column)
            stmatrix_x4_trans(ob + drow * 128u + ((bi ^ (drow & 7u)) << 4), v);
        }
        fence_proxy_async_shared();
        __syncwarp();
        if (leader) {
            int tx, ty;
            tile_xy(i, tx, ty);
            tma_store_2d(&dst, ob, ty * kTT, tx * kTT);
            bulk_commit_group();
            if (i + STAGES < n_my) issue_load(i + STAGES);  // stage s is consumed
        }
        __syncwarp();
    }
    if (leader) {
        if (i < n_my) {
            // Gave up: let the loads in flight land (bounded) before exit.
            volatile int no_abort = 0;
            const int last = (i + STAGES < n_my ? i + STAGES : n_my);
            for (int k = i; k < last; ++k)
                wait_bounded(full_bar(k % STAGES), static_cast<uint32_t>(k / STAGES) & 1u, p.wait,
                                    &no_abort, SITE_DRAIN);
        }
        bulk_wait_group<0>();
    }
    __syncwarp();
}

int transpose_smem_bytes(int stages) { return 1024 + (stages + 2) * static_cast<int>(kTileBytes) + 8 * stages + 16; }

template <int STAGES>
cudaError_t launch_tma_transpose_t(const CUtensorMap& s, const CUtensorMap& d, const TransposeParams& p, int grid,
                                   cudaStream_t st)
{
    const int smem = transpose_smem_bytes(STAGES);
    auto kern = tma_transpose_kernel<STAGES>;
    static std::atomic<uint64_t> smem_set{0};
    cudaError_t e = smem_limit_once(kern, smem, smem_set);  // fixed per instantiation
    if (e != cudaSuccess) return e;
    kern<<<grid, 32, smem, st>>>(s, d, p);
    return cudaGetLastError();
}

cudaError_t launch_tma_transpose(int stages, const CUtensorMap& s, const CUtensorMap& d, int tiles_x, int tiles_y,
                                 const WaitCtl& w, int grid, cudaStream_t st)
{
    TransposeParams p{tiles_x, tiles_y, w};
    switch (stages) {
    case 2: return launch_tma_transpose_t<2>(s, d, p, grid, st);
    case 4: return launch_tma_transpose_t<4>(s, d, p, grid, st);
    case 6: return launch_tma_transpose_t<6>(s, d, p, grid, st);
    case 8: return launch_tma_transpose_t<8>(s, d, p, grid, st);
    default: return cudaErrorInvalidValue;
    }
}

// ------------------------------------------------------------ fallback ---

// dst[c * ld_dst + r] = src[r * ld_src + c] for r in [r0, r0 + rows),
// c < cols, for operands TMA cannot describe: 64x64 tiles through shared
// memory, 32 x 8 threads. A lane moves an element pair per row, as one
// 4-byte access where the pair is 4-byte aligned and as two 2-byte accesses
// otherwise. A thread's eight rows lie 8 pitches apart, a multiple of 16
// bytes, so they share that alignment: the choice is made once per tile,
// and all eight rows' loads are issued before any is used. Tile rows are
// 65 elements apart, so the transposed reads (element k of rows 2 lx and
// 2 lx + 1) hit distinct banks. Edge tiles check every element.
constexpr int kVecT = 64;

__global__ void __launch_bounds__(256)
    vec_transpose_kernel(const uint16_t* __restrict__ src, uint16_t* __restrict__ dst, int64_t r0, int64_t rows,
                         int64_t cols, int64_t ld_src, int64_t ld_dst)
{
    __shared__ uint16_t tile[kVecT][kVecT + 1];
    const int64_t tiles_c = (cols + kVecT - 1) / kVecT;
    const int64_t tiles_r = (rows + kVecT - 1) / kVecT;
    const int lx = static_cast<int>(threadIdx.x), ly = static_cast<int>(threadIdx.y);
    const int64_t r_end = r0 + rows;
    for (int64_t t = blockIdx.x; t < tiles_c * tiles_r; t += gridDim.x) {
        const int64_t tr = t / tiles_c, tc = t - tr * tiles_c;
        const int64_t rb = r0 + tr * kVecT, cb = tc * kVecT;
        const bool full = rb + kVecT <= r_end && cb + kVecT <= cols;
        // load: rows rb + ly + 8 i, columns cb + 2 lx, + 1
        const uint16_t* p0 = src + (rb + ly) * ld_src + cb + 2 * lx;
        if (full && (reinterpret_cast<uintptr_t>(p0) & 3u) == 0) {
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) w[i] = __ldg(reinterpret_cast<const unsigned int*>(p0 + 8 * i * ld_src));
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                tile[ly + 8 * i][2 * lx] = static_cast<uint16_t>(w[i] & 0xFFFFu);
                tile[ly + 8 * i][2 * lx + 1] = static_cast<uint16_t>(w[i] >> 16);
            }
        } else if (full) {
            // The row starts 2 bytes past a 4-byte boundary: lane lx loads
            // the aligned word holding elements 2 lx - 1 and 2 lx, and takes
            // element 2 lx + 1 from the next lane's word (lane 31 from one
            // more word). An aligned word holding one element of the row
            // lies in that element's page, so the extra halves never fault.
            const unsigned int* w0 = reinterpret_cast<const unsigned int*>(p0 - 1);
            uint32_t w[8], e[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                w[i] = __ldg(w0 + 4 * i * ld_src);
                e[i] = lx == 31 ? __ldg(w0 + 4 * i * ld_src + 1) : 0u;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uint32_t nxt = __shfl_down_sync(0xffffffffu, w[i], 1);
                if (lx == 31) nxt = e[i];
                tile[ly + 8 * i][2 * lx] = static_cast<uint16_t>(w[i] >> 16);
                tile[ly + 8 * i][2 * lx + 1] = static_cast<uint16_t>(nxt & 0xFFFFu);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int64_t r = rb + ly + 8 * i, c = cb + 2 * lx;
                uint16_t lo = 0, hi = 0;
                if (r < r_end) {
                    if (c < cols) lo = __ldg(p0 + 8 * i * ld_src);
                    if (c + 1 < cols) hi = __ldg(p0 + 8 * i * ld_src + 1);
                }
                tile[ly + 8 * i][2 * lx] = lo;
                tile[ly + 8 * i][2 * lx + 1] = hi;
            }
        }
        __syncthreads();
        // store: dst rows cb + ly + 8 i, columns (source rows) rb + 2 lx, + 1
        uint16_t* q0 = dst + (cb + ly) * ld_dst + rb + 2 * lx;
        if (full && (reinterpret_cast<uintptr_t>(q0) & 3u) == 0) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int k = ly + 8 * i;
                *reinterpret_cast<unsigned int*>(q0 + 8 * i * ld_dst) =
                    static_cast<uint32_t>(tile[2 * lx][k]) | (static_cast<uint32_t>(tile[2 * lx + 1][k]) << 16);
            }
        } else if (full) {
            // The row starts 2 bytes past a 4-byte boundary: lanes 1-31 each
            // write the aligned word of elements 2 lx - 1 and 2 lx; the tile's
            // first and last elements, whose words they share with the
            // neighbouring tiles, are written alone.
            unsigned int* qw = reinterpret_cast<unsigned int*>(q0 - 1);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int k = ly + 8 * i;
                if (lx == 0)
                    q0[8 * i * ld_dst] = tile[0][k];
                else
                    qw[4 * i * ld_dst] = static_cast<uint32_t>(tile[2 * lx - 1][k]) |
                                         (static_cast<uint32_t>(tile[2 * lx][k]) << 16);
                if (lx == 31) q0[8 * i * ld_dst + 1] = tile[kVecT - 1][k];
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int k = ly + 8 * i;
                const int64_t c = cb + k, r = rb + 2 * lx;
                if (c < cols && r < r_end) {
                    q0[8 * i * ld_dst] = tile[2 * lx][k];
                    if (r + 1 < r_end) q0[8 * i * ld_dst + 1] = tile[2 * lx + 1][k];
                }
            }
        }
        __syncthreads();
    }
}

cudaError_t launch_vec_transpose(const void* src, void* dst, int64_t r0, int64_t rows, int64_t cols, int64_t ld_src,
                                 int64_t ld_dst, int sm_count, cudaStream_t st)
{
    const int64_t tiles = ((rows + kVecT - 1) / kVecT) * ((cols + kVecT - 1) / kVecT);
    int64_t grid = static_cast<int64_t>(sm_count) * 8;
    if (grid > tiles) grid = tiles;
    if (grid < 1) grid = 1;
    vec_transpose_kernel<<<static_cast<unsigned>(grid), dim3(32, 8), 0, st>>>(
        static_cast<const uint16_t*>(src), static_cast<uint16_t*>(dst), r0, rows, cols, ld_src, ld_dst);
    return cudaGetLastError();
}

}  // namespace tp
