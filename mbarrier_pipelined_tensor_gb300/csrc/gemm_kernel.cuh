// Warp-specialized, persistent, TMA-fed tcgen05 BF16 mainloop: C = A.B with
// fp32 accumulation in TMEM, and its implicit-GEMM (im2col) convolution form.
//
// Roles (192 threads, 6 warps):
//   warp 0      producer: the lane picked by elect.sync waits for a free
//               stage, posts arrive.expect_tx on the stage's full barrier and
//               issues the TMA loads -- the same thread does both, so the one
//               arrival a stage expects always comes from the issuing lane
//               (CUTLASS issue #3722, "Expected behavior").
//   warp 1      MMA issuer and TMEM owner: waits full[s], issues 4 tcgen05.mma
//               (K = 16 each) per 64-deep stage, commits to empty[s]; after a
//               tile's last stage commits to acc_full[b].
//   warps 2..5  epilogue: wait acc_full[b], read TMEM with tcgen05.ld, free
//               the accumulator (acc_empty[b]) as soon as it is read, convert,
//               stage through swizzled shared memory and write C with TMA
//               stores drained by commit_group / wait_group.
//
// Stage ring ("B200 Tma Pipeline Designer", steps 4-7): PIPE_DEPTH stages of
// A (128x64 bf16) and B; full[s] / empty[s] each have exactly one producer
// and one consumer; initial phases let the producer's first pass through the
// ring run without waiting. Two TMEM accumulators let the epilogue of tile
// t-1 overlap the mainloop of tile t (the "store k-1" of the steady state).
//
// Plain-load producer (LDG = true, 1-SM only): for operands TMA cannot
// describe directly ("B200 Tma Pipeline Designer", step 1: keep the
// vectorized thread copy). A row's 64-element K segment starts at an address
// that is only 2-byte aligned, so the producer stages the 144-byte window of
// 16-byte aligned chunks around it, then shifts each row into place and
// writes it in the same 128-byte-swizzled layout TMA would produce; each
// unpacking warp fences its generic-proxy writes for the tensor core's
// async-proxy reads and makes one arrival on the stage's full barrier.
//   GEMM: rows r and r + 8 of an operand lie a multiple of 16 bytes apart,
//   so each row class r mod 8 is a tensor TMA can load (WinMaps). Warp 0's
//   elected lane loads a stage's windows, 16 boxes of 72 x 16 elements, into
//   one of three staging buffers; eight warps (6-13) unpack them.
//   Conv: the im2col rows follow no such pattern; eight producer warps (0
//   and 6-12) copy each row's window with cp.async (the copies of the next
//   stage go out before the current one is unpacked), then unpack it. The
//   epilogue writes the conv's C with plain stores.
//
// Atoms ("two-free-pipeline-stages" note): CG = 1 is the 1-SM atom (each CTA
// owns a 128 x BN tile and holds all of its B tile); CG = 2 is the 2-SM atom
// (a CTA pair owns 256 x BN, the leader issues cta_group::2 MMAs, and each
// CTA holds only its half of B, which is what frees shared memory for more
// stages at the same budget).
#pragma once

#include <cuda_bf16.h>

#include <type_traits>

#include "common.cuh"

namespace tp {

template <int CG, int BN, int STAGES, bool OUT_F32>
struct MainloopCfg {
    static constexpr int BM = 128;  // rows per CTA (TMEM lanes)
    static constexpr int BK = 64;   // one 128-byte swizzle row of bf16
    static constexpr int UMMA_K = 16;
    static constexpr int B_ROWS = BN / CG;
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = B_ROWS * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TX_BYTES = STAGE_BYTES * CG;  // the leader's expect_tx covers the pair
    // A narrow unit (the 2-SM, N = 256 narrow tail: a half or a quarter of a
    // tile's columns) loads that share of each CTA's B rows through a box of
    // that height.
    static constexpr int TX_HALF_BYTES = (A_BYTES + B_BYTES / 2) * CG;
    static constexpr int TX_QUARTER_BYTES = (A_BYTES + B_BYTES / 4) * CG;
    static constexpr int OUT_BYTES = OUT_F32 ? 4 : 2;
    static constexpr int EPI_COLS = 128 / OUT_BYTES;  // columns per 128-byte staging row
    static constexpr int EPI_WARPS = 4;
    static constexpr int EPI_BUF = 32 * 128;  // one warp's 32 rows x 128 B
    static constexpr int EPI_BYTES = EPI_WARPS * 2 * EPI_BUF;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES;
    static constexpr int THREADS = 192;

    static_assert(BN % (16 * CG) == 0 && BN >= 32 && BN <= 256, "UMMA N");
    static_assert(B_BYTES % 1024 == 0, "B stage must hold whole swizzle atoms");
    static_assert(TMEM_COLS == 64 || TMEM_COLS == 128 || TMEM_COLS == 256 || TMEM_COLS == 512,
                  "TMEM allocation must be a power of two");
    static_assert(BN % EPI_COLS == 0, "epilogue chunking");
    static_assert(2 * STAGES + 5 <= (BAR_BYTES - 8) / 8, "barrier area");
    static_assert(STAGES <= PROTO_MAX_STAGES, "arrival accounting layout");
};

__device__ __forceinline__ void tile_coords(int t, const GemmParams& p, int& mt, int& nt)
{
    const int g = fdiv(t, p.div_group);
    const int first = g * p.group_m;
    // the last group may hold fewer M-tiles
    const FastDiv& dgm = first + p.group_m > p.m_tiles ? p.div_gm_last : p.div_gm;
    const int r = t - g * static_cast<int>(p.div_group.d);
    // odd groups sweep N from the far end, starting on the B columns the
    // group before ended on
    const int n = fdiv(r, dgm);
    mt = first + (r - n * static_cast<int>(dgm.d));
    nt = (g & 1) ? p.n_tiles - 1 - n : n;
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo_bits, uint32_t hi_bits)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// The plain-load producer: producer (or, for the GEMM, unpacking) warps,
// and for the conv's cp.async form its staging buffers (each holds a
// stage's rows as 144-byte windows of aligned 16-byte chunks, then one
// 32-bit code per row) and ring depth.
constexpr int kLdgWarps = 8;
constexpr int kLdgStaging = 2;
constexpr int kLdgStages = 3;
constexpr int kLdgWindow = 144;

template <int B_ROWS>
__host__ __device__ constexpr int ldg_staging_buffer_bytes()
{
    return (128 + B_ROWS) * (kLdgWindow + 4);
}

template <int B_ROWS>
__host__ __device__ constexpr int ldg_staging_bytes()
{
    return kLdgStaging * ldg_staging_buffer_bytes<B_ROWS>();
}

// The plain-load GEMM stages through row-class windows (WinMaps) instead:
// a staging buffer holds a stage's rows as 144-byte windows that TMA writes
// class by class (A: 8 classes of 16 rows, then B: 8 classes of B_ROWS / 8),
// and the buffers' full / empty barriers follow them.
constexpr int kWinRow = 144;      // GEMM windows: 72 elements, K blocks start on 16-byte boundaries
constexpr int kWinRowConv = 160;  // conv windows: 80 elements, a filter's K blocks need not
constexpr int kWinStaging = 3;    // staging buffers: the window loads run two stages ahead
constexpr int kWinStages = 2;     // ring stages (the tensor core drains one long before the next is unpacked)

// Plain-load forms (the LDG template argument): 0 none (TMA producer), 1 the
// GEMM's row-class windows or the conv's cp.async windows, 2 the conv's
// row-class windows (stride 1, output the size of the input).
constexpr int kLdgNone = 0, kLdgPlain = 1, kLdgConvWin = 2;

template <int B_ROWS, int ROW>
__host__ __device__ constexpr int win_staging_buffer_bytes()
{
    return (128 + B_ROWS) * ROW;
}

// The buffers, their full / empty barriers (64 bytes) and, for the conv,
// one 16-byte record per buffer of its K block's tap facts (WinConvStage).
template <int B_ROWS, int ROW>
__host__ __device__ constexpr int win_staging_bytes()
{
    return kWinStaging * win_staging_buffer_bytes<B_ROWS, ROW>() + 64 + (ROW == kWinRowConv ? 16 * kWinStaging : 0);
}

// Shared memory a plain-load variant adds to the ring: the conv's cp.async
// staging, or the row-class windows of the GEMM or the conv.
template <int B_ROWS, bool CONV, int LDG>
__host__ __device__ constexpr int ldg_extra_bytes()
{
    return LDG == kLdgConvWin ? win_staging_bytes<B_ROWS, kWinRowConv>()
                              : (CONV ? ldg_staging_bytes<B_ROWS>() : win_staging_bytes<B_ROWS, kWinRow>());
}

// Row of the stage that lane `sub` (0..3) of a producer warp handles in row
// quad q: the quad's four rows are 8 apart, so that in a GEMM operand
// (whose row pitch repeats its 16-byte alignment every 8 rows) all four
// shift by the same amount.
__device__ __forceinline__ int ldg_row(int pw, int rpw, int q, int sub)
{
    return pw * rpw + (q & 7) + 8 * (4 * (q >> 3) + sub);
}

// The conv's cp.async form: where stage row `row` (A: rows 0..127, the
// im2col rows of output pixels; B: 128.., filters) of K block kb comes from:
// the address of its first element (0 when the row is out of range or
// padding) and the number of valid channels from there (1..64). The operand
// fields are copied out of the kernel parameters once.
struct ConvRows {
    const uint16_t* A;
    const uint16_t* B;
    int M, N, m_row, n_row, c0, r, sx, nvalid;
    int P, Q, H, W, C, R, S, stride, pad;
    FastDiv div_pq, div_q;

    __device__ __forceinline__ ConvRows(const GemmParams& p, int m0, int n0, int kb)
        : A(p.A), B(p.B), M(p.M), N(p.N), m_row(m0), n_row(n0)
    {
        const int rs = fdiv(kb, p.div_cblocks);
        c0 = (kb - rs * p.conv_cblocks) * 64;
        r = fdiv(rs, p.div_s);
        sx = rs - r * p.conv_S;
        P = p.conv_P;
        Q = p.conv_Q;
        H = p.conv_H;
        W = p.conv_W;
        C = p.conv_C;
        R = p.conv_R;
        S = p.conv_S;
        stride = p.conv_stride;
        pad = p.conv_pad;
        div_pq = p.div_pq;
        div_q = p.div_q;
        nvalid = (C - c0) < 64 ? (C - c0) : 64;  // >= 1: c0 < C
    }

    __device__ __forceinline__ uintptr_t segment(int row) const
    {
        if (row < 128) {
            const int m = m_row + row;
            const int img = fdiv(m, div_pq);
            const int rem = m - img * P * Q;
            const int pp = fdiv(rem, div_q);
            const int qq = rem - pp * Q;
            const int h = pp * stride - pad + r;
            const int w = qq * stride - pad + sx;
            if (m >= M || h < 0 || h >= H || w < 0 || w >= W) return 0;
            return reinterpret_cast<uintptr_t>(A + ((static_cast<int64_t>(img) * H + h) * W + w) * C + c0);
        }
        const int n = n_row + (row - 128);
        if (n >= N) return 0;
        return reinterpret_cast<uintptr_t>(B + ((static_cast<int64_t>(n) * R + r) * S + sx) * C + c0);
    }
};

// Issues the cp.async copies of rows [pw * RPW, pw * RPW + RPW) of one stage
// into staging buffer `stg`. Lane i first works out row pw * RPW + i: the
// address of its segment rounded down to 16 bytes, and its code -- the
// window's first valid byte (a & 15) and one past its last (0: row out of
// range). The warp's 32 x 9 aligned 16-byte chunks are then copied in nine
// fully populated instructions, lane i of instruction k taking chunk
// (32 k + i) mod 9 of row (32 k + i) / 9. A chunk is copied only if it holds
// at least one element of the row's valid range, so no access touches a
// 16-byte block outside the operand (and none crosses a page).
template <int B_ROWS, int RPW>
__device__ __forceinline__ void ldg_issue_rows(const ConvRows& rows, uint32_t stg, int pw, uint32_t lane)
{
    static_assert(RPW == 32, "one row per lane");
    const uint32_t codes = stg + (128 + B_ROWS) * kLdgWindow;
    const int myrow = pw * RPW + static_cast<int>(lane);
    const uintptr_t a = rows.segment(myrow);
    const uint32_t mis = static_cast<uint32_t>(a & 15u);
    const uint32_t end = a ? mis + 2u * static_cast<uint32_t>(rows.nvalid) : 0u;
    st_shared_u32(codes + 4u * static_cast<uint32_t>(myrow), mis | (end << 8));
    const uint64_t base = static_cast<uint64_t>(a - mis);
    const uint32_t base_lo = static_cast<uint32_t>(base), base_hi = static_cast<uint32_t>(base >> 32);
    const uint32_t stg_warp = stg + static_cast<uint32_t>(pw * RPW) * kLdgWindow;
#pragma unroll
    for (int k = 0; k < kLdgWindow / 16; ++k) {
        const uint32_t g = 32u * static_cast<uint32_t>(k) + lane;
        const uint32_t r = g / 9u, ch = g - 9u * r;
        const uint32_t e = __shfl_sync(0xffffffffu, end, static_cast<int>(r));
        const uint32_t lo = __shfl_sync(0xffffffffu, base_lo, static_cast<int>(r));
        const uint32_t hi = __shfl_sync(0xffffffffu, base_hi, static_cast<int>(r));
        const uint64_t src = (static_cast<uint64_t>(hi) << 32) | lo;
        if (16u * ch < e) cp_async_16(stg_warp + r * kLdgWindow + 16u * ch, static_cast<uintptr_t>(src + 16u * ch));
    }
}

// Shifts the staged rows [pw * RPW, pw * RPW + RPW) into place: output chunk
// j of a row is bytes (a & 15) + 16 j .. + 15 of its window, picked with
// word selects and a 16-bit funnel shift. Chunks that were not copied,
// elements past the valid range and rows out of range read as zero, as
// TMA's fill would.
template <int B_ROWS, int RPW>
__device__ __forceinline__ void ldg_repack_rows(uint32_t stg, int nvalid, uint32_t dA, uint32_t dB, int pw,
                                                uint32_t lane)
{
    const int sub = static_cast<int>(lane >> 3);
    const uint32_t j = lane & 7u;
    const uint32_t codes = stg + (128 + B_ROWS) * kLdgWindow;
    const bool full_k = nvalid == 64;
    constexpr int kQuads = RPW / 4;
    // every quad's shared-memory reads first, so their latencies overlap
    uint32_t mis[kQuads], end[kQuads];
    uint4 lo[kQuads], hi[kQuads];
#pragma unroll
    for (int q = 0; q < kQuads; ++q) {
        const int row = ldg_row(pw, RPW, q, sub);
        const uint32_t code = ld_shared_u32(codes + 4u * static_cast<uint32_t>(row));
        mis[q] = code & 0xFFu;
        end[q] = code >> 8;
    }
#pragma unroll
    for (int q = 0; q < kQuads; ++q) {
        const int row = ldg_row(pw, RPW, q, sub);
        const uint32_t src = stg + static_cast<uint32_t>(row) * kLdgWindow + 16u * j;
        lo[q] = 16u * j < end[q] ? ld_shared_v4(src) : make_uint4(0u, 0u, 0u, 0u);
        hi[q] = 16u * (j + 1u) < end[q] ? ld_shared_v4(src + 16u) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int q = 0; q < kQuads; ++q) {
        const int row = ldg_row(pw, RPW, q, sub);
        uint32_t c[8] = {lo[q].x, lo[q].y, lo[q].z, lo[q].w, hi[q].x, hi[q].y, hi[q].z, hi[q].w};
        // drop (mis >> 2) whole words, then shift by (mis & 2) bytes
        if (mis[q] & 8u) {
#pragma unroll
            for (int i = 0; i < 6; ++i) c[i] = c[i + 2];
        }
        if (mis[q] & 4u) {
#pragma unroll
            for (int i = 0; i < 5; ++i) c[i] = c[i + 1];
        }
        const uint32_t sh = (mis[q] & 2u) << 3;  // 0 or 16 bits
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) o[k] = __funnelshift_r(c[k], c[k + 1], sh);
        if (!full_k) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                // columns 8 j + 2 k and 8 j + 2 k + 1 past the valid range read as zero
                const int col = static_cast<int>(8u * j) + 2 * k;
                if (col >= nvalid) o[k] = 0u;
                else if (col + 1 >= nvalid) o[k] &= 0xFFFFu;
            }
        }
        const int rr = row < 128 ? row : row - 128;
        const uint32_t dst = (row < 128 ? dA : dB) + static_cast<uint32_t>(rr) * 128u +
                             ((j ^ (static_cast<uint32_t>(rr) & 7u)) << 4);
        st_shared_v4(dst, o[0], o[1], o[2], o[3]);
    }
}

// Per-stage facts the conv's row-class windows add: the tap's pixel offset
// (input pixel of tile row t is pixel m0 + t + off), B's window start below
// its K block (xd elements, 0..7), the valid channels of the K block, and
// which of the lane's eight A rows lie inside the image (bit q).
struct WinConvStage {
    int off;
    uint32_t xd;
    int nvalid;
    uint32_t row_ok;
};

// Shifts the TMA-staged windows of stage rows [pw * RPW, pw * RPW + RPW)
// into place (row-class windows). B row rr (class rr & 7, row rr >> 3 of its
// class) is window cls * rows / 8 + (rr >> 3) of B's part of the buffer. A
// row t is window cls * 16 + (t >> 3) of A's part, cls = t & 7 for the GEMM
// and (t + off) & 7 for the conv, whose pixels for a tap start `off` pixels
// from the tile's. A window holds the row's elements shifted right by its
// class's offset (plus, for the conv's B, xd), up to 30 bytes: output chunk
// j is bytes mis .. mis + 15 of window chunks j + mis / 16 and the next.
// TMA has zero-filled what lies past the end of a row or past the last
// row; the conv also zeroes A rows outside the image (padding) and B
// columns past the K block's channels (they belong to the next tap). Lanes
// pair up as in ldg_repack_rows: the four rows of a quad are 8 apart, so
// they share a class and a shift.
template <int B_ROWS, int RPW, int ROW, bool CONVW>
__device__ __forceinline__ void win_repack_rows(uint32_t stg, uint32_t dA, uint32_t dB, int pw, uint32_t lane,
                                                uint32_t delta_a, uint32_t delta_b, const WinConvStage cs)
{
    const int sub = static_cast<int>(lane >> 3);
    const uint32_t j = lane & 7u;
    constexpr int kQuads = RPW / 4;
    uint32_t mis[kQuads];
    uint4 lo[kQuads], hi[kQuads];
#pragma unroll
    for (int q = 0; q < kQuads; ++q) {
        const int row = ldg_row(pw, RPW, q, sub);
        const bool is_a = row < 128;
        const int rr = is_a ? row : row - 128;
        const int cls = CONVW && is_a ? ((rr + cs.off) & 7) : (rr & 7);
        const int win = (is_a ? cls * 16 : 128 + cls * (B_ROWS / 8)) + (rr >> 3);
        mis[q] = 2u * (((is_a ? delta_a : delta_b) >> (3 * cls)) & 7u);
        if constexpr (CONVW) {
            if (!is_a) mis[q] += 2u * cs.xd;
        }
        const uint32_t src = stg + static_cast<uint32_t>(win) * ROW + 16u * (j + (mis[q] >> 4));
        lo[q] = ld_shared_v4(src);
        hi[q] = ld_shared_v4(src + 16u);
    }
#pragma unroll
    for (int q = 0; q < kQuads; ++q) {
        const int row = ldg_row(pw, RPW, q, sub);
        uint32_t c[8] = {lo[q].x, lo[q].y, lo[q].z, lo[q].w, hi[q].x, hi[q].y, hi[q].z, hi[q].w};
        if (mis[q] & 8u) {
#pragma unroll
            for (int i = 0; i < 6; ++i) c[i] = c[i + 2];
        }
        if (mis[q] & 4u) {
#pragma unroll
            for (int i = 0; i < 5; ++i) c[i] = c[i + 1];
        }
        const uint32_t sh = (mis[q] & 2u) << 3;
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) o[k] = __funnelshift_r(c[k], c[k + 1], sh);
        if constexpr (CONVW) {
            if (row < 128) {
                const uint32_t keep = 0u - ((cs.row_ok >> q) & 1u);  // all ones or zero
#pragma unroll
                for (int k = 0; k < 4; ++k) o[k] &= keep;
            } else if (cs.nvalid < 64) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int col = static_cast<int>(8u * j) + 2 * k;
                    if (col >= cs.nvalid) o[k] = 0u;
                    else if (col + 1 >= cs.nvalid) o[k] &= 0xFFFFu;
                }
            }
        }
        const int rr = row < 128 ? row : row - 128;
        const uint32_t dst = (row < 128 ? dA : dB) + static_cast<uint32_t>(rr) * 128u +
                             ((j ^ (static_cast<uint32_t>(rr) & 7u)) << 4);
        st_shared_v4(dst, o[0], o[1], o[2], o[3]);
    }
}

// Work unit u of a launch: output tile, its K-block range, and which part
// of the tile's columns it covers (-1: the whole tile; else one of
// p.tail_parts equal column parts of a narrow-tail tile).
struct Unit {
    int tile, split, kb0, kb1, part;
};

__device__ __forceinline__ Unit unit_of(int u, int num_tiles, const GemmParams& p)
{
    Unit w;
    if (p.tail_units > 0 && u >= p.n_full) {
        const int v = u - p.n_full;
        w.tile = p.n_full + (v >> (p.tail_parts == 4 ? 2 : 1));  // 2 or 4 parts
        w.part = v - (w.tile - p.n_full) * p.tail_parts;
        w.split = 0;
        w.kb0 = 0;
        w.kb1 = p.k_blocks;
        return w;
    }
    w.split = p.splits == 1 ? 0 : fdiv(u, p.div_tiles);
    w.tile = u - w.split * num_tiles;
    w.kb0 = w.split * p.kb_per_split;
    w.kb1 = min(p.k_blocks, w.kb0 + p.kb_per_split);
    w.part = -1;
    return w;
}

// Role timeline: adds `v` to this CTA's counter `slot` when tracing is on.
__device__ __forceinline__ void trace_add(const GemmParams& p, int slot, unsigned long long v)
{
    if (p.trace) atomicAdd(p.trace + static_cast<size_t>(blockIdx.x) * kTraceSlots + slot, v);
}

// Per-unit event timeline: this CTA's slot for event `ev` of its lt-th unit.
__device__ __forceinline__ void event_at(const GemmParams& p, int lt, int ev, unsigned long long v)
{
    if (p.events && lt < kEventUnits)
        p.events[static_cast<size_t>(blockIdx.x) * kEventSlots + lt * kEventsPerUnit + ev] = v;
}

// Bounded wait that charges its duration to a timeline slot.
__device__ __forceinline__ bool timed_wait(const GemmParams& p, uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           int site, unsigned long long& acc)
{
    if (!p.trace) return wait_bounded(bar, parity, p.wait, abort_flag, site);
    const uint64_t t0 = globaltimer_ns();
    const bool ok = wait_bounded(bar, parity, p.wait, abort_flag, site);
    acc += globaltimer_ns() - t0;
    return ok;
}

// Threads of a mainloop CTA: producer, MMA issuer, four epilogue warps;
// with the plain-load producer kLdgWarps - 1 more producer warps (conv) or
// kLdgWarps window-unpacking warps beside the window-loading warp 0 (GEMM).
template <int LDG, bool CONV = false>
__host__ __device__ constexpr int mainloop_threads()
{
    return !LDG ? 192 : ((CONV && LDG == kLdgPlain) ? 192 + 32 * (kLdgWarps - 1) : 192 + 32 * kLdgWarps);
}

struct NoWinMaps {
    int unused;
};

// Row-class windows are loaded by TMA: the plain-load GEMM, and the conv's
// form for stride-1 convolutions whose output is the input's size.
template <bool CONV, int LDG>
__host__ __device__ constexpr bool win_form()
{
    return (LDG == kLdgPlain && !CONV) || LDG == kLdgConvWin;
}

template <int CG, int BN, int STAGES, bool OUT_F32, bool CONV, int LDG = kLdgNone, bool SPLITK = false>
__global__ void __launch_bounds__(mainloop_threads<LDG, CONV>(), 1)
    mainloop_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                    const __grid_constant__ CUtensorMap mapC, const __grid_constant__ CUtensorMap mapBh,
                    const GemmParams p,
                    const __grid_constant__ std::conditional_t<win_form<CONV, LDG>(), WinMaps, NoWinMaps> wm)
{
    using Cfg = MainloopCfg<CG, BN, STAGES, OUT_F32>;
    constexpr bool WIN = win_form<CONV, LDG>();  // row-class windows by TMA
    constexpr bool CWIN = LDG == kLdgConvWin;    // ... of a convolution
    constexpr int WROW = CWIN ? kWinRowConv : kWinRow;
    constexpr bool CL = (CG == 2);
    static_assert(!LDG || CG == 1, "the plain-load producer feeds the 1-SM atom");
    static_assert(!SPLITK || (OUT_F32 && !CONV), "split-K writes fp32 GEMM partials");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // 128B-swizzle atoms need 1024-B alignment
    uint8_t* const base_ptr = smem_raw + (base - raw);

    const uint32_t sA = base;
    const uint32_t sB = sA + STAGES * Cfg::A_BYTES;
    const uint32_t sEpi = sB + STAGES * Cfg::B_BYTES;
    const uint32_t sBar = sEpi + Cfg::EPI_BYTES;
    auto full_bar = [&](int s) { return sBar + 8u * s; };
    auto empty_bar = [&](int s) { return sBar + 8u * (STAGES + s); };
    auto accf_bar = [&](int b) { return sBar + 8u * (2 * STAGES + b); };
    auto acce_bar = [&](int b) { return sBar + 8u * (2 * STAGES + 2 + b); };
    const uint32_t drain_bar = sBar + 8u * (2 * STAGES + 4);
    uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + (sBar - base) + 8 * (2 * STAGES + 5));
    volatile int* const abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) / 32, 0);
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t rank = CL ? cluster_ctarank() : 0u;
    const bool leader = (rank == 0);

    // ------------------------------------------------------------ setup ---
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            // one arrival: the producer's expect_tx (plain loads: one per producer warp)
            mbar_init(full_bar(s), LDG ? kLdgWarps : 1);
            mbar_init(empty_bar(s), 1);  // one arrival: the MMA issuer's commit
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), Cfg::EPI_WARPS * CG);
        }
        mbar_init(drain_bar, 1);
        if constexpr (WIN) {
            // staging buffers: filled by the window loads (one expect_tx),
            // freed by every unpacking warp
            const uint32_t sw = sBar + Cfg::BAR_BYTES + kWinStaging * win_staging_buffer_bytes<Cfg::B_ROWS, WROW>();
            for (int i = 0; i < kWinStaging; ++i) {
                mbar_init(sw + 8u * i, 1);
                mbar_init(sw + 8u * (kWinStaging + i), kLdgWarps);
            }
        }
        *abort_flag = 0;
        fence_mbarrier_init();
        if constexpr (!LDG) {
            prefetch_tensormap(&mapA);
            prefetch_tensormap(&mapB);
            prefetch_tensormap(&mapC);
            if (CG == 2 && BN == 256 && p.tail_units > 0) prefetch_tensormap(&mapBh);
        }
        if constexpr (WIN) {
            for (int q = 0; q < 8; ++q) {
                prefetch_tensormap(&wm.a[q]);
                prefetch_tensormap(&wm.b[q]);
            }
            if (p.n_tma > 0) prefetch_tensormap(&mapC);
        }
    }
    if (warp == 1) {
        tmem_alloc<CG>(smem_u32(tmem_slot), Cfg::TMEM_COLS);
        tmem_relinquish<CG>();
    }
    tcgen05_fence_before();
    if constexpr (CL) cluster_sync(); else __syncthreads();
    tcgen05_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // The setup above may overlap the tail of the kernel launched before
    // this one on the stream (programmatic dependent launch); global memory
    // is touched only after that kernel has completed. From here on, the
    // kernel queued behind this one may be scheduled (the split-K
    // reduction, which waits for this grid's end in the same way).
    griddep_wait();
    griddep_launch_dependents();

    const int num_tiles = p.m_tiles * p.n_tiles;
    const int num_units = p.tail_units > 0 ? p.n_full + p.tail_units : num_tiles * p.splits;
    const int cluster_id = static_cast<int>(blockIdx.x) / CG;
    const int num_clusters = static_cast<int>(gridDim.x) / CG;

    if (WIN && warp == 0) {
        // -------------------------------------- window loads ---
        if constexpr (WIN) {
            if (elect_one()) {
                constexpr uint32_t STG = static_cast<uint32_t>(win_staging_buffer_bytes<Cfg::B_ROWS, WROW>());
                constexpr int BPC = Cfg::B_ROWS / 8;  // B rows per class in a tile
                const uint32_t sStg = sBar + Cfg::BAR_BYTES;
                const uint32_t sw = sStg + kWinStaging * STG;
                int slot = 0, issued = 0;
                uint32_t sph = 0;
                bool ok = true;
                for (int u = cluster_id; ok && u < num_units; u += num_clusters) {
                    const Unit w = unit_of(u, num_tiles, p);
                    int mt, nt;
                    tile_coords(w.tile, p, mt, nt);
                    // a tile's rows are whole classes' rows m0 / 8 .. m0 / 8 + 15
                    const int m0 = mt * Cfg::BM, yb = nt * BPC;
                    for (int kb = w.kb0; kb < w.kb1; ++kb) {
                        const uint32_t fb = sw + 8u * slot;
                        if (!wait_bounded(sw + 8u * (kWinStaging + slot), sph ^ 1u, p.wait, abort_flag,
                                          SITE_PRODUCER_EMPTY)) {
                            ok = false;
                            break;
                        }
                        const uint32_t dst = sStg + slot * STG;
                        if constexpr (CWIN) {
                            // K block kb is channels c0 .. c0 + 63 of tap (r, s). Tile
                            // row t reads pixel m0 + t + off: for class q the rows
                            // t = ((q - off) & 7) + 8 i, i < 16, a class-row run.
                            const int rs = fdiv(kb, p.div_cblocks);
                            const int c0 = (kb - rs * p.conv_cblocks) * Cfg::BK;
                            const int r = fdiv(rs, p.div_s), sx = rs - r * p.conv_S;
                            const int off = (r - p.conv_pad) * p.conv_W + (sx - p.conv_pad);
                            const int xb = rs * p.conv_C + c0;  // the K block within a filter row
                            // the unpacking warps read these with the windows (the
                            // arrival below releases them)
                            const int nv = p.conv_C - c0 < Cfg::BK ? p.conv_C - c0 : Cfg::BK;
                            st_shared_v4(sw + 64u + 16u * slot, static_cast<uint32_t>(off), static_cast<uint32_t>(xb & 7),
                                         static_cast<uint32_t>(nv),
                                         static_cast<uint32_t>(r) | (static_cast<uint32_t>(sx) << 16));
                            mbar_arrive_expect_tx(fb, STG);
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                tma_load_2d(dst + q * 16 * WROW, &wm.a[q], fb, c0, (m0 + off + ((q - off) & 7)) >> 3);
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                tma_load_2d(dst + (128 + q * BPC) * WROW, &wm.b[q], fb, xb & ~7, yb);
                        } else {
                            mbar_arrive_expect_tx(fb, STG);
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                tma_load_2d(dst + q * 16 * WROW, &wm.a[q], fb, kb * Cfg::BK, m0 >> 3);
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                tma_load_2d(dst + (128 + q * BPC) * WROW, &wm.b[q], fb, kb * Cfg::BK, yb);
                        }
                        ++issued;
                        if (++slot == kWinStaging) {
                            slot = 0;
                            sph ^= 1u;
                        }
                    }
                }
                if (!ok) {
                    // Gave up: let the loads in flight land first (bounded).
                    volatile int no_abort = 0;
                    const int n = issued < kWinStaging ? issued : kWinStaging;
                    for (int i = 0; i < n; ++i) {
                        if (--slot < 0) {
                            slot = kWinStaging - 1;
                            sph ^= 1u;
                        }
                        wait_bounded(sw + 8u * slot, sph, p.wait, &no_abort, SITE_DRAIN);
                    }
                }
            }
            __syncwarp();
        }
    } else if (WIN && warp >= 6) {
        // ------------------------------------ window unpacking ---
        if constexpr (WIN) {
            const int pw = warp - 6;
            constexpr int RPW = (128 + Cfg::B_ROWS) / kLdgWarps;
            constexpr uint32_t STG = static_cast<uint32_t>(win_staging_buffer_bytes<Cfg::B_ROWS, WROW>());
            const uint32_t sStg = sBar + Cfg::BAR_BYTES;
            const uint32_t sw = sStg + kWinStaging * STG;
            int s = 0, it = 0, slot = 0;
            uint32_t ph = 0, sph = 0;
            bool ok = true;
            WinConvStage cs{0, 0u, 64, 0xFFFFFFFFu};
            for (int u = cluster_id; ok && u < num_units; u += num_clusters) {
                const Unit w = unit_of(u, num_tiles, p);
                // conv, A warps: where the lane's eight rows (t = 32 pw + q + 8 sub)
                // sit in the output image, minus the padding
                [[maybe_unused]] int hq[8] = {}, wq[8] = {};
                [[maybe_unused]] uint32_t tap_seen = 0xFFFFFFFFu;  // the tap row_ok was last worked out for
                if (CWIN && pw < 4) {
                    int mt, nt;
                    tile_coords(w.tile, p, mt, nt);
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int m = mt * Cfg::BM + pw * 32 + q + 8 * static_cast<int>(lane >> 3);
                        const int img = fdiv(m, p.div_pq);
                        const int rem = m - img * static_cast<int>(p.div_pq.d);
                        const int pp = fdiv(rem, p.div_q);
                        hq[q] = m < p.M ? pp - p.conv_pad : -(1 << 29);  // rows past M read as padding
                        wq[q] = rem - pp * p.conv_Q - p.conv_pad;
                    }
                }
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    const uint32_t fb = sw + 8u * slot;
                    int good = 1;
                    if (lane == 0)
                        good = wait_bounded(fb, sph, p.wait, abort_flag, SITE_COPY_FULL) &&
                               wait_bounded(empty_bar(s), ph ^ 1u, p.wait, abort_flag, SITE_PRODUCER_EMPTY);
                    if (!__shfl_sync(0xffffffffu, good, 0)) {
                        ok = false;
                        break;
                    }
                    // lane 0 saw the windows land; the phase cannot move on
                    // before this warp frees the buffer, so every lane's own
                    // wait returns at once and orders its reads after the copy
                    for (int i = 0; i < 1024 && !mbar_try_wait(fb, sph); ++i) {
                    }
                    if constexpr (CWIN) {
                        const uint4 rec = ld_shared_v4(sw + 64u + 16u * slot);
                        const int r = static_cast<int>(rec.w & 0xFFFFu), sx = static_cast<int>(rec.w >> 16);
                        cs.off = static_cast<int>(rec.x);
                        cs.xd = rec.y;
                        cs.nvalid = static_cast<int>(rec.z);
                        if (rec.w != tap_seen) {
                            // a new tap (the channel blocks of one tap share it)
                            tap_seen = rec.w;
                            uint32_t ok = 0u;
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                const uint32_t in_h =
                                    static_cast<uint32_t>(hq[q] + r) < static_cast<uint32_t>(p.conv_H);
                                const uint32_t in_w =
                                    static_cast<uint32_t>(wq[q] + sx) < static_cast<uint32_t>(p.conv_W);
                                ok |= (in_h & in_w) << q;
                            }
                            cs.row_ok = ok;
                        }
                    }
                    win_repack_rows<Cfg::B_ROWS, RPW, WROW, CWIN>(sStg + slot * STG, sA + s * Cfg::A_BYTES,
                                                                  sB + s * Cfg::B_BYTES, pw, lane, p.win_delta_a,
                                                                  p.win_delta_b, cs);
                    fence_proxy_async_shared();  // generic-proxy writes -> tensor-core reads
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(full_bar(s));
                        if (p.proto) proto_add(p.proto, static_cast<int>(blockIdx.x), PROTO_BAR_FULL, s, it / STAGES, 1);
                        mbar_arrive(sw + 8u * (kWinStaging + slot));
                    }
                    ++it;
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                    if (++slot == kWinStaging) {
                        slot = 0;
                        sph ^= 1u;
                    }
                }
            }
        }
    } else if (LDG && !WIN && (warp == 0 || warp >= 6)) {
        // ------------------------------------- plain-load producer ---
        if constexpr (LDG && !WIN) {
            const int pw = warp == 0 ? 0 : warp - 5;  // producer warp 0..kLdgWarps-1 (warps 0, 6, 7, ...)
            constexpr int RPW = (128 + Cfg::B_ROWS) / kLdgWarps;
            constexpr uint32_t STG = static_cast<uint32_t>(ldg_staging_buffer_bytes<Cfg::B_ROWS>());
            static_assert(RPW % 32 == 0, "row quads of 8-apart rows cover whole groups of 32 rows");
            const uint32_t sStg = sBar + Cfg::BAR_BYTES;
            // Stage uses in the order the MMA issuer consumes them: (tile rows,
            // K block). `ahead` is the next use to copy, `cur` the one to unpack.
            struct Use {
                int m0, n0, kb;
            };
            int ui = cluster_id, kb_next = 0, kb_end = 0;
            int mt = 0, nt = 0;
            if (ui < num_units) {
                const Unit w = unit_of(ui, num_tiles, p);
                tile_coords(w.tile, p, mt, nt);
                kb_next = w.kb0;
                kb_end = w.kb1;
            }
            auto fetch = [&](Use& use) -> bool {
                if (ui >= num_units) return false;
                use = Use{mt * Cfg::BM, nt * BN, kb_next};
                if (++kb_next == kb_end) {
                    ui += num_clusters;
                    if (ui < num_units) {
                        const Unit w = unit_of(ui, num_tiles, p);
                        tile_coords(w.tile, p, mt, nt);
                        kb_next = w.kb0;
                        kb_end = w.kb1;
                    }
                }
                return true;
            };
            int s = 0, it = 0;
            uint32_t ph = 0, slot = 0;
            Use cur{0, 0, 0}, nxt{0, 0, 0};
            bool have_cur = fetch(cur);
            if (have_cur)
                ldg_issue_rows<Cfg::B_ROWS, RPW>(ConvRows(p, cur.m0, cur.n0, cur.kb), sStg, pw, lane);
            cp_async_commit();
            while (have_cur) {
                // copies of the next use go out before this one is unpacked
                const bool have_nxt = fetch(nxt);
                if (have_nxt)
                    ldg_issue_rows<Cfg::B_ROWS, RPW>(ConvRows(p, nxt.m0, nxt.n0, nxt.kb),
                                                           sStg + (slot ^ 1u) * STG, pw, lane);
                cp_async_commit();
                cp_async_wait<1>();  // this use's copies (every lane's, after the warp sync)
                __syncwarp();
                int free_ok = 1;
                if (lane == 0)
                    free_ok = wait_bounded(empty_bar(s), ph ^ 1u, p.wait, abort_flag, SITE_PRODUCER_EMPTY);
                if (!__shfl_sync(0xffffffffu, free_ok, 0)) break;
                ldg_repack_rows<Cfg::B_ROWS, RPW>(sStg + slot * STG, ConvRows(p, cur.m0, cur.n0, cur.kb).nvalid,
                                                  sA + s * Cfg::A_BYTES, sB + s * Cfg::B_BYTES, pw, lane);
                fence_proxy_async_shared();  // generic-proxy writes -> tensor-core reads
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(full_bar(s));
                    if (p.proto) proto_add(p.proto, static_cast<int>(blockIdx.x), PROTO_BAR_FULL, s, it / STAGES, 1);
                }
                ++it;
                if (++s == STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
                slot ^= 1u;
                cur = nxt;
                have_cur = have_nxt;
                // the staging buffer just unpacked is refilled next iteration;
                // every lane must be done reading it
                __syncwarp();
            }
            cp_async_wait<0>();  // no copy may land after the CTA's shared memory is released
            __syncwarp();
        }
    } else if (warp == 0) {
        // --------------------------------------------------- producer ---
        if (elect_one()) {
            int s = 0;
            uint32_t ph = 0;
            int issued = 0;
            bool ok = true;
            unsigned long long t_wait = 0;
            const uint64_t t_start = p.trace ? globaltimer_ns() : 0;
            // The k-loop is one thread's critical path (a stage every ~256
            // cycles at MMA N = 128), so it is kept lean: the cache-hint
            // choice is made once, by instantiating the loop for it; the
            // leader's full barriers are addressed from one mapa; the conv's
            // (tap, channel block) coordinates step instead of dividing.
            // PR: the instrumented loop (arrival accounting), instantiated
            // apart so that the plain loop carries none of it.
            auto run = [&](auto hint_a_t, auto hint_b_t, auto pr_t) {
                constexpr bool HA = decltype(hint_a_t)::value;
                constexpr bool HB = decltype(hint_b_t)::value;
                constexpr bool PR = decltype(pr_t)::value;
                const uint64_t pol_a = HA ? make_l2_policy(p.l2_a) : 0;
                const uint64_t pol_b = HB ? make_l2_policy(p.l2_b) : 0;
                const uint32_t fb0 = CL ? mapa_shared(full_bar(0), 0) : full_bar(0);
                bool arrive = !p.withhold_first_arrival;  // the self test withholds the very first arrival
                for (int u = cluster_id, plt = 0; ok && u < num_units; u += num_clusters, ++plt) {
                    const Unit w = unit_of(u, num_tiles, p);
                    if (p.events) event_at(p, plt, EV_PRODUCER_START, globaltimer_ns());
                    int mt, nt;
                    tile_coords(w.tile, p, mt, nt);
                    const int m_row = mt * (Cfg::BM * CG) + static_cast<int>(rank) * Cfg::BM;
                    // A narrow unit (2-SM only) of the tile's p.tail_parts column
                    // parts needs BN / (2 parts) rows of B per CTA, starting at
                    // its part; the narrow box loads just them.
                    const int pw = BN / p.tail_parts;  // columns of a narrow unit
                    const int n_row = w.part < 0 ? nt * BN + static_cast<int>(rank) * Cfg::B_ROWS
                                                 : nt * BN + w.part * pw + static_cast<int>(rank) * (pw / 2);
                    // narrow units (2-SM, N = 256 only) load B through the narrow box
                    const bool hu = CG == 2 && BN == 256 && w.part >= 0;
                    const CUtensorMap* const mB = hu ? &mapBh : &mapB;
                    const uint32_t tx = !hu ? Cfg::TX_BYTES
                                            : (p.tail_parts == 4 ? Cfg::TX_QUARTER_BYTES : Cfg::TX_HALF_BYTES);
                    // GEMM units of odd waves walk K backwards: the clusters
                    // of one wave share A rows with the wave before, whose
                    // last K blocks are the ones still in L2.
                    [[maybe_unused]] const int kb_flip = (plt & 1) ? w.kb0 + w.kb1 - 1 : -1;
                    [[maybe_unused]] int img = 0, base_h = 0, base_w = 0, rs = 0, cb = 0, r = 0, sx = 0;
                    if constexpr (CONV) {
                        const int pq = static_cast<int>(p.div_pq.d);
                        img = m_row / pq;
                        const int rem = m_row - img * pq;
                        const int pp = rem / p.conv_Q;
                        const int qq = rem - pp * p.conv_Q;
                        base_h = pp * p.conv_stride - p.conv_pad;
                        base_w = qq * p.conv_stride - p.conv_pad;
                        rs = w.kb0 / p.conv_cblocks;
                        cb = w.kb0 - rs * p.conv_cblocks;
                        r = rs / p.conv_S;
                        sx = rs - r * p.conv_S;
                    }
                    for (int kb = w.kb0; kb < w.kb1; ++kb) {
                        if (!timed_wait(p, empty_bar(s), ph ^ 1u, abort_flag, SITE_PRODUCER_EMPTY, t_wait)) {
                            ok = false;
                            break;
                        }
                        const uint32_t fb = fb0 + 8u * static_cast<uint32_t>(s);
                        if (leader && arrive) mbar_arrive_expect_tx(full_bar(s), tx);
                        if constexpr (PR) {
                            // phase issued / STAGES of stage s, on the leader's barrier
                            const int lead = static_cast<int>(blockIdx.x) - static_cast<int>(rank);
                            const int k = issued / STAGES;
                            if (leader && arrive) {
                                proto_add(p.proto, lead, PROTO_BAR_FULL, s, k, 1);
                                proto_add(p.proto, lead, PROTO_ROW_TX_EXPECT, s, k, tx);
                            }
                            proto_add(p.proto, lead, PROTO_ROW_TX_ISSUED, s, k,
                                      Cfg::A_BYTES + (hu ? Cfg::B_BYTES / p.tail_parts : Cfg::B_BYTES));
                        }
                        arrive = true;
                        const uint32_t dA = sA + s * Cfg::A_BYTES;
                        const uint32_t dB = sB + s * Cfg::B_BYTES;
                        if constexpr (CONV) {
                            const int c0 = cb * Cfg::BK;
                            const uint16_t ow = static_cast<uint16_t>(sx), oh = static_cast<uint16_t>(r);
                            if constexpr (CL) {
                                if constexpr (HA) tma_load_im2col_4d_pair(dA, &mapA, fb, c0, base_w, base_h, img, ow, oh, pol_a);
                                else tma_load_im2col_4d_pair(dA, &mapA, fb, c0, base_w, base_h, img, ow, oh);
                                if constexpr (HB) tma_load_3d_pair(dB, mB, fb, c0, rs, n_row, pol_b);
                                else tma_load_3d_pair(dB, mB, fb, c0, rs, n_row);
                            } else {
                                if constexpr (HA) tma_load_im2col_4d(dA, &mapA, fb, c0, base_w, base_h, img, ow, oh, pol_a);
                                else tma_load_im2col_4d(dA, &mapA, fb, c0, base_w, base_h, img, ow, oh);
                                if constexpr (HB) tma_load_3d(dB, mB, fb, c0, rs, n_row, pol_b);
                                else tma_load_3d(dB, mB, fb, c0, rs, n_row);
                            }
                            if (++cb == p.conv_cblocks) {
                                cb = 0;
                                ++rs;
                                if (++sx == p.conv_S) {
                                    sx = 0;
                                    ++r;
                                }
                            }
                        } else {
                            const int kx = (kb_flip < 0 ? kb : kb_flip - kb) * Cfg::BK;
                            if constexpr (CL) {
                                if constexpr (HA) tma_load_2d_pair(dA, &mapA, fb, kx, m_row, pol_a);
                                else tma_load_2d_pair(dA, &mapA, fb, kx, m_row);
                                if constexpr (HB) tma_load_2d_pair(dB, mB, fb, kx, n_row, pol_b);
                                else tma_load_2d_pair(dB, mB, fb, kx, n_row);
                            } else {
                                if constexpr (HA) tma_load_2d(dA, &mapA, fb, kx, m_row, pol_a);
                                else tma_load_2d(dA, &mapA, fb, kx, m_row);
                                if constexpr (HB) tma_load_2d(dB, mB, fb, kx, n_row, pol_b);
                                else tma_load_2d(dB, mB, fb, kx, n_row);
                            }
                        }
                        ++issued;
                        if (++s == STAGES) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                    if (p.events) {
                        event_at(p, plt, EV_PRODUCER_END, globaltimer_ns());
                        event_at(p, plt, EV_UNIT, static_cast<unsigned long long>(u));
                    }
                }
            };
            // A load carries a cache-hint policy only when its operand's
            // priority asks for one (l2_a / l2_b != 0; 3 = explicit normal).
            using T = std::true_type;
            using F = std::false_type;
            auto go = [&](auto pr) {
                if (p.l2_a != 0) {
                    if (p.l2_b != 0) run(T{}, T{}, pr);
                    else run(T{}, F{}, pr);
                } else {
                    if (p.l2_b != 0) run(F{}, T{}, pr);
                    else run(F{}, F{}, pr);
                }
            };
            if (p.proto) go(T{});
            else go(F{});
            if (p.trace) {
                trace_add(p, TRACE_PRODUCER_SPAN, globaltimer_ns() - t_start);
                trace_add(p, TRACE_PRODUCER_WAIT_EMPTY, t_wait);
            }
            if (!ok && (!CL || leader)) {
                // Gave up: let the loads already in flight land before the
                // CTA's shared memory can be released (bounded as well).
                WaitCtl drain = p.wait;
                int n = issued < STAGES ? issued : STAGES;
                int ss = s;
                uint32_t pp = ph;
                volatile int no_abort = 0;
                for (int i = 0; i < n; ++i) {
                    if (--ss < 0) {
                        ss = STAGES - 1;
                        pp ^= 1u;
                    }
                    wait_bounded(full_bar(ss), pp, drain, &no_abort, SITE_DRAIN);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer ---
        if (!CL || leader) {
            if (elect_one()) {
                constexpr uint32_t IDESC = umma_idesc_bf16_f32(Cfg::BM * CG, BN);
                constexpr uint32_t IDESC_HALF = umma_idesc_bf16_f32(Cfg::BM * CG, BN / 2);
                constexpr uint32_t IDESC_QUARTER = umma_idesc_bf16_f32(Cfg::BM * CG, BN / 4 >= 16 * CG ? BN / 4 : BN / 2);
                const uint32_t idesc_narrow = p.tail_parts == 4 ? IDESC_QUARTER : IDESC_HALF;
                int s = 0;
                uint32_t ph = 0;
                int lt = 0;
                bool ok = true;
                unsigned long long t_full = 0, t_acc = 0;
                const uint64_t t_start = p.trace ? globaltimer_ns() : 0;
                // Like the producer's, this loop is a single thread's critical
                // path. The descriptors of stage s and K step k differ from
                // those of stage 0 only in the start-address field (address /
                // 16, below 2^14 in the CTA's shared window, so adding to it
                // never carries): they are formed once and advanced by adds.
                const uint64_t dA0 = umma_desc_sw128_kmajor(sA);
                const uint64_t dB0 = umma_desc_sw128_kmajor(sB);
                // PR: the instrumented loop (arrival accounting and the
                // skipped-commit self test), instantiated apart.
                auto mma_run = [&](auto pr_t) {
                    constexpr bool PR = decltype(pr_t)::value;
                    int it = 0;  // stage uses so far (phase of stage s = it / STAGES)
                    // Arrival of a commit on empty / acc_full barrier `bar` + `idx`,
                    // phase k, in this CTA and (pair) its peer.
                    [[maybe_unused]] auto count_commit = [&](int bar, int idx, int k) {
                        proto_add(p.proto, static_cast<int>(blockIdx.x), bar, idx, k, 1);
                        if constexpr (CL) proto_add(p.proto, static_cast<int>(blockIdx.x) + 1, bar, idx, k, 1);
                    };
                    for (int u = cluster_id; ok && u < num_units; u += num_clusters, ++lt) {
                        const Unit w = unit_of(u, num_tiles, p);
                        const int b = lt & 1;
                        const uint32_t aph = static_cast<uint32_t>(lt >> 1) & 1u;
                        if (!timed_wait(p, acce_bar(b), aph ^ 1u, abort_flag, SITE_MMA_ACC_EMPTY, t_acc)) break;
                        if (p.events) event_at(p, lt, EV_MMA_START, globaltimer_ns());
                        tcgen05_fence_after();
                        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * BN);
                        const uint32_t idesc = w.part < 0 ? IDESC : idesc_narrow;
                        uint32_t accumulate = 0;  // the unit's first MMA overwrites the accumulator
                        for (int kb = w.kb0; kb < w.kb1; ++kb) {
                            if (!timed_wait(p, full_bar(s), ph, abort_flag, SITE_MMA_FULL, t_full)) {
                                ok = false;
                                break;
                            }
                            tcgen05_fence_after();
                            const uint64_t da = dA0 + static_cast<uint64_t>(s * (Cfg::A_BYTES >> 4));
                            const uint64_t db = dB0 + static_cast<uint64_t>(s * (Cfg::B_BYTES >> 4));
#pragma unroll
                            for (int k = 0; k < Cfg::BK / Cfg::UMMA_K; ++k) {
                                // +32 bytes per K step of 16 inside the swizzle atom
                                umma_bf16<CG>(d_tmem, da + 2 * k, db + 2 * k, idesc, accumulate);
                                accumulate = 1;
                            }
                            bool commit = true;
                            if constexpr (PR) {
                                commit = !(p.skip_commit == 1 && it == 0);
                                if (commit && p.proto) count_commit(PROTO_BAR_EMPTY, s, it / STAGES);
                            }
                            if (commit) {
                                if constexpr (CL) umma_commit_pair(empty_bar(s), 0x3);
                                else umma_commit(empty_bar(s));
                            }
                            ++it;
                            if (++s == STAGES) {
                                s = 0;
                                ph ^= 1u;
                            }
                        }
                        if (!ok) break;
                        if (p.events) event_at(p, lt, EV_MMA_END, globaltimer_ns());
                        bool commit = true;
                        if constexpr (PR) {
                            commit = !(p.skip_commit == 2 && lt == 0);
                            if (commit && p.proto) count_commit(PROTO_BAR_ACC_FULL, b, lt >> 1);
                        }
                        if (commit) {
                            if constexpr (CL) umma_commit_pair(accf_bar(b), 0x3);
                            else umma_commit(accf_bar(b));
                        }
                    }
                };
                if (p.proto || p.skip_commit) mma_run(std::true_type{});
                else mma_run(std::false_type{});
                if (p.trace) {
                    trace_add(p, TRACE_MMA_SPAN, globaltimer_ns() - t_start);
                    trace_add(p, TRACE_MMA_WAIT_FULL, t_full);
                    trace_add(p, TRACE_MMA_WAIT_ACC_EMPTY, t_acc);
                    trace_add(p, TRACE_UNITS, static_cast<unsigned long long>(lt));
                }
                // Every MMA this thread issued completes before teardown.
                if constexpr (CL) umma_commit_pair(drain_bar, 0x1);
                else umma_commit(drain_bar);
                volatile int no_abort = 0;
                wait_bounded(drain_bar, 0, p.wait, &no_abort, SITE_DRAIN);
            }
            __syncwarp();
        }
    } else {
        // --------------------------------------------------- epilogue ---
        const int ew = warp - 2;           // staging slot of this warp
        const int quarter = warp & 3;      // TMEM lanes this warp may read
        const uint32_t stage0 = sEpi + static_cast<uint32_t>(ew) * 2u * Cfg::EPI_BUF;
        constexpr int CHUNKS = BN / Cfg::EPI_COLS;
        int buf = 0;
        int lt = 0;
        unsigned long long t_accf = 0;
        const uint64_t t_start = p.trace ? globaltimer_ns() : 0;
        for (int u = cluster_id; u < num_units; u += num_clusters, ++lt) {
            const Unit w = unit_of(u, num_tiles, p);
            const int b = lt & 1;
            const uint32_t aph = static_cast<uint32_t>(lt >> 1) & 1u;
            // where the unit's outputs go: worked out before the wait, off
            // the path from the last MMA to the stores
            int mt, nt;
            tile_coords(w.tile, p, mt, nt);
            const int m_row = mt * (Cfg::BM * CG) + static_cast<int>(rank) * Cfg::BM + quarter * 32;
            const int n0 = nt * BN + (w.part < 0 ? 0 : w.part * (BN / p.tail_parts));
            const int max_chunks = w.part < 0 ? CHUNKS : CHUNKS / p.tail_parts;
            int nchunks = 0;
            if (m_row < p.M && n0 < p.N) {
                nchunks = (p.N - n0 + Cfg::EPI_COLS - 1) / Cfg::EPI_COLS;
                nchunks = nchunks < max_chunks ? nchunks : max_chunks;
            }
            if (!timed_wait(p, accf_bar(b), aph, abort_flag, SITE_EPI_ACC_FULL, t_accf)) break;
            if (p.events && warp == 2 && lane == 0) event_at(p, lt, EV_EPI_READY, globaltimer_ns());
            tcgen05_fence_after();
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   static_cast<uint32_t>(b * BN);
            const uint32_t acce_target = CL ? mapa_shared(acce_bar(b), 0) : acce_bar(b);
            if (nchunks == 0) {
                tcgen05_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (CL) mbar_arrive_cluster(acce_target);
                    else mbar_arrive(acce_target);
                    if (p.proto)
                        proto_add(p.proto, static_cast<int>(blockIdx.x) - static_cast<int>(rank), PROTO_BAR_ACC_EMPTY,
                                  b, lt >> 1, 1);
                }
                continue;
            }
            for (int c = 0; c < nchunks; ++c) {
                uint32_t packed[32];
                if constexpr (OUT_F32) {
                    tmem_ld_32x32b_x32(t_row + c * 32, packed);
                    tmem_wait_ld();
                    tmem_regs_ready(packed);
                } else {
                    uint32_t v0[32], v1[32];
                    tmem_ld_32x32b_x32(t_row + c * 64, v0);
                    tmem_ld_32x32b_x32(t_row + c * 64 + 32, v1);
                    tmem_wait_ld();
                    tmem_regs_ready(v0);
                    tmem_regs_ready(v1);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        packed[i] = pack_bf16x2(v0[2 * i], v0[2 * i + 1]);
                        packed[16 + i] = pack_bf16x2(v1[2 * i], v1[2 * i + 1]);
                    }
                }
                if (c == nchunks - 1) {
                    // Accumulator fully read: hand it back to the MMA issuer.
                    tcgen05_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        // stamped before the arrival, so the MMA issuer cannot
                        // see the accumulator free before this time
                        if (p.events && warp == 2) event_at(p, lt, EV_EPI_RELEASED, globaltimer_ns());
                        if constexpr (CL) mbar_arrive_cluster(acce_target);
                        else mbar_arrive(acce_target);
                        if (p.proto)
                            proto_add(p.proto, static_cast<int>(blockIdx.x) - static_cast<int>(rank),
                                      PROTO_BAR_ACC_EMPTY, b, lt >> 1, 1);
                    }
                }
                const int cs = n0 + c * Cfg::EPI_COLS;
                if (cs < p.n_tma) {
                    // The staging buffer about to be written was last used two
                    // chunks ago; its TMA store must have finished reading it.
                    if (lane == 0) bulk_wait_group_read<1>();
                    __syncwarp();
                    const uint32_t sbuf = stage0 + static_cast<uint32_t>(buf) * Cfg::EPI_BUF;
                    const uint32_t row_addr = sbuf + lane * 128u;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t slot = static_cast<uint32_t>(j) ^ (lane & 7u);
                        st_shared_v4(row_addr + slot * 16u, packed[4 * j], packed[4 * j + 1], packed[4 * j + 2],
                                     packed[4 * j + 3]);
                    }
                    fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (SPLITK) tma_store_3d(&mapC, sbuf, cs, m_row, w.split);
                        else tma_store_2d(&mapC, sbuf, cs, m_row);
                        bulk_commit_group();
                    }
                    buf ^= 1;
                }
                if (cs + Cfg::EPI_COLS > p.n_tma) {
                    // Columns past the last full 16-byte granule of the row.
                    const int lo = (p.n_tma > cs ? p.n_tma : cs) - cs;
                    const int hi = (p.N - cs < Cfg::EPI_COLS ? p.N - cs : Cfg::EPI_COLS);
                    const int row = m_row + static_cast<int>(lane);
                    if (row < p.M && lo < hi) {
                        uint8_t* rowp = static_cast<uint8_t*>(p.C) + static_cast<int64_t>(row) * p.ldc_bytes;
#pragma unroll
                        for (int j = 0; j < Cfg::EPI_COLS; ++j) {
                            if (j >= lo && j < hi) {
                                if constexpr (OUT_F32)
                                    reinterpret_cast<uint32_t*>(rowp)[cs + j] = packed[j];
                                else
                                    reinterpret_cast<uint16_t*>(rowp)[cs + j] =
                                        static_cast<uint16_t>(packed[j >> 1] >> (16 * (j & 1)));
                            }
                        }
                    }
                }
            }
            if (p.events && warp == 2 && lane == 0) event_at(p, lt, EV_EPI_STORED, globaltimer_ns());
        }
        if (p.trace && warp == 2 && lane == 0) {
            trace_add(p, TRACE_EPI_SPAN, globaltimer_ns() - t_start);
            trace_add(p, TRACE_EPI_WAIT_ACC_FULL, t_accf);
        }
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }

    // --------------------------------------------------------- teardown ---
    tcgen05_fence_before();
    if constexpr (CL) cluster_sync(); else __syncthreads();
    if (warp == 1) {
        tcgen05_fence_after();
        tmem_dealloc<CG>(tmem_base, Cfg::TMEM_COLS);
    }
}

template <int CG, int BN, int STAGES, bool OUT_F32, bool CONV, int LDG = kLdgNone, bool SPLITK = false>
cudaError_t launch_mainloop(const GemmLaunch& L)
{
    using Cfg = MainloopCfg<CG, BN, STAGES, OUT_F32>;
    constexpr int SMEM = Cfg::SMEM_BYTES + (LDG ? ldg_extra_bytes<Cfg::B_ROWS, CONV, LDG>() : 0);
    auto kern = mainloop_kernel<CG, BN, STAGES, OUT_F32, CONV, LDG, SPLITK>;
    static std::atomic<uint64_t> smem_set{0};
    cudaError_t e = smem_limit_once(kern, SMEM, smem_set);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(L.grid), 1, 1);
    cfg.blockDim = dim3(mainloop_threads<LDG, CONV>(), 1, 1);
    cfg.dynamicSmemBytes = SMEM;
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    // the 1-SM atom launches as plain CTAs, without a cluster shape
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = CG;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = CG > 1 ? 2 : 1;
    if constexpr (win_form<CONV, LDG>())
        return cudaLaunchKernelEx(&cfg, kern, L.mapA, L.mapB, L.mapC, L.mapBh, L.params, L.win);
    else return cudaLaunchKernelEx(&cfg, kern, L.mapA, L.mapB, L.mapC, L.mapBh, L.params, NoWinMaps{0});
}

template <int CG, int BN, int STAGES, bool OUT_F32, bool CONV, int LDG = kLdgNone, bool SPLITK = false>
constexpr KernelEntry mainloop_entry()
{
    return KernelEntry{KernelKey{CG, BN, STAGES, OUT_F32 ? 1 : 0, CONV ? 1 : 0, LDG, SPLITK ? 1 : 0},
                       &launch_mainloop<CG, BN, STAGES, OUT_F32, CONV, LDG, SPLITK>,
                       MainloopCfg<CG, BN, STAGES, OUT_F32>::SMEM_BYTES +
                           (LDG ? ldg_extra_bytes<MainloopCfg<CG, BN, STAGES, OUT_F32>::B_ROWS, CONV, LDG>() : 0)};
}

}  // namespace tp
