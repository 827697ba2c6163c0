// Definitions shared by the kernels and the host launchers: the device status
// record, bounded barrier waits and the kernel parameter blocks.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace tp {

// Status codes (same values as tp_status in include/tp.h).
enum : int {
    ST_OK = 0,
    ST_INVALID_ARG = 1,
    ST_UNSUPPORTED = 2,
    ST_CUDA = 3,
    ST_DRIVER_ENCODE = 4,
    ST_TIMEOUT = 5,
    ST_SMEM_BUDGET = 6,
};

// Where a bounded wait gave up (recorded with ST_TIMEOUT).
enum : int {
    SITE_PRODUCER_EMPTY = 1,
    SITE_MMA_FULL = 2,
    SITE_MMA_ACC_EMPTY = 3,
    SITE_EPI_ACC_FULL = 4,
    SITE_COPY_FULL = 5,
    SITE_DRAIN = 6,
    SITE_SELFTEST = 7,
};

// One per device, a static __device__ object of the library. The first
// failure wins; tp_device_status reads and clears it.
struct DevStatus {
    int code;
    int site;
    int block;
    int thread;
};

struct WaitCtl {
    DevStatus* status;
    uint64_t limit_ns;  // give up after this long without progress
};

__device__ __forceinline__ void report_failure(DevStatus* st, int code, int site)
{
    if (atomicCAS(&st->code, 0, code) == 0) {
        st->site = site;
        st->block = static_cast<int>(blockIdx.x);
        st->thread = static_cast<int>(threadIdx.x);
    }
}

// Wait for the phase of parity `parity` of `bar` to complete. Gives up after
// w.limit_ns (or ~2^30 polls), records ST_TIMEOUT at `site`, raises the
// CTA's abort flag and returns false; also returns false as soon as another
// role of the CTA raised the flag. Never traps.
//
// The wait acquires at CTA scope, also in a 2-SM pair whose barriers receive
// arrivals from the peer CTA: what a pipeline barrier orders is data written
// by TMA (complete_tx lands it before the phase can complete) or tensor
// memory (ordered by the tcgen05 fences around the barrier), so no
// cluster-scope memory fence is needed, and on GB300 its cost showed: with
// cluster-scope acquire / release on these barriers a 4096 x 4096 x 512 GEMM
// took 17.8 us back to back, with CTA scope 14.4 us.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const WaitCtl& w,
                                             volatile int* abort_flag, int site)
{
    auto poll = [&]() { return mbar_try_wait(bar, parity); };
    if (poll()) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (poll()) return true;
        if ((i & 63u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > w.limit_ns || i > (1u << 30)) {
                report_failure(w.status, ST_TIMEOUT, site);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

// Division by a divisor fixed for the launch, for 0 <= n < 2^31: with
// l = ceil(log2 d) and m = ceil(2^(31+l) / d) (which fits 32 bits),
// n / d = (n * m) >> (31 + l) (Granlund and Montgomery, "Division by
// invariant integers using multiplication", 1994, round-up method with
// N = 31 bits). One wide multiply and a shift replace the division
// sequence, which the kernels' single-thread roles would otherwise wait on
// for every work unit.
struct FastDiv {
    uint32_t d, m;
    uint32_t sh;
};

inline FastDiv make_fastdiv(uint32_t d)
{
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;
    const uint64_t top = 1ull << (31 + l);
    return FastDiv{d, static_cast<uint32_t>((top + d - 1) / d), 31 + l};
}

__device__ __forceinline__ int fdiv(int n, const FastDiv& f)
{
    return static_cast<int>((static_cast<uint64_t>(static_cast<uint32_t>(n)) * f.m) >> f.sh);
}

// GEMM view of a launch. For the convolution M = N*P*Q output pixels,
// N = output channels, K = R*S*C (walked as (r, s) outer, 64-channel blocks
// inner).
struct GemmParams {
    int M, N, K;
    // TMA stores write whole 16-byte granules of a row, so the C map ends at
    // the last full granule (n_tma columns); columns n_tma..N-1 are written
    // with plain stores through C / ldc_bytes.
    int n_tma;
    void* C;
    int64_t ldc_bytes;
    int m_tiles;   // tiles of 128*CG rows
    int n_tiles;   // tiles of BN columns
    int k_blocks;  // 64-deep K blocks
    // split-K: work unit u is tile u % tiles over K blocks
    // [split * kb_per_split, min(k_blocks, (split + 1) * kb_per_split)),
    // split = u / tiles; its fp32 partial goes to slice `split` of the
    // workspace C map. splits == 1 is the plain GEMM.
    int splits, kb_per_split;
    // Narrow tail (2-SM atom, splits == 1): units [0, n_full) are whole
    // tiles; the last tail_units units are narrow tiles (N = BN / tail_parts,
    // tail_parts of 2 or 4 per remaining tile), so the last, partial wave
    // takes about a half or a quarter as long.
    int n_full, tail_units, tail_parts;
    int group_m;   // tile raster: group_m M-tiles share a sweep over N
    // divisors of the unit and tile arithmetic (set_divisors): tiles
    // (m_tiles * n_tiles), a raster group's tiles (group_m * n_tiles), its
    // M-tiles (group_m, and the last group's), and the conv's P * Q, Q, 64-
    // channel blocks and S
    FastDiv div_tiles, div_group, div_gm, div_gm_last, div_pq, div_q, div_cblocks, div_s;
    int l2_a, l2_b;  // L2 eviction priority of A / B loads (0 normal, 1 first, 2 last)
    // convolution only
    int conv_P, conv_Q, conv_stride, conv_pad, conv_S, conv_cblocks;
    // plain-load producer only (operands TMA cannot describe): A / B (or x /
    // w) with their pitches in elements, and the conv input extents
    const uint16_t* A;
    const uint16_t* B;
    int64_t lda, ldb;
    int conv_H, conv_W, conv_C, conv_R;
    // plain-load GEMM (row-class windows, below): element offset (0..7) of
    // row class q's rows inside their 16-byte-aligned windows, 3 bits per
    // class, for A and B
    uint32_t win_delta_a, win_delta_b;
    // Optional role timeline: kTraceSlots counters per CTA (nanoseconds,
    // accumulated with atomicAdd), or nullptr.
    unsigned long long* trace;
    // Optional per-unit event timeline: kEventSlots per CTA, or nullptr.
    unsigned long long* events;
    // Self-test only (tp_selftest_mainloop_withheld_arrival): 1 makes the
    // producer withhold the expect_tx arrival of its first stage while still
    // issuing its loads, so the consumer's bounded wait must give up.
    int withhold_first_arrival;
    // Self-test only (tp_selftest_mainloop_skipped_commit): 1 makes the MMA
    // issuer skip its first commit to empty[s], 2 its first commit to
    // acc_full[b], so the producer's or the epilogue's bounded wait must
    // give up.
    int skip_commit;
    // Optional arrival accounting: kProtoSlots counters per CTA (below), or
    // nullptr.
    unsigned int* proto;
    WaitCtl wait;
};

// Arrival accounting (GemmParams::proto), per CTA, uint32 counters indexed
// by barrier and phase: phase k of a barrier is the k-th time its stage (or
// accumulator) is used. Arrivals are counted where they are issued, on the
// CTA that owns the barrier (a 2-SM pair's full / acc_empty barriers are its
// leader's; its commits arrive on both CTAs' empty / acc_full barriers).
// Phases past the last counted one add to it.
enum : int {
    PROTO_MAX_STAGES = 9,
    PROTO_PHASES = 64,
    PROTO_BAR_FULL = 0,                                  // + stage
    PROTO_BAR_EMPTY = PROTO_MAX_STAGES,                  // + stage
    PROTO_BAR_ACC_FULL = 2 * PROTO_MAX_STAGES,           // + accumulator
    PROTO_BAR_ACC_EMPTY = 2 * PROTO_MAX_STAGES + 2,      // + accumulator
    PROTO_BARS = 2 * PROTO_MAX_STAGES + 4,
    // transaction bytes of full[s] phase k: posted by expect_tx ...
    PROTO_TX_EXPECT = PROTO_BARS * PROTO_PHASES,
    // ... and carried by the TMA loads issued into it (both CTAs of a pair)
    PROTO_TX_ISSUED = PROTO_TX_EXPECT + PROTO_MAX_STAGES * PROTO_PHASES,
    kProtoSlots = PROTO_TX_ISSUED + PROTO_MAX_STAGES * PROTO_PHASES,
};

// Rows of PROTO_PHASES counters: barrier rows, then the two byte tables.
enum : int {
    PROTO_ROW_TX_EXPECT = PROTO_TX_EXPECT / PROTO_PHASES,
    PROTO_ROW_TX_ISSUED = PROTO_TX_ISSUED / PROTO_PHASES,
};

// Adds v to phase `phase` of row `row` + `index` of CTA `cta`'s counters
// (row: a PROTO_BAR_* barrier row or a PROTO_ROW_TX_* table; index: the
// stage or accumulator).
__device__ __forceinline__ void proto_add(unsigned int* proto, int cta, int row, int index, int phase,
                                          unsigned int v)
{
    const int k = phase < PROTO_PHASES ? phase : PROTO_PHASES - 1;
    atomicAdd(proto + static_cast<size_t>(cta) * kProtoSlots + (row + index) * PROTO_PHASES + k, v);
}

// Role-timeline counters, per CTA (GemmParams::trace).
enum : int {
    TRACE_PRODUCER_SPAN = 0,      // producer: first wait -> last load issued
    TRACE_PRODUCER_WAIT_EMPTY,    // producer: waiting for a free stage
    TRACE_MMA_SPAN,               // MMA issuer: first wait -> last commit
    TRACE_MMA_WAIT_FULL,          // MMA issuer: waiting for a loaded stage
    TRACE_MMA_WAIT_ACC_EMPTY,     // MMA issuer: waiting for a drained accumulator
    TRACE_EPI_SPAN,               // epilogue (one warp): first wait -> last store issued
    TRACE_EPI_WAIT_ACC_FULL,      // epilogue: waiting for a finished accumulator
    TRACE_UNITS,                  // work units this CTA's MMA issuer processed
    kTraceSlots
};

// Per-unit event timeline (GemmParams::events): for each CTA's first
// kEventUnits work units, kEventsPerUnit slots of globaltimer nanoseconds,
// taken at the unit boundaries of each role, plus the unit's index.
enum : int {
    EV_PRODUCER_START = 0,  // producer: about to wait for the unit's first free stage
    EV_PRODUCER_END,        // producer: the unit's last loads issued
    EV_MMA_START,           // MMA issuer: the unit's accumulator is free
    EV_MMA_END,             // MMA issuer: the unit's last MMAs issued
    EV_EPI_READY,           // epilogue (warp 2): the accumulator is complete
    EV_EPI_RELEASED,        // epilogue (warp 2): accumulator read, handed back
    EV_EPI_STORED,          // epilogue (warp 2): the unit's last store issued
    EV_UNIT,                // the work unit's index (not a time)
    kEventsPerUnit
};
constexpr int kEventUnits = 8;
constexpr int kEventSlots = kEventsPerUnit * kEventUnits;

struct CopyParams {
    int tiles_x, tiles_y;      // tiles along columns / rows
    int box_cols, box_rows;
    uint32_t tile_bytes;
    WaitCtl wait;
};

// Raises a kernel's dynamic shared-memory limit to `bytes` once per device
// (the attribute is per function and context; setting it on every launch
// costs host time a small problem cannot hide). `done` is one bit per device,
// owned by the caller's kernel instantiation.
template <typename Kern>
inline cudaError_t smem_limit_once(Kern kern, int bytes, std::atomic<uint64_t>& done)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return e;
}

// Key of one compiled GEMM/conv mainloop.
struct KernelKey {
    int cta_group;  // 1 or 2
    int bn;         // MMA N (pair tile N for cta_group 2)
    int stages;     // PIPE_DEPTH
    int out_f32;
    int conv;
    int ldg;        // 1: plain-load producer instead of TMA
    int splitk;     // 1: fp32 partials per K slice into a workspace
};

// Row-class windows of a GEMM operand whose rows TMA cannot address (a row
// pitch that is not a multiple of 16 bytes, or a misaligned base). Rows r
// and r + 8 always lie a multiple of 16 bytes apart, so the rows of one
// class q = r mod 8 form a tensor TMA can describe: its base is row q's
// address rounded down to 16 bytes, its row stride 8 pitches, its width K
// plus the class's offset (win_delta_*). A box 72 elements wide starting at
// element 64 kb holds K block kb of every row of the class, shifted right by
// that offset; the producer shifts it back in shared memory.
struct WinMaps {
    CUtensorMap a[8];
    CUtensorMap b[8];
};

struct GemmLaunch {
    CUtensorMap mapA, mapB, mapC;
    CUtensorMap mapBh;  // B with narrow boxes (half or quarter height): the 2-SM, N = 256 narrow tail
    WinMaps win;        // plain-load GEMM only
    GemmParams params;
    int grid;
    cudaStream_t stream;
};

using GemmLauncher = cudaError_t (*)(const GemmLaunch&);

struct KernelEntry {
    KernelKey key;
    GemmLauncher launch;
    int smem_bytes;
};

}  // namespace tp
