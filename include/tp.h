/*
 * tp.h -- C ABI of libtp: a warp-specialized, multi-stage, TMA-fed tcgen05
 * BF16 mainloop for sm_103a (GEMM and its implicit-GEMM convolution form) and
 * a TMA-only 2D copy.
 *
 * Conventions for every entry point:
 *  - Pointers are caller-owned DEVICE memory (any allocator). The library
 *    allocates no device memory; its state is a static device status
 *    record per GPU, the static split-K array behind
 *    tp_gemm_bf16_splitk_noalloc, and a cached driver entry point.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream). Calls are asynchronous on it; they return after the launch.
 *  - The return value reports what the host can see: invalid arguments, a
 *    descriptor the driver rejects, a launch error. Device-side failures (a
 *    bounded barrier wait that gave up) surface through tp_device_status.
 *  - Entry points may be called from several host threads at once: the
 *    per-device state is set up once under a lock, and the last-plan and
 *    last-CUDA-error records are per thread. The device status record is
 *    per GPU, so a tp_device_status call sees (and clears) a failure of any
 *    thread's launch on that GPU. tp_gemm_bf16_splitk_noalloc shares one
 *    workspace per GPU (see there).
 *  - bf16 is IEEE-style bfloat16; results are rounded to nearest even.
 *  - Empty problems (a zero M, N, rows or cols) are a no-op returning TP_OK.
 *    Negative sizes, a leading dimension below the row width, or a NULL
 *    pointer with a non-empty problem return TP_ERR_INVALID_ARG.
 *  - A base address or leading dimension that TMA cannot describe (not
 *    16-byte aligned) is not an error: the copy takes the vectorized thread
 *    copy, the GEMM and convolution a plain-load producer that feeds the same
 *    tcgen05 mainloop ("B200 Tma Pipeline Designer", step 1 and "Do not use
 *    when"). Elements must still be naturally aligned (2 bytes for bf16, 4
 *    for a float C), else TP_ERR_INVALID_ARG.
 */
#ifndef TP_H
#define TP_H

#include <stdint.h>

#if defined(__GNUC__)
#define TP_API __attribute__((visibility("default")))
#else
#define TP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TP_OK = 0,
    TP_ERR_INVALID_ARG = 1,
    TP_ERR_UNSUPPORTED = 2,
    TP_ERR_CUDA = 3,
    TP_ERR_DRIVER_ENCODE = 4,
    TP_ERR_TIMEOUT = 5,
    TP_ERR_SMEM_BUDGET = 6,
    TP_ERR_WORKSPACE_LIMIT = 7
} tp_status;

/* Which code path a call took (tp_plan.path). */
enum {
    TP_PATH_NONE = 0,          /* empty problem, nothing launched */
    TP_PATH_MAINLOOP = 1,      /* TMA + tcgen05 mainloop */
    TP_PATH_ZERO_FILL = 2,     /* K == 0: C is the empty sum */
    TP_PATH_TMA_COPY = 3,      /* TMA load -> smem -> TMA store ring */
    TP_PATH_VEC_COPY = 4,      /* vectorized ld/st fallback copy */
    TP_PATH_FALLBACK_MAINLOOP = 5, /* plain-load producer + tcgen05 mainloop */
    TP_PATH_TMA_TRANSPOSE = 6,     /* TMA load -> ldmatrix/stmatrix.trans -> TMA store */
    TP_PATH_VEC_TRANSPOSE = 7,     /* shared-memory tile transpose fallback */
    TP_PATH_TMA_READ = 8           /* TMA load ring only (tp_tma_read_2d) */
};

/*
 * C = A . B, bf16 inputs, fp32 accumulation in tensor memory, bf16 output.
 * Defined by the BF16 GEMM the pipelined mainloop serves ("two-free-pipeline-
 * stages" note, the 256x128x64 tile) and by the load/compute/store timeline
 * of "B200 Tma Pipeline Designer", steps 4-7.
 *   A: M x K row-major, element (i,k) at A[i*lda + k], lda >= K.
 *   B: K x N column-major, element (k,j) at B[j*ldb + k], ldb >= K.
 *   C: M x N row-major, element (i,j) at C[i*ldc + j], ldc >= N; overwritten
 *      (no alpha/beta). K == 0 writes zeros.
 * The TMA producer needs A, B, C 16-byte aligned and lda*2, ldb*2, ldc*2
 * multiples of 16; other layouts take the plain-load producer (1-SM atom,
 * N = 128; atom / tile_n choices other than those return TP_ERR_UNSUPPORTED).
 * It loads each row class (rows r mod 8, which sit a multiple of 16 bytes
 * apart) through its own TMA window and shifts the rows into place in
 * shared memory: about a quarter of the TMA producer's rate on a large
 * GEMM. C is still written with TMA stores when it is aligned.
 * Repeating a call gives the same bits. The fp32 summation order of a tile
 * depends on the variant and on the wave the tile runs in (a persistent
 * CTA's odd-numbered tiles take their K blocks last to first), so calls
 * whose options or grid differ may differ in rounding, within the same
 * accumulator error bound.
 */
TP_API int tp_gemm_bf16(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int64_t lda,
                 int64_t ldb, int64_t ldc, void* stream);

/* Same as tp_gemm_bf16 with the fp32 accumulator written out (C is float,
 * ldc*4 a multiple of 16). */
TP_API int tp_gemm_bf16_f32(const void* A, const void* B, float* C, int64_t M, int64_t N, int64_t K, int64_t lda,
                     int64_t ldb, int64_t ldc, void* stream);

/*
 * Mainloop choices, for sweeps and tests. Zero fields mean "choose".
 *   atom:       1 = 1-SM atom (a CTA owns a 128 x tile_n tile and holds all of
 *               its B tile), 2 = 2-SM atom (a CTA pair owns 256 x tile_n; each
 *               CTA holds half of B, which frees shared memory for more
 *               stages: "two-free-pipeline-stages", stage budget table).
 *   pipe_depth: PIPE_DEPTH, stages in the ring (2..9).
 *   tile_n:     MMA N: 64 (1-SM atom only; 128 x 64 tiles with up to 8
 *               stages, for problems whose wider tiles would leave most SMs
 *               idle), 128 or 256. "Choose" estimates each compiled
 *               variant's time from its waves of tiles, K blocks and measured
 *               throughput; the split-K entry points choose among N >= 128
 *               only.
 *   group_m:    tile raster: group_m M-tiles share one sweep over N
 *               (0 = 3072 rows of A per group: 24 tiles of the 1-SM atom,
 *               12 pair tiles of the 2-SM atom).
 *   max_ctas:   cap on the persistent grid (0 = one CTA per SM). A cap at
 *               or above the work-unit count (CTAs = units x atom; units =
 *               tiles, plus the narrow tail's extra parts) launches one
 *               work unit per cluster, i.e. a non-persistent grid that the
 *               hardware schedules in waves. The narrow tail is sized by the
 *               clusters that run at once: the cap or SMs / atom, whichever
 *               is smaller.
 *   l2_hint:    L2 eviction priorities of the operand loads: 0 choose,
 *               1 none (no cache-hint policy), 2 A evict-last / B
 *               evict-first, 3 A evict-last, 4 B evict-first, 5 A
 *               evict-first / B evict-last, 6 B evict-last, 7 an explicit
 *               evict_normal policy on both (not the same as 1: on GB300
 *               the unhinted loads measured faster for every variant).
 *               "Choose" (GEMM only; the convolution keeps 1) picks 2 when
 *               at most two tile rows read B and A is small (<= 16 MB,
 *               under a quarter of B): B then streams through L2 once while
 *               A, read by every tile, stays. It picks 5 in the mirrored
 *               case, else 1.
 *   no_tail:    1 keeps whole tiles in the last wave (the 2-SM, N = 256
 *               variant otherwise runs a partial last wave of r tiles as
 *               narrow tiles: 4r quarter-width ones when they fit one wave,
 *               else 2r half-width ones when those do).
 *   trace:      NULL, or a caller-owned, zeroed device buffer of
 *               TP_TRACE_SLOTS x (CTAs of the launch, tp_plan.grid) uint64
 *               that the mainloop fills with its role timeline (below):
 *               nanoseconds each role spent waiting on each barrier and its
 *               active span, per CTA (the pair's leader holds the MMA
 *               issuer's counters). Tracing adds a timer read per wait.
 *   events:     NULL, or a caller-owned, zeroed device buffer of
 *               TP_EVENT_SLOTS x (CTAs of the launch) uint64: the per-unit
 *               event timeline below. Both buffers may be given at once.
 *   protocol:   NULL, or a caller-owned, zeroed device buffer of
 *               TP_PROTO_SLOTS x (CTAs of the launch) uint32: the arrival
 *               accounting below (GEMM without split-K, and conv).
 * A (atom, depth, tile_n) whose stages do not fit the 232,448-byte shared
 * memory of a CTA returns TP_ERR_SMEM_BUDGET, the analogue of the note's
 * "StageCount<9> fails the capacity assert"; a combination that fits but is
 * not compiled returns TP_ERR_UNSUPPORTED.
 */
typedef struct {
    int atom;
    int pipe_depth;
    int tile_n;
    int group_m;
    int max_ctas;
    int l2_hint;
    int no_tail;
    uint64_t* trace;
    uint64_t* events;
    uint32_t* protocol;
} tp_gemm_opts;

/* Arrival accounting per CTA (tp_gemm_opts.protocol), TP_PROTO_SLOTS uint32
 * counters, for checking the stage ring's protocol on the device ("B200 Tma
 * Pipeline Designer", step 8: each ready / free barrier has one producer and
 * one consumer). Phase k of a barrier is the k-th use of its stage or
 * accumulator; counters of phases past TP_PROTO_PHASES - 1 add to the last.
 *   [bar * TP_PROTO_PHASES + k]  arrivals issued on barrier `bar` in phase k:
 *     bar = s (full[s]), TP_PROTO_MAX_STAGES + s (empty[s]),
 *     2 * TP_PROTO_MAX_STAGES + b (acc_full[b]),
 *     2 * TP_PROTO_MAX_STAGES + 2 + b (acc_empty[b]).
 *   [TP_PROTO_TX_EXPECT + s * TP_PROTO_PHASES + k]  bytes full[s] was told to
 *     expect (arrive.expect_tx) in phase k;
 *   [TP_PROTO_TX_ISSUED + s * TP_PROTO_PHASES + k]  bytes of the TMA loads
 *     issued into it (both CTAs of a pair).
 * Counts sit on the CTA that owns the barrier: a 2-SM pair's full and
 * acc_empty barriers are its leader's (even CTA); its MMA commits arrive on
 * both CTAs' empty and acc_full barriers. The plain-load producer arrives on
 * full[s] without transaction bytes. A counted launch runs an instrumented
 * copy of the producer and MMA loops (one atomic per arrival). */
#define TP_PROTO_MAX_STAGES 9
#define TP_PROTO_PHASES 64
#define TP_PROTO_BARS (2 * TP_PROTO_MAX_STAGES + 4)
#define TP_PROTO_TX_EXPECT (TP_PROTO_BARS * TP_PROTO_PHASES)
#define TP_PROTO_TX_ISSUED (TP_PROTO_TX_EXPECT + TP_PROTO_MAX_STAGES * TP_PROTO_PHASES)
#define TP_PROTO_SLOTS (TP_PROTO_TX_ISSUED + TP_PROTO_MAX_STAGES * TP_PROTO_PHASES)

/* Role-timeline counters per CTA (tp_gemm_opts.trace), in this order:
 * producer span, producer waiting for a free stage, MMA issuer span, MMA
 * waiting for a loaded stage, MMA waiting for a drained accumulator, epilogue
 * span (one warp), epilogue waiting for a finished accumulator, work units.
 * A stage ring that keeps the tensor core fed shows MMA waits that are a
 * small share of the MMA span ("B200 Tma Pipeline Designer", step 8: copies
 * genuinely overlapping tensor-core work). */
#define TP_TRACE_SLOTS 8

/* Per-unit event timeline per CTA (tp_gemm_opts.events): for the CTA's first
 * TP_EVENT_UNITS work units (output tiles, split-K slices or narrow tail
 * units, in the order it runs them), TP_EVENTS_PER_UNIT slots each, in this
 * order: producer about to wait for the unit's first free stage, producer
 * issued the unit's last loads, MMA issuer found the unit's accumulator free,
 * MMA issuer issued the unit's last MMAs, epilogue (warp 2) found the
 * accumulator complete, epilogue handed it back, epilogue issued the unit's
 * last store; all globaltimer nanoseconds. The last slot holds the unit's
 * index. The MMA events of a 2-SM pair are in its leader CTA's slots; the
 * plain-load producer records no producer events. Slots of units the CTA
 * did not run stay as the caller left them. */
#define TP_EVENTS_PER_UNIT 8
#define TP_EVENT_UNITS 8
#define TP_EVENT_SLOTS (TP_EVENTS_PER_UNIT * TP_EVENT_UNITS)

/* tp_gemm_bf16 / tp_gemm_bf16_f32 with explicit choices (opts may be NULL).
 * out_f32 selects a float C (1) or a bf16 C (0). */
TP_API int tp_gemm_bf16_ex(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int64_t lda,
                    int64_t ldb, int64_t ldc, int out_f32, const tp_gemm_opts* opts, void* stream);

/*
 * Split-K GEMM for problems with few output tiles (skinny M or N, deep K):
 * each (output tile, K slice) work unit runs the same mainloop and writes its
 * fp32 partial sum into slice `s` of a caller-provided workspace; a second
 * kernel adds the slices in order (fp32) and writes C (bf16 RNE or fp32).
 * Results equal C = A . B within the fp32 accumulator's error bound; the
 * summation order differs from tp_gemm_bf16's.
 *   splits:    K slices (1..k_blocks, k_blocks = ceil(K/64)); 0 chooses a
 *              count that fills the GPU, capped by what the workspace holds.
 *              Slice counts are adjusted down so that none is empty.
 *   workspace: caller-owned device memory, 16-byte aligned, at least
 *              tp_gemm_splitk_workspace_bytes(M, N, splits) bytes; the call
 *              overwrites it. Calls that overlap on the GPU must not share a
 *              workspace. With one slice it is not touched (may be NULL).
 * A and B that TMA cannot describe directly (misaligned bases, pitches not
 * multiples of 8 elements) take the plain-load producer (1-SM atom, N = 128)
 * with its row-class windows; C needs only natural alignment. A workspace
 * that is too small for an explicit `splits` returns TP_ERR_INVALID_ARG. Two
 * kernels are launched on `stream`.
 */
TP_API int tp_gemm_bf16_splitk(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                               int64_t lda, int64_t ldb, int64_t ldc, int out_f32, int splits, void* workspace,
                               int64_t workspace_bytes, const tp_gemm_opts* opts, void* stream);

/* Workspace bytes tp_gemm_bf16_splitk needs for `splits` slices:
 * splits x M x round_up(N, 4) x 4. Host-only. */
TP_API int tp_gemm_splitk_workspace_bytes(int64_t M, int64_t N, int splits, int64_t* bytes);

/*
 * tp_gemm_bf16_splitk without a caller workspace, for callers that may not
 * allocate device memory while they run (a fixed device-memory budget
 * reserved up front by another allocator, or code where cudaMalloc's
 * implicit device-wide synchronization is not allowed). The pages have no
 * counterpart: this is a property of the library, not of the method.
 *  - The partial sums live in a fixed 32 MiB array inside the library
 *    (tp_gemm_splitk_noalloc_capacity()); every GPU that loads the library
 *    holds it until the process exits. Nothing is allocated per call.
 *  - The array is created on a device when the library's module first loads
 *    there, which CUDA's lazy loading puts at the library's first call of
 *    any kind on that device. A caller that must not allocate later makes
 *    one library call per device during its set-up (tp_device_status, for
 *    example), so that the creation happens then.
 *  - The first call of this entry point on a device looks up the array's
 *    device address for that device; make that first call before any
 *    stream capture.
 *  - An explicit `splits` whose workspace (tp_gemm_splitk_workspace_bytes)
 *    exceeds the array returns TP_ERR_WORKSPACE_LIMIT; splits = 0 chooses
 *    only counts that fit (one slice needs no workspace).
 *  - Every call shares the one array and leaves its partials there. Each
 *    call writes every partial it reads, so nothing has to start at zero,
 *    but calls that overlap on the GPU (other streams, other threads) race
 *    on it: serialize them.
 * Arguments, layout and results are those of tp_gemm_bf16_splitk.
 */
TP_API int tp_gemm_bf16_splitk_noalloc(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                                       int64_t lda, int64_t ldb, int64_t ldc, int out_f32, int splits,
                                       void* stream);

/* Bytes of the fixed workspace array behind tp_gemm_bf16_splitk_noalloc. */
TP_API int64_t tp_gemm_splitk_noalloc_capacity(void);

/*
 * tp_gemm_bf16_ex on operands in host memory, end to end on `stream`: copies
 * A (M rows) and B (N rows) into the caller's device buffers dA and dB,
 * runs the GEMM into the caller's device buffer dC, and copies C back into
 * C_host. Host and device buffers have the same layout and pitches (lda,
 * ldb, ldc elements; A, B bf16; C bf16 or fp32 by out_f32), so dA holds
 * M x lda, dB N x ldb and dC M x ldc elements. The pages define only the
 * device-resident GEMM; this is its form for callers whose data lives on
 * the host (the end-to-end measurement uses it).
 *
 * Ownership: every buffer is the caller's. The call only enqueues work. C_host
 * is valid after `stream` has been synchronized, and no buffer may be reused
 * before then. Host buffers should be page-locked (cudaHostAlloc), so that
 * the copies run asynchronously on the copy engines; pageable memory works,
 * but those copies block the host.
 *
 * Errors: TP_ERR_INVALID_ARG for negative sizes, pitches below the row
 * length or NULL buffers; TP_ERR_CUDA when a copy cannot be enqueued (its
 * code via tp_last_cuda_error); otherwise the statuses of tp_gemm_bf16_ex.
 * M == 0 or N == 0 is a no-op; K == 0 copies nothing in and returns zeros.
 */
TP_API int tp_gemm_bf16_host(const void* A_host, const void* B_host, void* C_host, int64_t M, int64_t N, int64_t K,
                             int64_t lda, int64_t ldb, int64_t ldc, int out_f32, void* dA, void* dB, void* dC,
                             const tp_gemm_opts* opts, void* stream);

/*
 * Forward convolution as an implicit GEMM on the same mainloop; the A tile is
 * an im2col TMA load ("two-free-pipeline-stages": SM100_TMA_2SM_LOAD_IM2COL).
 * Cross-correlation, zero padding, no dilation, no groups:
 *   y[n][p][q][k] = sum_{r,s,c} x[n][p*stride-pad+r][q*stride-pad+s][c] * w[k][r][s][c]
 *   x: N x H x W x C (NHWC), w: K x R x S x C (KRSC), y: N x P x Q x K
 *   (NHWC), P = (H + 2 pad - R)/stride + 1, Q = (W + 2 pad - S)/stride + 1.
 * GEMM view: M = N*P*Q, N = K, K = R*S*C, walked as (r,s) outer, 64-channel
 * blocks inner. The im2col TMA producer needs C and K multiples of 8,
 * 16-byte aligned buffers, 1 <= stride <= 8, R, S <= 32 and pad < 128; other
 * problems take the plain-load producer: for a stride-1 convolution whose
 * output has the input's height and width, row-class TMA windows (pixels 8
 * apart lie 16 C bytes apart) unpacked in shared memory; otherwise each
 * row's window copied with cp.async.
 */
TP_API int tp_conv2d_fprop_bf16(const void* x_nhwc, const void* w_krsc, void* y_nhwk, int64_t N, int64_t H, int64_t W,
                         int64_t C, int64_t K, int64_t R, int64_t S, int64_t stride, int64_t pad, void* stream);

/* The convolution with explicit mainloop choices and output type. */
TP_API int tp_conv2d_fprop_bf16_ex(const void* x_nhwc, const void* w_krsc, void* y_nhwk, int64_t N, int64_t H,
                            int64_t W, int64_t C, int64_t K, int64_t R, int64_t S, int64_t stride, int64_t pad,
                            int out_f32, const tp_gemm_opts* opts, void* stream);

/*
 * dst = src, bit for bit, for a rows x cols matrix of 2-byte elements, both
 * buffers with row pitch ld (>= cols) elements. TMA path: a persistent ring
 * of tiles, TMA load -> shared memory -> TMA store, stores drained with
 * commit_group / wait_group ("B200 Tma Pipeline Designer", steps 4-7).
 * Buffers that TMA cannot describe (base not 16-byte aligned, ld*2 not a
 * multiple of 16) or copies under 64 KiB take the vectorized ld/st path.
 * src and dst must not overlap; both must be 2-byte aligned.
 */
TP_API int tp_tma_copy_2d(const void* src, void* dst, int64_t rows, int64_t cols, int64_t ld, void* stream);

/* Copy choices: box_cols x box_rows tiles (box_cols*2 a multiple of 16, both
 * <= 256), stages in {2,3,4,6,8,12}, ctas_per_sm >= 1, force_vec = 1 takes
 * the fallback path. Zero fields mean "choose". */
typedef struct {
    int box_cols;
    int box_rows;
    int stages;
    int ctas_per_sm;
    int force_vec;
} tp_copy_opts;

TP_API int tp_tma_copy_2d_ex(const void* src, void* dst, int64_t rows, int64_t cols, int64_t ld,
                      const tp_copy_opts* opts, void* stream);

/*
 * dst = transpose(src), bit for bit, for 2-byte elements: src is rows x cols
 * with row pitch ld_src (>= cols), dst is cols x rows with row pitch ld_dst
 * (>= rows): dst[c*ld_dst + r] = src[r*ld_src + c]. The copy ring of "B200
 * Tma Pipeline Designer" (steps 4-7) with a transpose between load and
 * store: 64x64 tiles arrive by TMA with 128-byte swizzle, each warp turns
 * them around in shared memory (ldmatrix / stmatrix.trans) and a TMA store
 * writes them at the swapped coordinates, drained with commit_group /
 * wait_group. Buffers TMA cannot describe (base not 16-byte aligned, a pitch
 * times 2 not a multiple of 16), copies under 64 KiB, and destination columns
 * past the last multiple of 8 take a 32x32 shared-memory tile transpose.
 * src and dst must not overlap; both must be 2-byte aligned.
 */
TP_API int tp_tma_transpose_2d(const void* src, void* dst, int64_t rows, int64_t cols, int64_t ld_src,
                               int64_t ld_dst, void* stream);

/* The transpose with ring choices: opts->stages in {2,4,6,8}, ctas_per_sm
 * (persistent one-warp CTAs per SM), force_vec; box fields are ignored (the
 * tile is 64x64). */
TP_API int tp_tma_transpose_2d_ex(const void* src, void* dst, int64_t rows, int64_t cols, int64_t ld_src,
                                  int64_t ld_dst, const tp_copy_opts* opts, void* stream);

/*
 * Streams a rows x cols matrix of 2-byte elements (row pitch `ld` elements)
 * through the TMA load ring of the copy -- persistent one-warp CTAs, each
 * taking a contiguous run of box_rows x box_cols tiles through a
 * stages-deep ring -- and discards it: the load half of "B200 Tma Pipeline
 * Designer" steps 4-7 on its own, with no store traffic beside it. It
 * measures how fast the GPU pulls an operand (the bound of a skinny GEMM
 * that streams its B once). opts may be NULL (128 x 64 tiles, 8 stages, one
 * CTA per SM); stages in {2, 4, 8, 12}. src must be 16-byte aligned with a
 * pitch of whole 16-byte granules and cols a multiple of 8
 * (TP_ERR_UNSUPPORTED otherwise: there is no fallback). Reads only.
 */
TP_API int tp_tma_read_2d(const void* src, int64_t rows, int64_t cols, int64_t ld, const tp_copy_opts* opts,
                          void* stream);

/* Synchronizes `stream`, returns the current device's status (TP_OK or the
 * first device-side failure since the last call, e.g. TP_ERR_TIMEOUT from a
 * bounded barrier wait) and clears it. Returns TP_ERR_CUDA when the
 * synchronization itself fails. */
TP_API int tp_device_status(void* stream);

/* As tp_device_status, also reporting where the failure happened (site code,
 * block and thread); any output pointer may be NULL. Sites: 1 a producer
 * waiting for a free ring stage or staging buffer, 2 the MMA issuer waiting
 * for a loaded stage, 3 the MMA issuer waiting for a drained accumulator,
 * 4 the epilogue waiting for a finished accumulator, 5 a copy ring's or the
 * plain-load GEMM's loads landing, 6 the wait for loads or MMAs in flight
 * before a CTA exits, 7 the bounded-wait self test. */
TP_API int tp_device_status_detail(void* stream, int* site, int* block, int* thread);

/* Static string naming a tp_status value. */
TP_API const char* tp_status_string(int status);

/* The CUDA error code behind the last TP_ERR_CUDA on this thread. */
TP_API int tp_last_cuda_error(void);

/*
 * Dynamic shared memory per CTA of the mainloop for (atom, pipe_depth,
 * tile_n, out_f32): stages x (A 128x64 + B (tile_n/atom)x64 bf16) plus the
 * epilogue staging, barriers and alignment slack. Writes *bytes and returns
 * TP_OK when it fits the 232,448-byte opt-in limit, TP_ERR_SMEM_BUDGET when
 * it does not ("two-free-pipeline-stages", stage budget table), or
 * TP_ERR_INVALID_ARG for an impossible combination. Host-only; needs no GPU.
 */
TP_API int tp_query_smem_bytes(int atom, int pipe_depth, int tile_n, int out_f32, int64_t* bytes);

/* What a call dispatched: the path, the mainloop variant and launch shape. */
typedef struct {
    int path;        /* TP_PATH_* */
    int atom;
    int pipe_depth;
    int tile_n;
    int out_f32;
    int conv;
    int grid;        /* CTAs launched */
    int cluster;     /* CTAs per cluster */
    int smem_bytes;  /* dynamic shared memory per CTA */
    int64_t m_tiles, n_tiles, k_blocks;
    int splits;      /* K slices (1 unless split-K ran) */
    int tail_units;  /* narrow units of the last wave (0: none) */
    int l2_hint;     /* operand L2 priorities used (tp_gemm_opts.l2_hint 1-6) */
    int tail_parts;  /* column parts of each narrow-tail tile (2 or 4; 0: no tail) */
} tp_plan;

/*
 * The plan tp_gemm_bf16_ex would launch for these arguments on a GPU with
 * sm_count SMs (0 = ask the current device). Host-only when sm_count > 0:
 * alignment, tile counts, variant choice and shared-memory budget, no launch.
 * Returns the status tp_gemm_bf16_ex would return before launching.
 */
TP_API int tp_gemm_plan(const void* A, const void* B, const void* C, int64_t M, int64_t N, int64_t K, int64_t lda,
                 int64_t ldb, int64_t ldc, int out_f32, const tp_gemm_opts* opts, int sm_count, tp_plan* plan);

/* The plan of the last GEMM / conv / copy call made on this thread. */
TP_API int tp_last_plan(tp_plan* plan);

/* One compiled mainloop variant. */
typedef struct {
    int atom, pipe_depth, tile_n, out_f32, conv, smem_bytes;
    int ldg;    /* plain-load producer: 0 none (TMA), 1 GEMM row-class windows or conv cp.async
                   windows, 2 conv row-class windows (stride 1, output the input's size) */
    int splitk; /* 1: split-K partials into a workspace */
} tp_kernel_desc;

/* Writes up to cap compiled variants to out (may be NULL) and returns how
 * many there are. Host-only. */
TP_API int tp_list_kernels(tp_kernel_desc* out, int cap);

/*
 * Read-after-write latency of a fused multiply-add, measured on this GPU
 * ("hardware-hazards-b200" note, "Fixed-latency RAW under-stalls": a chain
 * a = a*1 + 1 whose result must be exactly seed + chain). One thread runs
 * `chain` dependent fma.rn links (kind 0: fp32, kind 1: fp64; chain a
 * multiple of 64, at most 2^26) between two clock64 reads. Writes the chain's
 * result and the SM cycles per link, an upper bound on the latency (loop and
 * clock-read overhead included). Synchronizes `stream`. The note's B200
 * figures: 4 cycles fp32, 8 cycles fp64.
 */
TP_API int tp_probe_fma_latency(int kind, int chain, double seed, double* result, double* cycles_per_link,
                                void* stream);

/*
 * Failure-detection self test of the real mainloop: runs the 1-SM GEMM
 * C = A.B (fp32 C, lda = ldb = K, ldc = N) with its producer withholding the
 * expect_tx arrival of the first stage while still issuing that stage's TMA
 * loads -- the lost-arrival bug of CUTLASS issue #3722 ("Cause"). The MMA
 * issuer's bounded wait on that stage, and the waits that depend on it
 * (epilogue, producer), must give up after limit_ms (1..10000); the first to
 * expire records TP_ERR_TIMEOUT (site 2 MMA issuer, 4 epilogue, 1 producer),
 * and the kernel must let its landed loads drain, free tensor memory and return;
 * tp_device_status then reports the timeout and the context stays usable.
 * C is left unspecified. Sizes: M, N <= 4096, 64 <= K <= 4096.
 */
TP_API int tp_selftest_mainloop_withheld_arrival(const void* A, const void* B, float* C, int64_t M, int64_t N,
                                                 int64_t K, uint32_t limit_ms, void* stream);

/*
 * The other half of the lost-completion self test: the MMA issuer skips one
 * tcgen05.commit, the failure "consuming right after the load is issued,
 * missing the barrier wait" seen from the consumer's side ("B200 Tma Pipeline
 * Designer", Failure modes). which = 1 skips the commit to empty[s] after its
 * first k-block, so the producer's bounded wait for that stage (and the MMA
 * issuer's wait for its refill) must give up (site 1 producer or 2 MMA
 * issuer); which = 2 skips the commit to acc_full[b] after its first tile,
 * so the epilogue's wait (site 4), and an MMA issuer's wait for that
 * accumulator (site 3), must give up. The GEMM is C = A.B (fp32 C, lda =
 * ldb = K, ldc = N) on atom 1 or 2 at MMA N = 128, each CTA's waits limited
 * to limit_ms (1..10000); the kernel drains its MMAs and loads, frees tensor
 * memory and returns, and tp_device_status reports TP_ERR_TIMEOUT. C is left
 * unspecified. Sizes: M, N <= 4096, 64 <= K <= 4096; which = 1 needs more
 * k-blocks (K / 64) than stages to reach a stage's second use.
 */
TP_API int tp_selftest_mainloop_skipped_commit(const void* A, const void* B, float* C, int64_t M, int64_t N,
                                               int64_t K, int which, int atom, uint32_t limit_ms, void* stream);

/* Launches one CTA that waits on an mbarrier nothing arrives on, with a
 * limit of limit_us microseconds: the wait must give up and record
 * TP_ERR_TIMEOUT, which tp_device_status then returns. Checks that a stuck
 * pipeline ends with a status instead of a hang. */
TP_API int tp_selftest_wait_timeout(uint32_t limit_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TP_H */
