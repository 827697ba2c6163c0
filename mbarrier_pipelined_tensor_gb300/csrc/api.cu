// C ABI of libtp (declared in include/tp.h): argument checks, TMA-vs-fallback
// dispatch ("B200 Tma Pipeline Designer", step 1), tensor-map construction
// (step 2; "CUDA 13 TMA Descriptor Notes": byte strides, BFLOAT16 type),
// mainloop variant choice against the shared-memory budget
// ("two-free-pipeline-stages", stage budget table) and the device status
// record.
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "gemm_kernel.cuh"
#include "tensor_map.h"
#include "tp.h"

static_assert(TP_TRACE_SLOTS == tp::kTraceSlots, "trace layout");
static_assert(TP_EVENT_SLOTS == tp::kEventSlots && TP_EVENTS_PER_UNIT == tp::kEventsPerUnit, "event layout");
static_assert(TP_PROTO_SLOTS == tp::kProtoSlots && TP_PROTO_PHASES == tp::PROTO_PHASES &&
                  TP_PROTO_MAX_STAGES == tp::PROTO_MAX_STAGES && TP_PROTO_TX_EXPECT == tp::PROTO_TX_EXPECT &&
                  TP_PROTO_TX_ISSUED == tp::PROTO_TX_ISSUED,
              "arrival accounting layout");

namespace tp {
const KernelEntry* table_mainloop_cg1(int* n);
const KernelEntry* table_mainloop_cg2(int* n);
const KernelEntry* table_mainloop_conv(int* n);
const KernelEntry* table_mainloop_fallback(int* n);
const KernelEntry* table_mainloop_splitk(int* n);
const KernelEntry* table_mainloop_n64(int* n);
cudaError_t launch_splitk_reduce(const float* ws, void* C, int M, int N, int64_t ldw, int64_t ldc, int splits,
                                 int out_f32, int sm_count, cudaStream_t st);
cudaError_t launch_tma_copy_any(int stages, const CUtensorMap& s, const CUtensorMap& d, const CopyParams& p,
                                int grid, cudaStream_t st);
int copy_smem_bytes(int stages, uint32_t tile_bytes);
cudaError_t launch_tma_read_any(int stages, const CUtensorMap& s, const CopyParams& p, int grid, cudaStream_t st);
cudaError_t launch_vec_copy(const void* src, void* dst, int64_t rows, int64_t cols, int64_t ld, int sm_count,
                            cudaStream_t st);
cudaError_t launch_zero_fill(void* c, int64_t M, int64_t N, int64_t ldc, int elem_bytes, cudaStream_t st);
cudaError_t launch_wait_selftest(const WaitCtl& w, cudaStream_t st);
int transpose_smem_bytes(int stages);
cudaError_t run_fma_probe(int kind, double seed, int blocks, cudaStream_t st, double* result, long long* cycles);
cudaError_t launch_tma_transpose(int stages, const CUtensorMap& s, const CUtensorMap& d, int tiles_x, int tiles_y,
                                 const WaitCtl& w, int grid, cudaStream_t st);
cudaError_t launch_vec_transpose(const void* src, void* dst, int64_t r0, int64_t rows, int64_t cols, int64_t ld_src,
                                 int64_t ld_dst, int sm_count, cudaStream_t st);
}  // namespace tp

using namespace tp;

namespace {

__device__ DevStatus g_status;  // one per device that loads the library

constexpr int kMaxSmemPerCta = 232448;  // sm_100-class opt-in limit (227 KiB)
constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready;
    int sm_count;
    DevStatus* status;
};

DeviceState g_dev[kMaxDevices];
std::mutex g_dev_mu;
thread_local int t_last_cuda_error = 0;
// Set only inside tp_selftest_mainloop_withheld_arrival /
// tp_selftest_mainloop_skipped_commit for their one launch.
thread_local int t_selftest_withhold = 0;
thread_local int t_selftest_skip_commit = 0;
thread_local uint64_t t_selftest_limit_ns = 0;
thread_local tp_plan t_last_plan = {};

int cuda_fail(cudaError_t e)
{
    t_last_cuda_error = static_cast<int>(e);
    return TP_ERR_CUDA;
}

int device_state(DeviceState** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return TP_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DeviceState& d = g_dev[dev];
    if (!d.ready) {
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e);
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_status);
        if (e != cudaSuccess) return cuda_fail(e);
        d.sm_count = sms;
        d.status = static_cast<DevStatus*>(p);
        d.ready = true;
    }
    *out = &d;
    return TP_OK;
}

uint64_t wait_limit_ns()
{
    static uint64_t v = [] {
        const char* s = std::getenv("TP_WAIT_LIMIT_MS");
        long ms = s ? std::strtol(s, nullptr, 10) : 0;
        if (ms <= 0) ms = 4000;
        return static_cast<uint64_t>(ms) * 1000000ull;
    }();
    return v;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// fp32 workspace row of split-K: N rounded up to whole 16-byte granules.
int64_t splitk_ldw(int64_t N) { return (N + 3) / 4 * 4; }

// ------------------------------------------------------ variant table ---

constexpr int kTables = 6;

struct Tables {
    const KernelEntry* t[kTables];
    int n[kTables];
};

const Tables& tables()
{
    static Tables tb = [] {
        Tables x{};
        x.t[0] = table_mainloop_cg1(&x.n[0]);
        x.t[1] = table_mainloop_cg2(&x.n[1]);
        x.t[2] = table_mainloop_conv(&x.n[2]);
        x.t[3] = table_mainloop_fallback(&x.n[3]);
        x.t[4] = table_mainloop_splitk(&x.n[4]);
        x.t[5] = table_mainloop_n64(&x.n[5]);
        return x;
    }();
    return tb;
}

const KernelEntry* find_kernel(const KernelKey& k)
{
    const Tables& tb = tables();
    for (int i = 0; i < kTables; ++i)
        for (int j = 0; j < tb.n[i]; ++j) {
            const KernelKey& e = tb.t[i][j].key;
            if (e.cta_group == k.cta_group && e.bn == k.bn && e.stages == k.stages && e.out_f32 == k.out_f32 &&
                e.conv == k.conv && e.ldg == k.ldg && e.splitk == k.splitk)
                return &tb.t[i][j];
        }
    return nullptr;
}

// Mirrors MainloopCfg::SMEM_BYTES (plus, for the plain-load producer, its
// staging buffers: ldg_extra_bytes).
int64_t mainloop_smem(int atom, int depth, int tile_n, int ldg = 0, int conv = 0)
{
    const int64_t a = 128 * 64 * 2;
    const int64_t rows = 128 + tile_n / atom;
    const int64_t b = static_cast<int64_t>(tile_n / atom) * 64 * 2;
    const int64_t epi = 4 * 2 * 32 * 128;
    const int64_t staging = !ldg ? 0
                            : ldg == kLdgConvWin ? static_cast<int64_t>(kWinStaging) * (rows * kWinRowConv + 16) + 64
                            : conv ? static_cast<int64_t>(kLdgStaging) * rows * (kLdgWindow + 4)
                                   : static_cast<int64_t>(kWinStaging) * rows * kWinRow + 64;
    return 1024 + depth * (a + b) + epi + 256 + staging;
}

int deepest_fitting(int atom, int tile_n)
{
    int d = 9;
    while (d > 2 && mainloop_smem(atom, d, tile_n) > kMaxSmemPerCta) --d;
    return d;
}

// Picks the (atom, MMA N) not fixed by the caller: the variant with the
// least estimated time, waves x tile_n / eff, where waves counts rounds of
// output tiles over the persistent clusters and eff is the variant's
// measured throughput on a large square GEMM relative to the best one
// (2-SM, N = 256 at its deepest ring). A fixed field (*atom or *tile_n
// nonzero) restricts the candidates, and so does the kernel table: only
// variants built for this output type and operand form (GEMM or conv) at
// their deepest ring compete. (An explicit ring depth is checked after the
// choice, against the shared-memory budget and the table.) For a split-K
// call the N = 64 tile is left out: there the K slices already spread a
// short tile row over the SMs, and a wider tile keeps more of B in flight
// per CTA and re-reads A less (128 x 8192 x 16384 on GB300: N = 128 in 2
// slices 59.7 us, N = 256 in 4 slices 58.8 us, N = 64 unsplit 61.9 us).
// Returns false when no variant qualifies.
bool choose_variant(int64_t M, int64_t N, int64_t k_blocks, int sm_count, int out_f32, int conv, int splitk,
                    int* atom, int* tile_n)
{
    struct Cand {
        int atom, tile_n;
        double eff;
    };
    // Efficiency relative to the 2-SM / N = 256 variant: the PIPE_DEPTH
    // sweep at 8192^3 on GB300 (deepest ring of each variant).
    static const Cand kCands[] = {{2, 256, 1.00}, {1, 256, 0.86}, {2, 128, 0.89}, {1, 128, 0.75}, {1, 64, 0.54}};
    double best = 0;
    Cand pick = kCands[0];
    bool have = false;
    for (const Cand& c : kCands) {
        if ((*atom && c.atom != *atom) || (*tile_n && c.tile_n != *tile_n)) continue;
        if (splitk && c.tile_n == 64) continue;
        if (!find_kernel(KernelKey{c.atom, c.tile_n, deepest_fitting(c.atom, c.tile_n), out_f32, conv, 0, 0}))
            continue;
        const int64_t tiles = cdiv(M, 128 * c.atom) * cdiv(N, c.tile_n);
        const int64_t clusters = std::max<int64_t>(1, sm_count / c.atom);
        double waves = static_cast<double>(cdiv(tiles, clusters));
        // The 2-SM, N = 256 variant runs a partial last wave that fits twice
        // as half-width units: after at least one full wave it counts half.
        const int64_t r = tiles % clusters;
        if (c.atom == 2 && c.tile_n == 256 && tiles >= clusters && r > 0 && 2 * r <= clusters)
            waves -= 4 * r <= clusters ? 0.6 : 0.5;
        // Estimated time (ns): one k-block of a 128 x tile_n tile is 1.31 *
        // tile_n ns at one SM's dense BF16 rate, scaled by the variant's
        // measured efficiency.
        double cost = waves * static_cast<double>(k_blocks) * 1.31 * c.tile_n / c.eff;
        // Short K: a narrow tile's fixed per-tile cost (ring fill, epilogue)
        // is a larger share of its work (4096 x 4096 x 512: N = 128 tiles
        // measured 27 us against 23 us for N = 256).
        if (k_blocks <= 16 && c.tile_n <= 128) cost *= 1.25;
        // A cluster launch and its pair barriers cost about 2 us more per
        // call than the 1-SM atom (a one-tile GEMM: 10.9 against 8.9 us).
        if (c.atom == 2) cost += 2000.0;
        if (!have || cost < best) {
            best = cost;
            pick = c;
            have = true;
        }
    }
    *atom = pick.atom;
    *tile_n = pick.tile_n;
    return have;
}

// Variant and launch shape for a GEMM view M x N x K (k_blocks given).
int plan_mainloop(int64_t M, int64_t N, int64_t k_blocks, int out_f32, int conv, int ldg, const tp_gemm_opts* o,
                  int sm_count, tp_plan* pl, int splitk = 0)
{
    int atom = o && o->atom ? o->atom : 0;
    int tile_n = o && o->tile_n ? o->tile_n : 0;
    if (atom != 0 && atom != 1 && atom != 2) return TP_ERR_INVALID_ARG;
    if (tile_n != 0 && tile_n != 64 && tile_n != 128 && tile_n != 256) return TP_ERR_INVALID_ARG;
    if (ldg) {
        // The plain-load producer exists for the 1-SM atom at N = 128 only.
        if ((atom && atom != 1) || (tile_n && tile_n != 128)) return TP_ERR_UNSUPPORTED;
        atom = 1;
        tile_n = 128;
    }
    if ((atom == 0 || tile_n == 0) &&
        !choose_variant(M, N, k_blocks, sm_count, out_f32, conv, splitk, &atom, &tile_n))
        return TP_ERR_UNSUPPORTED;
    // The plain-load producer stages its copies outside the ring, which
    // leaves room for kLdgStages ring stages (the GEMM's row-class windows:
    // kWinStages).
    int depth = o && o->pipe_depth ? o->pipe_depth
                                   : (ldg ? (conv && ldg == kLdgPlain ? kLdgStages : kWinStages)
                                          : deepest_fitting(atom, tile_n));
    if (depth < 2 || depth > 9) return TP_ERR_INVALID_ARG;
    const int64_t smem = mainloop_smem(atom, depth, tile_n, ldg, conv);
    if (smem > kMaxSmemPerCta) return TP_ERR_SMEM_BUDGET;
    const KernelEntry* k = find_kernel(KernelKey{atom, tile_n, depth, out_f32, conv, ldg, 0});
    if (!k) return TP_ERR_UNSUPPORTED;

    const int64_t m_tiles = cdiv(M, 128 * atom);
    const int64_t n_tiles = cdiv(N, tile_n);
    const int64_t tiles = m_tiles * n_tiles;
    if (tiles > (1ll << 31) - 1 || k_blocks > (1ll << 31) - 1) return TP_ERR_UNSUPPORTED;
    int64_t clusters = sm_count / atom;
    if (o && o->max_ctas > 0) clusters = std::max<int64_t>(1, o->max_ctas / atom);
    if (clusters > tiles) clusters = tiles;
    if (clusters < 1) clusters = 1;

    pl->path = ldg ? TP_PATH_FALLBACK_MAINLOOP : TP_PATH_MAINLOOP;
    pl->atom = atom;
    pl->pipe_depth = depth;
    pl->tile_n = tile_n;
    pl->out_f32 = out_f32;
    pl->conv = conv;
    pl->grid = static_cast<int>(clusters * atom);
    pl->cluster = atom;
    pl->smem_bytes = k->smem_bytes;
    pl->m_tiles = m_tiles;
    pl->n_tiles = n_tiles;
    pl->k_blocks = k_blocks;
    pl->splits = 1;
    return TP_OK;
}

// K slices for split-K. Splitting pays only when the output tiles leave most
// of the GPU idle and the fp32 partials (written and re-read once per slice)
// stay small next to the operands: on a GB300, 128 x 8192 x 16384 gains 12%
// with 2 slices, while 4096 x 4096 x 512 loses 3x and 1000^3 loses 25%.
int choose_splits(int64_t tiles, int64_t clusters, int64_t k_blocks, int64_t M, int64_t N, int64_t K)
{
    if (tiles * 2 > clusters) return 1;
    int64_t s = clusters / tiles;
    s = std::min<int64_t>(s, std::max<int64_t>(1, k_blocks / 4));
    s = std::min<int64_t>(s, 16);
    const double operand_bytes = 2.0 * static_cast<double>(M * K + N * K);
    while (s > 1 && 8.0 * static_cast<double>(s * M * splitk_ldw(N)) > 0.25 * operand_bytes) --s;
    return static_cast<int>(s);
}

// Slices actually used so that none is empty.
void normalize_splits(int64_t k_blocks, int* splits, int* kb_per_split)
{
    int s = *splits < 1 ? 1 : *splits;
    if (s > k_blocks) s = static_cast<int>(k_blocks);
    const int kps = static_cast<int>(cdiv(k_blocks, s));
    *kb_per_split = kps;
    *splits = static_cast<int>(cdiv(k_blocks, kps));
}

int64_t max_clusters_for(const tp_gemm_opts* o, int sm_count, int atom);

// Narrow tail for the 2-SM atom at N = 256: when the tiles left for the last,
// partial wave (r = tiles mod W) fit twice into one wave, they run as 2r
// half-width units, so that wave takes about half as long. W is the number
// of clusters that run at once: the grid cap (max_ctas) or the GPU's SMs /
// 2, whichever is smaller. When they fit four times into one wave they run
// as 4r quarter-width units instead (N = 64): the tail is bound by each
// CTA's operand stream, which a quarter unit cuts by a sixth against a half
// (A 16 KiB + B 4 KiB against 16 + 8 per K block) while it also halves the
// MMAs; the conv 32x56x56x256 (12 tiles left on 76 clusters) ran its tail
// in 5.6 instead of 6.7 us. A problem with fewer tiles than W is all tail.
// The grid is W clusters (persistent), or one per unit when the cap allows
// as many (non-persistent).
void set_narrow_tail(tp_plan& pl, GemmParams& p, const tp_gemm_opts* o, int sm_count)
{
    p.n_full = 0;
    p.tail_units = 0;
    p.tail_parts = 2;
    pl.tail_parts = 0;
    if (pl.atom != 2 || pl.tile_n != 256) return;
    const int64_t cap = max_clusters_for(o, sm_count, pl.atom);
    const int64_t wave = std::min<int64_t>(cap, std::max<int64_t>(1, sm_count / pl.atom));
    if (wave < 2) return;
    const int64_t tiles = pl.m_tiles * pl.n_tiles;
    const int64_t r = tiles % wave;
    if (r == 0 || 2 * r > wave) return;
    const int parts = 4 * r <= wave ? 4 : 2;
    p.n_full = static_cast<int>(tiles - r);
    p.tail_units = static_cast<int>(parts * r);
    p.tail_parts = parts;
    const int64_t units = tiles - r + parts * r;
    pl.grid = static_cast<int>(std::min<int64_t>(cap, units) * pl.atom);
    pl.tail_units = p.tail_units;
    pl.tail_parts = parts;
}

int64_t max_clusters_for(const tp_gemm_opts* o, int sm_count, int atom)
{
    const int64_t c = (o && o->max_ctas > 0) ? o->max_ctas / atom : sm_count / atom;
    return c < 1 ? 1 : c;
}

// Tile raster: group_m M-tiles share one sweep over N. By default a group
// spans 3072 rows of A (24 tiles of the 1-SM atom, 12 pair tiles of the 2-SM
// atom). With the GEMM's odd waves walking K backwards, consecutive waves
// reuse the A rows they share from L2; on GB300 at 8192^3 the 2-SM atom's
// DRAM reads per launch were 1237, 1123, 914, 820, 856 and 1410 MB for
// groups of 4, 6, 8, 12, 16 and 32 pair tiles, and 12 ran 0.4-0.9% faster
// than 8 at 8192^3, 12288^2 x 8192 and 16384^2 x 4096 (power-capped).
int group_m_for(const tp_gemm_opts* o, int64_t m_tiles, int atom)
{
    int g = o && o->group_m > 0 ? o->group_m : 3072 / (128 * (atom > 0 ? atom : 1));
    if (g > m_tiles) g = static_cast<int>(m_tiles);
    return g < 1 ? 1 : g;
}

// L2 priorities of the A / B loads (0 normal, 1 evict first, 2 evict last).
// Chosen (l2_hint 0, GEMM) from how often each operand is read: B, read by
// at most two tile rows, streams through L2 once and goes first, while a
// small A, read by every tile of the row, is kept; likewise mirrored. The
// convolution's A is an im2col view that overlapping windows re-read from
// L2, so it keeps normal priority.
int l2_mode_for(const tp_gemm_opts* o, int64_t m_tiles, int64_t n_tiles, double a_bytes, double b_bytes, bool gemm)
{
    const int h = o ? o->l2_hint : 0;
    if (h != 0) return h;
    if (!gemm) return 1;
    constexpr double kKeep = 16.0e6;
    if (m_tiles <= 2 && a_bytes <= kKeep && 4.0 * a_bytes <= b_bytes) return 2;
    if (n_tiles <= 2 && b_bytes <= kKeep && 4.0 * b_bytes <= a_bytes) return 5;
    return 1;
}

// Per-operand load policies (GemmParams::l2_a / l2_b): 0 no policy, 1 evict
// first, 2 evict last, 3 an explicit evict_normal policy.
void l2_hints_for(int mode, int* a, int* b)
{
    *a = 0;
    *b = 0;
    switch (mode) {
    case 2: *a = 2; *b = 1; break;
    case 3: *a = 2; break;
    case 4: *b = 1; break;
    case 5: *a = 1; *b = 2; break;
    case 6: *b = 2; break;
    case 7: *a = 3; *b = 3; break;
    default: break;  // 1: normal priority, no policy
    }
}

// Row-class windows (WinMaps) of a bf16 operand of `rows` rows of K
// elements at pitch ld (elements; any base with 2-byte alignment): class
// q's map starts at row q's address rounded down to 16 bytes, steps 8 rows
// (16 ld bytes) per row, and is K plus the rounding (delta, in elements)
// wide, so TMA reads nothing outside the operand and fills past K with
// zeros. A class with no rows (rows < 8) repeats class 0: the tile rows it
// feeds lie past the last row and are never stored.
int encode_windows(CUtensorMap* maps, const void* X, int64_t K, int64_t rows, int64_t ld, uint32_t box_rows,
                   uint32_t* deltas, uint32_t box_cols = 72)
{
    *deltas = 0;
    for (int q = 0; q < 8; ++q) {
        const int64_t c = q < rows ? q : 0;
        const uintptr_t row = reinterpret_cast<uintptr_t>(X) + static_cast<uintptr_t>(c * ld * 2);
        const uintptr_t base = row & ~static_cast<uintptr_t>(15);
        const uint32_t delta = static_cast<uint32_t>((row - base) / 2);
        TiledDesc d{CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, reinterpret_cast<void*>(base),
                    {static_cast<uint64_t>(K + delta), static_cast<uint64_t>((rows - c + 7) / 8)},
                    {static_cast<uint64_t>(ld) * 16}, {box_cols, box_rows}, CU_TENSOR_MAP_SWIZZLE_NONE};
        const int st = encode_tiled(&maps[q], d);
        if (st) return st;
        *deltas |= delta << (3 * q);
    }
    return TP_OK;
}

// The split-K workspace as the epilogue's store map: `splits` slices of M
// rows of ldw floats, 32 x 32 boxes.
int encode_splitk_workspace(CUtensorMap* map, void* ws, int64_t ldw, int64_t M, int splits)
{
    TiledDesc dw{CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ws,
                 {static_cast<uint64_t>(ldw), static_cast<uint64_t>(M), static_cast<uint64_t>(splits)},
                 {static_cast<uint64_t>(ldw) * 4, static_cast<uint64_t>(M * ldw) * 4},
                 {32, 32, 1}, CU_TENSOR_MAP_SWIZZLE_128B};
    return encode_tiled(map, dw);
}

int gemm_plan_impl(const void* A, const void* B, const void* C, int64_t M, int64_t N, int64_t K, int64_t lda,
                   int64_t ldb, int64_t ldc, int out_f32, const tp_gemm_opts* opts, int sm_count, tp_plan* pl,
                   int splitk = 0)
{
    std::memset(pl, 0, sizeof(*pl));
    if (M < 0 || N < 0 || K < 0) return TP_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return TP_OK;
    if (lda < K || ldb < K || ldc < N) return TP_ERR_INVALID_ARG;
    if (!C || (K > 0 && (!A || !B))) return TP_ERR_INVALID_ARG;
    const int eb = out_f32 ? 4 : 2;
    if (K == 0) {
        pl->path = TP_PATH_ZERO_FILL;
        pl->out_f32 = out_f32;
        return TP_OK;
    }
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return TP_ERR_UNSUPPORTED;
    // Elements must at least be naturally aligned.
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B)) & 1u ||
        reinterpret_cast<uintptr_t>(C) % eb)
        return TP_ERR_INVALID_ARG;
    // TMA suitability of the operands: 16-byte aligned bases and byte
    // pitches; otherwise the plain-load producer feeds the same mainloop. C
    // does not decide it: a C that TMA cannot store is written with plain
    // stores by the epilogue.
    const int ldg = (!aligned16(A) || !aligned16(B) || (lda * 2) % 16 || (ldb * 2) % 16) ? 1 : 0;
    if (opts && (opts->l2_hint < 0 || opts->l2_hint > 7)) return TP_ERR_INVALID_ARG;
    const int st = plan_mainloop(M, N, cdiv(K, 64), out_f32, 0, ldg, opts, sm_count, pl, splitk);
    if (st == TP_OK)
        pl->l2_hint = l2_mode_for(opts, pl->m_tiles, pl->n_tiles, 2.0 * static_cast<double>(M) * static_cast<double>(K),
                                  2.0 * static_cast<double>(N) * static_cast<double>(K), true);
    return st;
}

// The kernels' FastDiv divisors, from the launch's tile counts and (conv)
// extents; a divisor that does not apply is 1.
void set_divisors(GemmParams& p)
{
    auto one = [](int64_t v) { return static_cast<uint32_t>(v > 0 ? v : 1); };
    const int64_t tiles = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
    const int gm = std::max(1, p.group_m);
    const int64_t groups = (p.m_tiles + gm - 1) / gm;
    p.div_tiles = make_fastdiv(one(tiles));
    p.div_group = make_fastdiv(one(static_cast<int64_t>(gm) * p.n_tiles));
    p.div_gm = make_fastdiv(one(gm));
    p.div_gm_last = make_fastdiv(one(p.m_tiles - (groups - 1) * gm));
    p.div_pq = make_fastdiv(one(static_cast<int64_t>(p.conv_P) * p.conv_Q));
    p.div_q = make_fastdiv(one(p.conv_Q));
    p.div_cblocks = make_fastdiv(one(p.conv_cblocks));
    p.div_s = make_fastdiv(one(p.conv_S));
}

// ldg: the plain-load form of a fallback plan (kLdgPlain or kLdgConvWin).
int launch_plan(const tp_plan& pl, GemmLaunch& L, cudaStream_t st, int ldg = kLdgPlain)
{
    const KernelEntry* k = find_kernel(KernelKey{pl.atom, pl.tile_n, pl.pipe_depth, pl.out_f32, pl.conv,
                                                 pl.path == TP_PATH_FALLBACK_MAINLOOP ? ldg : 0,
                                                 pl.splits > 1 ? 1 : 0});
    if (!k) return TP_ERR_UNSUPPORTED;
    L.grid = pl.grid;
    L.stream = st;
    set_divisors(L.params);
    cudaError_t e = k->launch(L);
    if (e != cudaSuccess) return cuda_fail(e);
    return TP_OK;
}

}  // namespace

// ===================================================================== ABI ==

extern "C" {

const char* tp_status_string(int s)
{
    switch (s) {
    case TP_OK: return "TP_OK";
    case TP_ERR_INVALID_ARG: return "TP_ERR_INVALID_ARG";
    case TP_ERR_UNSUPPORTED: return "TP_ERR_UNSUPPORTED";
    case TP_ERR_CUDA: return "TP_ERR_CUDA";
    case TP_ERR_DRIVER_ENCODE: return "TP_ERR_DRIVER_ENCODE";
    case TP_ERR_TIMEOUT: return "TP_ERR_TIMEOUT";
    case TP_ERR_SMEM_BUDGET: return "TP_ERR_SMEM_BUDGET";
    case TP_ERR_WORKSPACE_LIMIT: return "TP_ERR_WORKSPACE_LIMIT";
    default: return "TP_ERR_UNKNOWN";
    }
}

int tp_last_cuda_error(void) { return t_last_cuda_error; }

int tp_last_plan(tp_plan* plan)
{
    if (!plan) return TP_ERR_INVALID_ARG;
    *plan = t_last_plan;
    return TP_OK;
}

int tp_query_smem_bytes(int atom, int pipe_depth, int tile_n, int out_f32, int64_t* bytes)
{
    (void)out_f32;  // the staging buffers are 128-byte rows for either output type
    if ((atom != 1 && atom != 2) || (tile_n != 64 && tile_n != 128 && tile_n != 256) || pipe_depth < 1 || !bytes)
        return TP_ERR_INVALID_ARG;
    *bytes = mainloop_smem(atom, pipe_depth, tile_n);
    return *bytes <= kMaxSmemPerCta ? TP_OK : TP_ERR_SMEM_BUDGET;
}

int tp_list_kernels(tp_kernel_desc* out, int cap)
{
    const Tables& tb = tables();
    int n = 0;
    for (int i = 0; i < kTables; ++i)
        for (int j = 0; j < tb.n[i]; ++j, ++n) {
            if (out && n < cap) {
                const KernelEntry& e = tb.t[i][j];
                out[n] = tp_kernel_desc{e.key.cta_group, e.key.stages, e.key.bn, e.key.out_f32, e.key.conv,
                                        e.smem_bytes, e.key.ldg, e.key.splitk};
            }
        }
    return n;
}

int tp_gemm_plan(const void* A, const void* B, const void* C, int64_t M, int64_t N, int64_t K, int64_t lda,
                 int64_t ldb, int64_t ldc, int out_f32, const tp_gemm_opts* opts, int sm_count, tp_plan* plan)
{
    if (!plan) return TP_ERR_INVALID_ARG;
    if (sm_count <= 0) {
        DeviceState* d = nullptr;
        int st = device_state(&d);
        if (st) return st;
        sm_count = d->sm_count;
    }
    const int st = gemm_plan_impl(A, B, C, M, N, K, lda, ldb, ldc, out_f32 ? 1 : 0, opts, sm_count, plan);
    if (st == TP_OK && plan->path == TP_PATH_MAINLOOP && !(opts && opts->no_tail)) {
        GemmParams unused{};
        set_narrow_tail(*plan, unused, opts, sm_count);
    }
    return st;
}

}  // extern "C"

namespace {

// The GEMM launch shared by the plain and the split-K entry points.
// splitk: 0 plain; 1 split-K with `splits` slices (0 = choose) into the
// caller's fp32 workspace, then a reduction into C.
int gemm_impl(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
              int64_t ldc, int out_f32, const tp_gemm_opts* opts, int splitk, int splits, void* ws,
              int64_t ws_bytes, void* stream)
{
    out_f32 = out_f32 ? 1 : 0;
    tp_plan pl;
    std::memset(&pl, 0, sizeof(pl));
    t_last_plan = pl;
    if (M < 0 || N < 0 || K < 0 || splits < 0 || ws_bytes < 0) return TP_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return TP_OK;
    DeviceState* dev = nullptr;
    int st = device_state(&dev);
    if (st) return st;
    // Split-K of a single-tile-row problem (M <= 128): the 2-SM atom would
    // compute a pair tile half of which is out of bounds; use the 1-SM atom.
    tp_gemm_opts local{};
    if (splitk && M <= 128 && !(opts && opts->atom)) {
        if (opts) local = *opts;
        local.atom = 1;
        opts = &local;
    }
    st = gemm_plan_impl(A, B, C, M, N, K, lda, ldb, ldc, out_f32, opts, dev->sm_count, &pl, splitk);
    if (st) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (pl.path == TP_PATH_ZERO_FILL) {
        cudaError_t e = launch_zero_fill(C, M, N, ldc, out_f32 ? 4 : 2, s);
        t_last_plan = pl;
        return e == cudaSuccess ? TP_OK : cuda_fail(e);
    }
    const bool ldg = pl.path == TP_PATH_FALLBACK_MAINLOOP;
    const int64_t ldw = splitk_ldw(N);
    int kps = static_cast<int>(pl.k_blocks);
    if (splitk) {
        const int64_t slice_bytes = M * ldw * 4;
        const int64_t cap = (ws && slice_bytes > 0) ? ws_bytes / slice_bytes : 0;
        const int64_t tiles = pl.m_tiles * pl.n_tiles;
        const int64_t clusters = std::max<int64_t>(1, (opts && opts->max_ctas > 0 ? opts->max_ctas : dev->sm_count) /
                                                          pl.atom);
        int sp = splits > 0 ? splits : choose_splits(tiles, clusters, pl.k_blocks, M, N, K);
        if (splits == 0 && sp > cap) sp = static_cast<int>(std::max<int64_t>(1, cap));
        normalize_splits(pl.k_blocks, &sp, &kps);
        if (sp > 1) {
            if (sp > cap || (reinterpret_cast<uintptr_t>(ws) & 15u)) return TP_ERR_INVALID_ARG;
            const KernelEntry* k = find_kernel(KernelKey{pl.atom, pl.tile_n, pl.pipe_depth, 1, 0, ldg ? 1 : 0, 1});
            if (!k) return TP_ERR_UNSUPPORTED;
            pl.splits = sp;
            int64_t units = tiles * sp;
            int64_t cl = std::min<int64_t>(clusters, units);
            pl.grid = static_cast<int>(cl * pl.atom);
            pl.smem_bytes = k->smem_bytes;
        }
    }
    const bool use_splitk = pl.splits > 1;
    const int cg = pl.atom;
    const int b_rows = pl.tile_n / cg;
    GemmLaunch L;
    std::memset(&L, 0, sizeof(L));
    GemmParams& p = L.params;
    // the narrow tail (2-SM, N = 256) before the maps: it sets their box
    if (!use_splitk && !(opts && opts->no_tail)) set_narrow_tail(pl, p, opts, dev->sm_count);
    const uint32_t eb = out_f32 ? 4 : 2;
    // TMA stores write whole 16-byte granules of a row: the C map ends at the
    // last full granule, the epilogue stores the rest (all of C when the
    // plain-load path runs). Split-K partials go to the workspace, whose rows
    // are whole granules.
    const bool c_tma = aligned16(C) && (ldc * eb) % 16 == 0;
    const int64_t n_tma = use_splitk ? ldw : (!c_tma ? 0 : N / (16 / eb) * (16 / eb));
    if (ldg) {
        // the plain-load GEMM: row-class windows of A and B, and C's map
        if ((st = encode_windows(L.win.a, A, K, M, lda, 16, &p.win_delta_a)) ||
            (st = encode_windows(L.win.b, B, K, N, ldb, static_cast<uint32_t>(b_rows / 8), &p.win_delta_b)))
            return st;
        if (use_splitk) {
            if ((st = encode_splitk_workspace(&L.mapC, ws, ldw, M, pl.splits))) return st;
        } else if (c_tma) {
            TiledDesc dc{out_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C,
                         {static_cast<uint64_t>(n_tma > 0 ? n_tma : N), static_cast<uint64_t>(M)},
                         {static_cast<uint64_t>(ldc) * eb}, {128 / eb, 32}, CU_TENSOR_MAP_SWIZZLE_128B};
            if ((st = encode_tiled(&L.mapC, dc))) return st;
        }
    } else {
        TiledDesc da{CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(A),
                     {static_cast<uint64_t>(K), static_cast<uint64_t>(M)}, {static_cast<uint64_t>(lda) * 2},
                     {64, 128}, CU_TENSOR_MAP_SWIZZLE_128B};
        TiledDesc db{CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(B),
                     {static_cast<uint64_t>(K), static_cast<uint64_t>(N)}, {static_cast<uint64_t>(ldb) * 2},
                     {64, static_cast<uint32_t>(b_rows)}, CU_TENSOR_MAP_SWIZZLE_128B};
        if ((st = encode_tiled(&L.mapA, da)) || (st = encode_tiled(&L.mapB, db))) return st;
        L.mapBh = L.mapB;
        if (p.tail_units > 0) {
            // the narrow tail's units: a half or a quarter of each CTA's B rows
            TiledDesc dbh = db;
            dbh.box[1] = static_cast<uint32_t>(b_rows / p.tail_parts);
            if ((st = encode_tiled(&L.mapBh, dbh))) return st;
        }
        if (use_splitk) {
            if ((st = encode_splitk_workspace(&L.mapC, ws, ldw, M, pl.splits))) return st;
        } else if (c_tma) {
            TiledDesc dc{out_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C,
                         {static_cast<uint64_t>(n_tma > 0 ? n_tma : N), static_cast<uint64_t>(M)},
                         {static_cast<uint64_t>(ldc) * eb}, {128 / eb, 32}, CU_TENSOR_MAP_SWIZZLE_128B};
            if ((st = encode_tiled(&L.mapC, dc))) return st;
        } else {
            // n_tma = 0: the epilogue writes all of C with plain stores and
            // never uses its map, which stays a valid copy of A's.
            L.mapC = L.mapA;
        }
    }
    p.A = static_cast<const uint16_t*>(A);
    p.B = static_cast<const uint16_t*>(B);
    p.lda = lda;
    p.ldb = ldb;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.m_tiles = static_cast<int>(pl.m_tiles);
    p.n_tiles = static_cast<int>(pl.n_tiles);
    p.k_blocks = static_cast<int>(pl.k_blocks);
    p.splits = use_splitk ? pl.splits : 1;
    p.kb_per_split = use_splitk ? kps : p.k_blocks;
    p.group_m = group_m_for(opts, pl.m_tiles, pl.atom);
    l2_hints_for(pl.l2_hint, &p.l2_a, &p.l2_b);
    p.n_tma = static_cast<int>(n_tma);
    p.trace = opts ? reinterpret_cast<unsigned long long*>(opts->trace) : nullptr;
    p.events = opts ? reinterpret_cast<unsigned long long*>(opts->events) : nullptr;
    p.C = use_splitk ? ws : C;
    p.ldc_bytes = use_splitk ? ldw * 4 : ldc * eb;
    p.wait = WaitCtl{dev->status, t_selftest_limit_ns ? t_selftest_limit_ns : wait_limit_ns()};
    p.withhold_first_arrival = t_selftest_withhold;
    p.skip_commit = t_selftest_skip_commit;
    p.proto = opts ? opts->protocol : nullptr;
    if (use_splitk) {
        const KernelEntry* k = find_kernel(KernelKey{pl.atom, pl.tile_n, pl.pipe_depth, 1, 0, ldg ? 1 : 0, 1});
        L.grid = pl.grid;
        L.stream = s;
        set_divisors(p);
        cudaError_t e = k->launch(L);
        if (e != cudaSuccess) return cuda_fail(e);
        e = launch_splitk_reduce(static_cast<const float*>(ws), C, static_cast<int>(M), static_cast<int>(N), ldw,
                                 ldc, pl.splits, out_f32, dev->sm_count, s);
        if (e != cudaSuccess) return cuda_fail(e);
        pl.out_f32 = out_f32;
        t_last_plan = pl;
        return TP_OK;
    }
    st = launch_plan(pl, L, s);
    if (st == TP_OK) t_last_plan = pl;
    return st;
}

}  // namespace

extern "C" {

int tp_gemm_bf16_ex(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int64_t lda,
                    int64_t ldb, int64_t ldc, int out_f32, const tp_gemm_opts* opts, void* stream)
{
    return gemm_impl(A, B, C, M, N, K, lda, ldb, ldc, out_f32, opts, 0, 0, nullptr, 0, stream);
}

int tp_gemm_splitk_workspace_bytes(int64_t M, int64_t N, int splits, int64_t* bytes)
{
    if (!bytes || M < 0 || N < 0 || splits < 1) return TP_ERR_INVALID_ARG;
    *bytes = static_cast<int64_t>(splits) * M * splitk_ldw(N) * 4;
    return TP_OK;
}

int tp_gemm_bf16_splitk(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int64_t lda,
                        int64_t ldb, int64_t ldc, int out_f32, int splits, void* workspace, int64_t workspace_bytes,
                        const tp_gemm_opts* opts, void* stream)
{
    return gemm_impl(A, B, C, M, N, K, lda, ldb, ldc, out_f32, opts, 1, splits, workspace, workspace_bytes, stream);
}

int tp_gemm_bf16(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int64_t lda,
                 int64_t ldb, int64_t ldc, void* stream)
{
    return tp_gemm_bf16_ex(A, B, C, M, N, K, lda, ldb, ldc, 0, nullptr, stream);
}

int tp_gemm_bf16_f32(const void* A, const void* B, float* C, int64_t M, int64_t N, int64_t K, int64_t lda,
                     int64_t ldb, int64_t ldc, void* stream)
{
    return tp_gemm_bf16_ex(A, B, C, M, N, K, lda, ldb, ldc, 1, nullptr, stream);
}

int tp_conv2d_fprop_bf16_ex(const void* x, const void* w, void* y, int64_t N, int64_t H, int64_t W, int64_t C,
                            int64_t K, int64_t R, int64_t S, int64_t stride, int64_t pad, int out_f32,
                            const tp_gemm_opts* opts, void* stream)
{
    out_f32 = out_f32 ? 1 : 0;
    tp_plan pl;
    std::memset(&pl, 0, sizeof(pl));
    t_last_plan = pl;
    if (N < 0 || H < 0 || W < 0 || C < 0 || K < 0 || R < 1 || S < 1 || stride < 1 || pad < 0)
        return TP_ERR_INVALID_ARG;
    const int64_t hp = H + 2 * pad - R, wp = W + 2 * pad - S;
    if (hp < 0 || wp < 0) return TP_ERR_INVALID_ARG;
    const int64_t P = hp / stride + 1, Q = wp / stride + 1;
    const int64_t M = N * P * Q;
    if (M == 0 || K == 0) return TP_OK;
    if (!y || (C > 0 && (!x || !w))) return TP_ERR_INVALID_ARG;
    DeviceState* dev = nullptr;
    int st = device_state(&dev);
    if (st) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (C == 0) {
        pl.path = TP_PATH_ZERO_FILL;
        cudaError_t e = launch_zero_fill(y, M, K, K, out_f32 ? 4 : 2, s);
        t_last_plan = pl;
        return e == cudaSuccess ? TP_OK : cuda_fail(e);
    }
    const int eb_out = out_f32 ? 4 : 2;
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w)) & 1u ||
        reinterpret_cast<uintptr_t>(y) % eb_out)
        return TP_ERR_INVALID_ARG;
    if (M > INT32_MAX || N * H * W > INT32_MAX || R * S > INT32_MAX / 64 || K > INT32_MAX)
        return TP_ERR_UNSUPPORTED;
    // im2col TMA limits (cuTensorMapEncodeIm2col: rank-4 corners in
    // [-128, 127], traversal strides <= 8) and 16-byte byte strides;
    // otherwise the plain-load producer gathers the same tiles.
    int ldg = (C % 8 || !aligned16(x) || !aligned16(w) || stride > 8 || R > 32 || S > 32 || pad > 127) ? kLdgPlain
                                                                                                      : kLdgNone;
    // A stride-1 convolution whose output is the input's size reads, for a
    // tap, the pixels of a tile's outputs shifted by one offset: a run of
    // consecutive pixels, which row-class windows can load.
    if (ldg && stride == 1 && P == H && Q == W) ldg = kLdgConvWin;
    // y rows of whole 16-byte granules at a 16-byte aligned base go out by
    // TMA; otherwise the epilogue writes y with plain stores.
    const bool y_tma = aligned16(y) && (K * eb_out) % 16 == 0;
    const int64_t cblocks = cdiv(C, 64);
    if (opts && (opts->l2_hint < 0 || opts->l2_hint > 7)) return TP_ERR_INVALID_ARG;
    st = plan_mainloop(M, K, R * S * cblocks, out_f32, 1, ldg, opts, dev->sm_count, &pl);
    if (st) return st;
    const int cg = pl.atom;
    const int b_rows = pl.tile_n / cg;
    GemmLaunch L;
    std::memset(&L, 0, sizeof(L));
    GemmParams& p = L.params;
    // the narrow tail (2-SM, N = 256) before the maps: it sets their box
    if (!(opts && opts->no_tail)) set_narrow_tail(pl, p, opts, dev->sm_count);
    if (ldg == kLdgConvWin) {
        // rows: pixels (C elements each) and filters (R * S * C elements);
        // 80-element boxes, since a filter's K blocks start anywhere
        if ((st = encode_windows(L.win.a, x, C, N * H * W, C, 16, &p.win_delta_a, 80)) ||
            (st = encode_windows(L.win.b, w, R * S * C, K, R * S * C, static_cast<uint32_t>(b_rows / 8),
                                 &p.win_delta_b, 80)))
            return st;
        if (y_tma) {
            const uint32_t eb = out_f32 ? 4 : 2;
            TiledDesc dy{out_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, y,
                         {static_cast<uint64_t>(K), static_cast<uint64_t>(M)}, {static_cast<uint64_t>(K) * eb},
                         {128 / eb, 32}, CU_TENSOR_MAP_SWIZZLE_128B};
            if ((st = encode_tiled(&L.mapC, dy))) return st;
        }
    }
    if (!ldg) {
        Im2colDesc dx{};
        dx.dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        dx.base = const_cast<void*>(x);
        dx.dims[0] = static_cast<uint64_t>(C);
        dx.dims[1] = static_cast<uint64_t>(W);
        dx.dims[2] = static_cast<uint64_t>(H);
        dx.dims[3] = static_cast<uint64_t>(N);
        dx.strides_bytes[0] = static_cast<uint64_t>(C) * 2;
        dx.strides_bytes[1] = static_cast<uint64_t>(W * C) * 2;
        dx.strides_bytes[2] = static_cast<uint64_t>(H * W * C) * 2;
        // Bounding box of the filter window's first tap: from -pad to
        // (extent - 1) + pad - (filter - 1), the positions output pixels start at.
        dx.lower[0] = static_cast<int>(-pad);
        dx.lower[1] = static_cast<int>(-pad);
        dx.upper[0] = static_cast<int>(pad - (S - 1));
        dx.upper[1] = static_cast<int>(pad - (R - 1));
        dx.channels = 64;
        dx.pixels = 128;
        dx.elem_strides[0] = 1;
        dx.elem_strides[1] = static_cast<uint32_t>(stride);
        dx.elem_strides[2] = static_cast<uint32_t>(stride);
        dx.elem_strides[3] = 1;
        dx.swizzle = CU_TENSOR_MAP_SWIZZLE_128B;
        if (dx.upper[0] < -128 || dx.upper[1] < -128) return TP_ERR_UNSUPPORTED;
        TiledDesc dw{CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(w),
                     {static_cast<uint64_t>(C), static_cast<uint64_t>(R * S), static_cast<uint64_t>(K)},
                     {static_cast<uint64_t>(C) * 2, static_cast<uint64_t>(R * S * C) * 2},
                     {64, 1, static_cast<uint32_t>(b_rows)}, CU_TENSOR_MAP_SWIZZLE_128B};
        const uint32_t eb = out_f32 ? 4 : 2;
        TiledDesc dy{out_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, y,
                     {static_cast<uint64_t>(K), static_cast<uint64_t>(M)}, {static_cast<uint64_t>(K) * eb},
                     {128 / eb, 32}, CU_TENSOR_MAP_SWIZZLE_128B};
        if ((st = encode_im2col(&L.mapA, dx)) || (st = encode_tiled(&L.mapB, dw))) return st;
        L.mapBh = L.mapB;
        if (p.tail_units > 0) {
            TiledDesc dwh = dw;
            dwh.box[2] = static_cast<uint32_t>(b_rows / p.tail_parts);
            if ((st = encode_tiled(&L.mapBh, dwh))) return st;
        }
        if (y_tma) {
            if ((st = encode_tiled(&L.mapC, dy))) return st;
        } else {
            L.mapC = L.mapB;  // never stored through (n_tma = 0)
        }
    }
    p.A = static_cast<const uint16_t*>(x);
    p.B = static_cast<const uint16_t*>(w);
    p.conv_H = static_cast<int>(H);
    p.conv_W = static_cast<int>(W);
    p.conv_C = static_cast<int>(C);
    p.conv_R = static_cast<int>(R);
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(K);
    p.K = static_cast<int>(R * S * C);
    p.m_tiles = static_cast<int>(pl.m_tiles);
    p.n_tiles = static_cast<int>(pl.n_tiles);
    p.k_blocks = static_cast<int>(pl.k_blocks);
    p.splits = 1;
    p.kb_per_split = p.k_blocks;
    p.group_m = group_m_for(opts, pl.m_tiles, pl.atom);
    pl.l2_hint = l2_mode_for(opts, pl.m_tiles, pl.n_tiles, 0.0, 0.0, false);
    l2_hints_for(pl.l2_hint, &p.l2_a, &p.l2_b);
    p.conv_P = static_cast<int>(P);
    p.conv_Q = static_cast<int>(Q);
    p.conv_stride = static_cast<int>(stride);
    p.conv_pad = static_cast<int>(pad);
    p.conv_S = static_cast<int>(S);
    p.conv_cblocks = static_cast<int>(cblocks);
    // TMA stores (rows of whole 16-byte granules) unless the cp.async form runs
    p.n_tma = (ldg == kLdgPlain || !y_tma) ? 0 : static_cast<int>(K);
    p.trace = opts ? reinterpret_cast<unsigned long long*>(opts->trace) : nullptr;
    p.events = opts ? reinterpret_cast<unsigned long long*>(opts->events) : nullptr;
    p.proto = opts ? opts->protocol : nullptr;
    p.C = y;
    p.ldc_bytes = K * eb_out;
    p.wait = WaitCtl{dev->status, wait_limit_ns()};
    st = launch_plan(pl, L, s, ldg ? ldg : kLdgPlain);
    if (st == TP_OK) t_last_plan = pl;
    return st;
}

int tp_conv2d_fprop_bf16(const void* x, const void* w, void* y, int64_t N, int64_t H, int64_t W, int64_t C,
                         int64_t K, int64_t R, int64_t S, int64_t stride, int64_t pad, void* stream)
{
    return tp_conv2d_fprop_bf16_ex(x, w, y, N, H, W, C, K, R, S, stride, pad, 0, nullptr, stream);
}

int tp_tma_copy_2d_ex(const void* src, void* dst, int64_t rows, int64_t cols, int64_t ld,
                      const tp_copy_opts* o, void* stream)
{
    tp_plan pl;
    std::memset(&pl, 0, sizeof(pl));
    t_last_plan = pl;
    if (rows < 0 || cols < 0 || ld < cols) return TP_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return TP_OK;
    if (!src || !dst) return TP_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 1u) return TP_ERR_INVALID_ARG;
    DeviceState* dev = nullptr;
    int st = device_state(&dev);
    if (st) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int box_cols = o && o->box_cols ? o->box_cols : 64;
    const int box_rows = o && o->box_rows ? o->box_rows : 128;
    // Defaults from a sweep on GB300 (1 GiB): 6 stages of 128 x 64 tiles,
    // one CTA per SM, 6.77 TB/s (8 stages: 6.23 TB/s).
    const int stages = o && o->stages ? o->stages : 6;
    const int per_sm = o && o->ctas_per_sm ? o->ctas_per_sm : 1;
    if (box_cols < 8 || box_cols > 256 || (box_cols * 2) % 16 || box_rows < 1 || box_rows > 256 || per_sm < 1)
        return TP_ERR_INVALID_ARG;
    const bool tma_ok = aligned16(src) && aligned16(dst) && (ld * 2) % 16 == 0 && rows * cols * 2 >= 65536 &&
                        rows <= INT32_MAX && cols <= INT32_MAX && !(o && o->force_vec);
    if (!tma_ok) {
        cudaError_t e = launch_vec_copy(src, dst, rows, cols, ld, dev->sm_count, s);
        if (e != cudaSuccess) return cuda_fail(e);
        pl.path = TP_PATH_VEC_COPY;
        t_last_plan = pl;
        return TP_OK;
    }
    // TMA stores write whole 16-byte granules of a row: the TMA ring copies
    // the first cols_tma columns, the ragged tail goes through the
    // vectorized path.
    const int64_t cols_tma = cols / 8 * 8;
    if (cols_tma == 0) {
        cudaError_t e = launch_vec_copy(src, dst, rows, cols, ld, dev->sm_count, s);
        if (e != cudaSuccess) return cuda_fail(e);
        pl.path = TP_PATH_VEC_COPY;
        t_last_plan = pl;
        return TP_OK;
    }
    const uint32_t tile_bytes = static_cast<uint32_t>(box_cols * box_rows * 2);
    const int smem = copy_smem_bytes(stages, tile_bytes);
    if (smem > kMaxSmemPerCta) return TP_ERR_SMEM_BUDGET;
    TiledDesc d{CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(src),
                {static_cast<uint64_t>(cols_tma), static_cast<uint64_t>(rows)}, {static_cast<uint64_t>(ld) * 2},
                {static_cast<uint32_t>(box_cols), static_cast<uint32_t>(box_rows)}, CU_TENSOR_MAP_SWIZZLE_NONE};
    CUtensorMap ms, md;
    if ((st = encode_tiled(&ms, d))) return st;
    d.base = dst;
    if ((st = encode_tiled(&md, d))) return st;
    CopyParams p{};
    p.tiles_x = static_cast<int>(cdiv(cols_tma, box_cols));
    p.tiles_y = static_cast<int>(cdiv(rows, box_rows));
    p.box_cols = box_cols;
    p.box_rows = box_rows;
    p.tile_bytes = tile_bytes;
    p.wait = WaitCtl{dev->status, wait_limit_ns()};
    const int64_t tiles = static_cast<int64_t>(p.tiles_x) * p.tiles_y;
    if (tiles > INT32_MAX) return TP_ERR_UNSUPPORTED;
    int64_t grid = static_cast<int64_t>(dev->sm_count) * per_sm;
    if (grid > tiles) grid = tiles;
    cudaError_t e = launch_tma_copy_any(stages, ms, md, p, static_cast<int>(grid), s);
    if (e == cudaErrorInvalidValue && stages != 2 && stages != 3 && stages != 4 && stages != 6 && stages != 8 &&
        stages != 12)
        return TP_ERR_INVALID_ARG;
    if (e != cudaSuccess) return cuda_fail(e);
    if (cols_tma < cols) {
        e = launch_vec_copy(static_cast<const uint16_t*>(src) + cols_tma, static_cast<uint16_t*>(dst) + cols_tma,
                            rows, cols - cols_tma, ld, dev->sm_count, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    pl.path = TP_PATH_TMA_COPY;
    pl.pipe_depth = stages;
    pl.grid = static_cast<int>(grid);
    pl.cluster = 1;
    pl.smem_bytes = smem;
    pl.m_tiles = p.tiles_y;
    pl.n_tiles = p.tiles_x;
    t_last_plan = pl;
    return TP_OK;
}

int tp_tma_copy_2d(const void* src, void* dst, int64_t rows, int64_t cols, int64_t ld, void* stream)
{
    return tp_tma_copy_2d_ex(src, dst, rows, cols, ld, nullptr, stream);
}

int tp_tma_read_2d(const void* src, int64_t rows, int64_t cols, int64_t ld, const tp_copy_opts* o, void* stream)
{
    tp_plan pl;
    std::memset(&pl, 0, sizeof(pl));
    t_last_plan = pl;
    if (rows < 0 || cols < 0 || ld < cols) return TP_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return TP_OK;
    if (!src) return TP_ERR_INVALID_ARG;
    DeviceState* dev = nullptr;
    int st = device_state(&dev);
    if (st) return st;
    // Defaults from a sweep on GB300 (256 MiB after a 256 MiB write flush):
    // 128 x 64 tiles, 8 stages, one CTA per SM, 57 us (4.7 TB/s); 42.5 us
    // back to back.
    const int box_cols = o && o->box_cols ? o->box_cols : 64;
    const int box_rows = o && o->box_rows ? o->box_rows : 128;
    const int stages = o && o->stages ? o->stages : 8;
    const int per_sm = o && o->ctas_per_sm ? o->ctas_per_sm : 1;
    if (box_cols < 8 || box_cols > 256 || (box_cols * 2) % 16 || box_rows < 1 || box_rows > 256 || per_sm < 1 ||
        (stages != 2 && stages != 4 && stages != 8 && stages != 12))
        return TP_ERR_INVALID_ARG;
    // TMA only: rows of whole 16-byte granules at a 16-byte aligned base.
    if (!aligned16(src) || (ld * 2) % 16 || cols % 8 || rows > INT32_MAX || cols > INT32_MAX)
        return TP_ERR_UNSUPPORTED;
    const uint32_t tile_bytes = static_cast<uint32_t>(box_cols * box_rows * 2);
    const int smem = copy_smem_bytes(stages, tile_bytes);
    if (smem > kMaxSmemPerCta) return TP_ERR_SMEM_BUDGET;
    TiledDesc d{CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(src),
                {static_cast<uint64_t>(cols), static_cast<uint64_t>(rows)}, {static_cast<uint64_t>(ld) * 2},
                {static_cast<uint32_t>(box_cols), static_cast<uint32_t>(box_rows)}, CU_TENSOR_MAP_SWIZZLE_NONE};
    CUtensorMap ms;
    if ((st = encode_tiled(&ms, d))) return st;
    CopyParams p{};
    p.tiles_x = static_cast<int>(cdiv(cols, box_cols));
    p.tiles_y = static_cast<int>(cdiv(rows, box_rows));
    p.box_cols = box_cols;
    p.box_rows = box_rows;
    p.tile_bytes = tile_bytes;
    p.wait = WaitCtl{dev->status, wait_limit_ns()};
    const int64_t tiles = static_cast<int64_t>(p.tiles_x) * p.tiles_y;
    if (tiles > INT32_MAX) return TP_ERR_UNSUPPORTED;
    int64_t grid = static_cast<int64_t>(dev->sm_count) * per_sm;
    if (grid > tiles) grid = tiles;
    cudaError_t e = launch_tma_read_any(stages, ms, p, static_cast<int>(grid), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    pl.path = TP_PATH_TMA_READ;
    pl.pipe_depth = stages;
    pl.grid = static_cast<int>(grid);
    pl.cluster = 1;
    pl.smem_bytes = smem;
    pl.m_tiles = p.tiles_y;
    pl.n_tiles = p.tiles_x;
    t_last_plan = pl;
    return TP_OK;
}

int tp_tma_transpose_2d_ex(const void* src, void* dst, int64_t rows, int64_t cols, int64_t ld_src, int64_t ld_dst,
                           const tp_copy_opts* o, void* stream)
{
    tp_plan pl;
    std::memset(&pl, 0, sizeof(pl));
    t_last_plan = pl;
    if (rows < 0 || cols < 0 || ld_src < cols || ld_dst < rows) return TP_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return TP_OK;
    if (!src || !dst) return TP_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 1u) return TP_ERR_INVALID_ARG;
    DeviceState* dev = nullptr;
    int st = device_state(&dev);
    if (st) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // Defaults from a sweep on GB300 (1 GiB): 8 stages, two one-warp CTAs per
    // SM, 6.50 TB/s (4 stages x 4 CTAs: 5.87 TB/s).
    const int stages = o && o->stages ? o->stages : 8;
    const int per_sm = o && o->ctas_per_sm ? o->ctas_per_sm : 2;
    if (stages != 2 && stages != 4 && stages != 6 && stages != 8) return TP_ERR_INVALID_ARG;
    if (per_sm < 1) return TP_ERR_INVALID_ARG;
    // TMA stores write whole 16-byte granules of a destination row: the TMA
    // path covers destination columns (source rows) 0..rows_tma-1, the rest
    // goes through the shared-memory tile transpose.
    const int64_t rows_tma = rows / 8 * 8;
    const bool tma_ok = aligned16(src) && aligned16(dst) && (ld_src * 2) % 16 == 0 && (ld_dst * 2) % 16 == 0 &&
                        rows * cols * 2 >= 65536 && rows_tma > 0 && rows <= INT32_MAX && cols <= INT32_MAX &&
                        !(o && o->force_vec);
    if (!tma_ok) {
        cudaError_t e = launch_vec_transpose(src, dst, 0, rows, cols, ld_src, ld_dst, dev->sm_count, s);
        if (e != cudaSuccess) return cuda_fail(e);
        pl.path = TP_PATH_VEC_TRANSPOSE;
        t_last_plan = pl;
        return TP_OK;
    }
    const int smem = transpose_smem_bytes(stages);
    if (smem > kMaxSmemPerCta) return TP_ERR_SMEM_BUDGET;
    TiledDesc ds{CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(src),
                 {static_cast<uint64_t>(cols), static_cast<uint64_t>(rows)}, {static_cast<uint64_t>(ld_src) * 2},
                 {64, 64}, CU_TENSOR_MAP_SWIZZLE_128B};
    TiledDesc dd{CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, dst,
                 {static_cast<uint64_t>(rows_tma), static_cast<uint64_t>(cols)}, {static_cast<uint64_t>(ld_dst) * 2},
                 {64, 64}, CU_TENSOR_MAP_SWIZZLE_128B};
    CUtensorMap ms, md;
    if ((st = encode_tiled(&ms, ds)) || (st = encode_tiled(&md, dd))) return st;
    const int64_t tiles_x = cdiv(cols, 64), tiles_y = cdiv(rows_tma, 64);
    if (tiles_x * tiles_y > INT32_MAX) return TP_ERR_UNSUPPORTED;
    int64_t grid = static_cast<int64_t>(dev->sm_count) * per_sm;
    if (grid > tiles_x * tiles_y) grid = tiles_x * tiles_y;
    cudaError_t e = launch_tma_transpose(stages, ms, md, static_cast<int>(tiles_x), static_cast<int>(tiles_y),
                                         WaitCtl{dev->status, wait_limit_ns()}, static_cast<int>(grid), s);
    if (e != cudaSuccess) return cuda_fail(e);
    if (rows_tma < rows) {
        e = launch_vec_transpose(src, dst, rows_tma, rows - rows_tma, cols, ld_src, ld_dst, dev->sm_count, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    pl.path = TP_PATH_TMA_TRANSPOSE;
    pl.pipe_depth = stages;
    pl.grid = static_cast<int>(grid);
    pl.cluster = 1;
    pl.smem_bytes = smem;
    pl.m_tiles = tiles_y;
    pl.n_tiles = tiles_x;
    pl.splits = 1;
    t_last_plan = pl;
    return TP_OK;
}

int tp_tma_transpose_2d(const void* src, void* dst, int64_t rows, int64_t cols, int64_t ld_src, int64_t ld_dst,
                        void* stream)
{
    return tp_tma_transpose_2d_ex(src, dst, rows, cols, ld_src, ld_dst, nullptr, stream);
}

int tp_device_status_detail(void* stream, int* site, int* block, int* thread)
{
    DeviceState* dev = nullptr;
    int st = device_state(&dev);
    if (st) return st;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    DevStatus h{};
    e = cudaMemcpy(&h, dev->status, sizeof(h), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    if (h.code != 0) {
        DevStatus z{};
        e = cudaMemcpy(dev->status, &z, sizeof(z), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (site) *site = h.site;
    if (block) *block = h.block;
    if (thread) *thread = h.thread;
    return h.code;
}

int tp_device_status(void* stream) { return tp_device_status_detail(stream, nullptr, nullptr, nullptr); }

int tp_probe_fma_latency(int kind, int chain, double seed, double* result, double* cycles_per_link, void* stream)
{
    if ((kind != 0 && kind != 1) || chain < 64 || chain % 64 || chain > (1 << 26) || !result || !cycles_per_link)
        return TP_ERR_INVALID_ARG;
    DeviceState* dev = nullptr;
    int st = device_state(&dev);
    if (st) return st;
    long long cycles = 0;
    cudaError_t e = run_fma_probe(kind, seed, chain / 64, static_cast<cudaStream_t>(stream), result, &cycles);
    if (e != cudaSuccess) return cuda_fail(e);
    *cycles_per_link = static_cast<double>(cycles) / static_cast<double>(chain);
    return TP_OK;
}

int tp_selftest_mainloop_withheld_arrival(const void* A, const void* B, float* C, int64_t M, int64_t N,
                                          int64_t K, uint32_t limit_ms, void* stream)
{
    if (limit_ms == 0 || limit_ms > 10000 || M > 4096 || N > 4096 || K < 64 || K > 4096) return TP_ERR_INVALID_ARG;
    tp_gemm_opts o{};
    o.atom = 1;
    o.tile_n = 128;
    t_selftest_withhold = 1;
    t_selftest_limit_ns = static_cast<uint64_t>(limit_ms) * 1000000ull;
    const int st = gemm_impl(A, B, C, M, N, K, K, K, N, 1, &o, 0, 0, nullptr, 0, stream);
    t_selftest_withhold = 0;
    t_selftest_limit_ns = 0;
    return st;
}

int tp_selftest_mainloop_skipped_commit(const void* A, const void* B, float* C, int64_t M, int64_t N, int64_t K,
                                        int which, int atom, uint32_t limit_ms, void* stream)
{
    if (limit_ms == 0 || limit_ms > 10000 || M > 4096 || N > 4096 || K < 64 || K > 4096) return TP_ERR_INVALID_ARG;
    if ((which != 1 && which != 2) || (atom != 1 && atom != 2)) return TP_ERR_INVALID_ARG;
    tp_gemm_opts o{};
    o.atom = atom;
    o.tile_n = 128;
    o.no_tail = 1;
    t_selftest_skip_commit = which;
    t_selftest_limit_ns = static_cast<uint64_t>(limit_ms) * 1000000ull;
    const int st = gemm_impl(A, B, C, M, N, K, K, K, N, 1, &o, 0, 0, nullptr, 0, stream);
    t_selftest_skip_commit = 0;
    t_selftest_limit_ns = 0;
    return st;
}

int tp_selftest_wait_timeout(uint32_t limit_us, void* stream)
{
    DeviceState* dev = nullptr;
    int st = device_state(&dev);
    if (st) return st;
    if (limit_us == 0 || limit_us > 10u * 1000u * 1000u) return TP_ERR_INVALID_ARG;
    WaitCtl w{dev->status, static_cast<uint64_t>(limit_us) * 1000ull};
    cudaError_t e = launch_wait_selftest(w, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TP_OK : cuda_fail(e);
}

// ------------------------------------------- split-K without allocation ---
//
// Some callers may not allocate device memory while they run: code that lives
// inside a fixed device-memory budget reserved up front by another allocator,
// or code where cudaMalloc's implicit device-wide synchronization is not
// allowed. tp_gemm_bf16_splitk_noalloc serves them with a workspace that is a
// fixed array inside the library instead of a caller buffer.

}  // extern "C"

namespace {

constexpr int64_t kNoallocWorkspaceBytes = 32ll << 20;  // 32 MiB per GPU

// The split-K partial sums of tp_gemm_bf16_splitk_noalloc. Every GPU that
// loads the library holds this array until the process exits. In host code
// the name is only a host-side stand-in; its device address comes from
// cudaGetSymbolAddress.
static __device__ __align__(256) float g_noalloc_workspace[kNoallocWorkspaceBytes / sizeof(float)];

float* g_noalloc_ptr[kMaxDevices];
std::mutex g_noalloc_mu;

// Once per device, with that device current: the array's device address.
int noalloc_workspace(float** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return TP_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_workspace);
        if (e != cudaSuccess) return cuda_fail(e);
        g_noalloc_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_noalloc_ptr[dev];
    return TP_OK;
}

}  // namespace

extern "C" {

int tp_gemm_bf16_host(const void* A_host, const void* B_host, void* C_host, int64_t M, int64_t N, int64_t K,
                      int64_t lda, int64_t ldb, int64_t ldc, int out_f32, void* dA, void* dB, void* dC,
                      const tp_gemm_opts* opts, void* stream)
{
    std::memset(&t_last_plan, 0, sizeof(t_last_plan));
    if (M < 0 || N < 0 || K < 0) return TP_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return TP_OK;
    if (lda < K || ldb < K || ldc < N) return TP_ERR_INVALID_ARG;
    if (!C_host || !dC || (K > 0 && (!A_host || !B_host || !dA || !dB))) return TP_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t eb = out_f32 ? 4 : 2;
    cudaError_t e = cudaSuccess;
    if (K > 0) {
        e = cudaMemcpy2DAsync(dA, static_cast<size_t>(lda) * 2, A_host, static_cast<size_t>(lda) * 2,
                              static_cast<size_t>(K) * 2, static_cast<size_t>(M), cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess)
            e = cudaMemcpy2DAsync(dB, static_cast<size_t>(ldb) * 2, B_host, static_cast<size_t>(ldb) * 2,
                                  static_cast<size_t>(K) * 2, static_cast<size_t>(N), cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    const int st = gemm_impl(dA, dB, dC, M, N, K, lda, ldb, ldc, out_f32, opts, 0, 0, nullptr, 0, stream);
    if (st) return st;
    e = cudaMemcpy2DAsync(C_host, static_cast<size_t>(ldc) * eb, dC, static_cast<size_t>(ldc) * eb,
                          static_cast<size_t>(N) * eb, static_cast<size_t>(M), cudaMemcpyDeviceToHost, s);
    return e == cudaSuccess ? TP_OK : cuda_fail(e);
}

int tp_gemm_bf16_splitk_noalloc(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                                int64_t lda, int64_t ldb, int64_t ldc, int out_f32, int splits, void* stream)
{
    if (M < 0 || N < 0 || K < 0 || splits < 0) return TP_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return TP_OK;
    if (splits > 0 && K > 0) {
        int sp = splits, kps = 0;
        normalize_splits(cdiv(K, 64), &sp, &kps);
        if (sp > 1 && static_cast<int64_t>(sp) * M * splitk_ldw(N) * 4 > kNoallocWorkspaceBytes)
            return TP_ERR_WORKSPACE_LIMIT;
    }
    float* ws = nullptr;
    const int st = noalloc_workspace(&ws);
    if (st) return st;
    return gemm_impl(A, B, C, M, N, K, lda, ldb, ldc, out_f32, nullptr, 1, splits, ws, kNoallocWorkspaceBytes,
                     stream);
}

int64_t tp_gemm_splitk_noalloc_capacity(void) { return kNoallocWorkspaceBytes; }

}  // extern "C"
