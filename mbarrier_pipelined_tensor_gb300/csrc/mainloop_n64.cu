// 1-SM atom at MMA N = 64: 128 x 64 output tiles. Against N = 128 it doubles
// the tile count of a small problem, so that more SMs stream its operands
// (each CTA then loads 24 KiB per k-block instead of 32 KiB), and it has the
// deepest ring of all variants (8 stages of 24 KiB). The PIPE_DEPTH sweep with
// bf16 output, and the fp32, conv and split-K forms at the deepest ring.
#include "gemm_kernel.cuh"

namespace tp {

static const KernelEntry k_table[] = {
    mainloop_entry<1, 64, 2, false, false>(),
    mainloop_entry<1, 64, 3, false, false>(),
    mainloop_entry<1, 64, 4, false, false>(),
    mainloop_entry<1, 64, 5, false, false>(),
    mainloop_entry<1, 64, 6, false, false>(),
    mainloop_entry<1, 64, 7, false, false>(),
    mainloop_entry<1, 64, 8, false, false>(),
    mainloop_entry<1, 64, 8, true, false>(),
    mainloop_entry<1, 64, 8, false, true>(),
    mainloop_entry<1, 64, 8, true, true>(),
    mainloop_entry<1, 64, 8, true, false, false, true>(),
};

const KernelEntry* table_mainloop_n64(int* n)
{
    *n = static_cast<int>(sizeof(k_table) / sizeof(k_table[0]));
    return k_table;
}

}  // namespace tp
