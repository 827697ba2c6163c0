// Plain-load producer variants of the mainloop (operands TMA cannot
// describe): 1-SM atom, MMA N = 128, GEMM (row-class windows, 2 ring
// stages; also with split-K partials), conv (cp.async windows, 3; row-class
// windows for stride-1 same-size convolutions, 2), bf16 and fp32 outputs.
#include "gemm_kernel.cuh"

namespace tp {

static const KernelEntry k_table[] = {
    mainloop_entry<1, 128, 2, false, false, true>(),
    mainloop_entry<1, 128, 2, true, false, true>(),
    mainloop_entry<1, 128, 3, false, true, true>(),
    mainloop_entry<1, 128, 3, true, true, true>(),
    mainloop_entry<1, 128, 2, true, false, true, true>(),  // split-K partials
    mainloop_entry<1, 128, 2, false, true, kLdgConvWin>(),
    mainloop_entry<1, 128, 2, true, true, kLdgConvWin>(),
};

const KernelEntry* table_mainloop_fallback(int* n)
{
    *n = static_cast<int>(sizeof(k_table) / sizeof(k_table[0]));
    return k_table;
}

}  // namespace tp
