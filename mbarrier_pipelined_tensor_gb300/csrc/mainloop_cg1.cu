// 1-SM atom variants of the mainloop: the PIPE_DEPTH sweep at MMA N = 128 and
// 256 with bf16 output, plus the fp32-output variants at the deepest ring.
#include "gemm_kernel.cuh"

namespace tp {

static const KernelEntry k_table[] = {
    mainloop_entry<1, 128, 2, false, false>(),
    mainloop_entry<1, 128, 3, false, false>(),
    mainloop_entry<1, 128, 4, false, false>(),
    mainloop_entry<1, 128, 5, false, false>(),
    mainloop_entry<1, 128, 6, false, false>(),
    mainloop_entry<1, 256, 2, false, false>(),
    mainloop_entry<1, 256, 3, false, false>(),
    mainloop_entry<1, 256, 4, false, false>(),
    mainloop_entry<1, 128, 6, true, false>(),
    mainloop_entry<1, 256, 4, true, false>(),
};

const KernelEntry* table_mainloop_cg1(int* n)
{
    *n = static_cast<int>(sizeof(k_table) / sizeof(k_table[0]));
    return k_table;
}

}  // namespace tp
