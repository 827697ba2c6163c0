// 2-SM atom variants of the mainloop (cluster of two CTAs, cta_group::2):
// the PIPE_DEPTH sweep at pair tile N = 128 and 256 with bf16 output, plus
// the fp32-output variants at the deepest ring.
#include "gemm_kernel.cuh"

namespace tp {

static const KernelEntry k_table[] = {
    mainloop_entry<2, 128, 2, false, false>(),
    mainloop_entry<2, 128, 3, false, false>(),
    mainloop_entry<2, 128, 4, false, false>(),
    mainloop_entry<2, 128, 5, false, false>(),
    mainloop_entry<2, 128, 6, false, false>(),
    mainloop_entry<2, 128, 7, false, false>(),
    mainloop_entry<2, 128, 8, false, false>(),
    mainloop_entry<2, 256, 2, false, false>(),
    mainloop_entry<2, 256, 3, false, false>(),
    mainloop_entry<2, 256, 4, false, false>(),
    mainloop_entry<2, 256, 5, false, false>(),
    mainloop_entry<2, 256, 6, false, false>(),
    mainloop_entry<2, 128, 8, true, false>(),
    mainloop_entry<2, 256, 6, true, false>(),
};

const KernelEntry* table_mainloop_cg2(int* n)
{
    *n = static_cast<int>(sizeof(k_table) / sizeof(k_table[0]));
    return k_table;
}

}  // namespace tp
