// Implicit-GEMM convolution variants of the mainloop (im2col TMA producer):
// both atoms and both MMA N at their deepest rings, bf16 and fp32 outputs.
#include "gemm_kernel.cuh"

namespace tp {

static const KernelEntry k_table[] = {
    mainloop_entry<1, 128, 6, false, true>(),
    mainloop_entry<1, 256, 4, false, true>(),
    mainloop_entry<1, 128, 6, true, true>(),
    mainloop_entry<1, 256, 4, true, true>(),
    mainloop_entry<2, 128, 8, false, true>(),
    mainloop_entry<2, 256, 6, false, true>(),
    mainloop_entry<2, 128, 8, true, true>(),
    mainloop_entry<2, 256, 6, true, true>(),
};

const KernelEntry* table_mainloop_conv(int* n)
{
    *n = static_cast<int>(sizeof(k_table) / sizeof(k_table[0]));
    return k_table;
}

}  // namespace tp
