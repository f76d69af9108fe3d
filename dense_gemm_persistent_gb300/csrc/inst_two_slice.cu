// inst_two_slice.cu -- single-CTA tile kernels that load two 128-byte K slices
// per pipeline stage (each operand of a stage in one 3-D TMA copy), BF16 and
// FP8 E4M3, for tiles 128 and 64 wide (a 128 x 256 tile would keep only two
// stages of 96 KB, which streamed slower than four of 48 KB). A translation
// unit of their own so that they compile in parallel with the others.
#include "kernels.h"

namespace dg {

const KernelInfo* kernels_two_slice(int* count) {
    //                  BN  FP8    A_MN   B_MN   MODE       PAIR   GS     KS
    static const KernelInfo table[] = {
        make_info<Cfg<128, false, false, true, MODE_TILE, false, false, 2>>(),   // BF16, B stored K x N
        make_info<Cfg<64, false, false, true, MODE_TILE, false, false, 2>>(),
        make_info<Cfg<128, false, false, false, MODE_TILE, false, false, 2>>(),  // BF16, B stored N x K
        make_info<Cfg<64, false, false, false, MODE_TILE, false, false, 2>>(),
        make_info<Cfg<128, true, false, false, MODE_TILE, false, false, 2>>(),   // E4M3, B stored N x K
        make_info<Cfg<64, true, false, false, MODE_TILE, false, false, 2>>(),
        make_info<Cfg<128, true, false, true, MODE_TILE, false, false, 2>>(),    // E4M3, B stored K x N
    };
    *count = static_cast<int>(sizeof(table) / sizeof(table[0]));
    return table;
}

}  // namespace dg
