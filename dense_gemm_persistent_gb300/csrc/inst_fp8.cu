// inst_fp8.cu -- the FP8 E4M3 (kind::f8f6f4) kernel variants.
#include "kernels.h"

namespace dg {

const KernelInfo* kernels_fp8(int* count) {
    //                  BN  FP8   A_MN   B_MN   MODE
    static const KernelInfo table[] = {
        make_info<Cfg<256, true, false, false, MODE_TILE>>(),   // B stored N x K
        make_info<Cfg<128, true, false, false, MODE_TILE>>(),
        make_info<Cfg<64, true, false, false, MODE_TILE>>(),
        make_info<Cfg<256, true, false, true, MODE_TILE>>(),    // B stored K x N
        make_info<Cfg<128, true, false, true, MODE_TILE>>(),
        make_info<Cfg<16, true, false, false, MODE_SWAP>>(),    // small M, B stored N x K
        make_info<Cfg<32, true, false, false, MODE_SWAP>>(),
        make_info<Cfg<64, true, false, false, MODE_SWAP>>(),
        make_info<Cfg<16, true, true, false, MODE_SWAP>>(),     // small M, B stored K x N
        make_info<Cfg<32, true, true, false, MODE_SWAP>>(),
        make_info<Cfg<64, true, true, false, MODE_SWAP>>(),
        make_info<Cfg<256, true, false, false, MODE_ROWQ>>(),   // E4M3 row requantisation
        make_info<Cfg<256, true, false, true, MODE_ROWQ>>(),
        // CTA pairs: 256 x 256 tiles over two SMs
        make_info<Cfg<256, true, false, false, MODE_TILE, true>>(),
        make_info<Cfg<256, true, false, true, MODE_TILE, true>>(),
        make_info<Cfg<256, true, false, false, MODE_ROWQ, true>>(),
        make_info<Cfg<256, true, false, true, MODE_ROWQ, true>>(),
        // CTA pairs with two K slices per stage (3-D TMA copies)
        make_info<Cfg<256, true, false, false, MODE_TILE, true, false, 2>>(),
        make_info<Cfg<256, true, false, true, MODE_TILE, true, false, 2>>(),
        make_info<Cfg<256, true, false, false, MODE_ROWQ, true, false, 2>>(),
        make_info<Cfg<256, true, false, true, MODE_ROWQ, true, false, 2>>(),
    };
    *count = static_cast<int>(sizeof(table) / sizeof(table[0]));
    return table;
}

}  // namespace dg
