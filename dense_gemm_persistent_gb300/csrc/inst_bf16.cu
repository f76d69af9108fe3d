// inst_bf16.cu -- the BF16 (kind::f16) kernel variants.
#include "kernels.h"

namespace dg {

const KernelInfo* kernels_bf16(int* count) {
    //                  BN  FP8    A_MN   B_MN   MODE
    static const KernelInfo table[] = {
        make_info<Cfg<256, false, false, true, MODE_TILE>>(),   // B stored K x N
        make_info<Cfg<128, false, false, true, MODE_TILE>>(),
        make_info<Cfg<64, false, false, true, MODE_TILE>>(),
        make_info<Cfg<256, false, false, false, MODE_TILE>>(),  // B stored N x K
        make_info<Cfg<128, false, false, false, MODE_TILE>>(),
        make_info<Cfg<64, false, false, false, MODE_TILE>>(),
        make_info<Cfg<16, false, false, false, MODE_SWAP>>(),   // small M, B stored N x K
        make_info<Cfg<32, false, false, false, MODE_SWAP>>(),
        make_info<Cfg<64, false, false, false, MODE_SWAP>>(),
        make_info<Cfg<16, false, true, false, MODE_SWAP>>(),    // small M, B stored K x N
        make_info<Cfg<32, false, true, false, MODE_SWAP>>(),
        make_info<Cfg<64, false, true, false, MODE_SWAP>>(),
        make_info<Cfg<256, false, false, false, MODE_ROWQ>>(),  // E4M3 row requantisation
        make_info<Cfg<256, false, false, true, MODE_ROWQ>>(),
        // CTA pairs: 256 x 256 tiles over two SMs
        make_info<Cfg<256, false, false, true, MODE_TILE, true>>(),
        make_info<Cfg<256, false, false, false, MODE_TILE, true>>(),
        make_info<Cfg<256, false, false, false, MODE_ROWQ, true>>(),
        make_info<Cfg<256, false, false, true, MODE_ROWQ, true>>(),
        // CTA pairs with two K slices per stage (3-D TMA copies)
        make_info<Cfg<256, false, false, true, MODE_TILE, true, false, 2>>(),
        make_info<Cfg<256, false, false, false, MODE_TILE, true, false, 2>>(),
        make_info<Cfg<256, false, false, false, MODE_ROWQ, true, false, 2>>(),
        make_info<Cfg<256, false, false, true, MODE_ROWQ, true, false, 2>>(),
    };
    *count = static_cast<int>(sizeof(table) / sizeof(table[0]));
    return table;
}

}  // namespace dg
