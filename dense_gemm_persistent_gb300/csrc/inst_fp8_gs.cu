// inst_fp8_gs.cu -- the FP8 E4M3 kernel variants with per-K-group scales
// (one FP32 scale per row of A and per output channel for every K group).
#include "kernels.h"

namespace dg {

const KernelInfo* kernels_fp8_grouped(int* count) {
    //                  BN  FP8   A_MN   B_MN   MODE        PAIR   GS
    static const KernelInfo table[] = {
        make_info<Cfg<256, true, false, false, MODE_TILE, true, true>>(),    // B stored N x K
        make_info<Cfg<256, true, false, false, MODE_TILE, false, true>>(),
        make_info<Cfg<128, true, false, false, MODE_TILE, false, true>>(),
        make_info<Cfg<64, true, false, false, MODE_TILE, false, true>>(),
        make_info<Cfg<256, true, false, true, MODE_TILE, true, true>>(),     // B stored K x N
        make_info<Cfg<256, true, false, true, MODE_TILE, false, true>>(),
        make_info<Cfg<128, true, false, true, MODE_TILE, false, true>>(),
        make_info<Cfg<16, true, false, false, MODE_SWAP, false, true>>(),    // small M, B stored N x K
        make_info<Cfg<32, true, false, false, MODE_SWAP, false, true>>(),
        make_info<Cfg<64, true, false, false, MODE_SWAP, false, true>>(),
        make_info<Cfg<16, true, true, false, MODE_SWAP, false, true>>(),     // small M, B stored K x N
        make_info<Cfg<32, true, true, false, MODE_SWAP, false, true>>(),
        make_info<Cfg<64, true, true, false, MODE_SWAP, false, true>>(),
    };
    *count = static_cast<int>(sizeof(table) / sizeof(table[0]));
    return table;
}

}  // namespace dg
