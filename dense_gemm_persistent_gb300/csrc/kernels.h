// kernels.h -- registry of the compiled kernel variants, shared by the
// instantiation units and the host-side planner / launcher.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_kernel.cuh"

namespace dg {

struct KernelInfo;
using LaunchFn = cudaError_t (*)(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& d,
                                 const Params& p, int grid, cudaStream_t s, bool cooperative);

struct KernelInfo {
    int bn, fp8, a_mn, b_mn, mode;
    int stages, smem_bytes, tmem_cols;
    const void* func;  // host stub of the __global__ function (for attributes)
    LaunchFn launch;
};

template <class CF>
cudaError_t launch_variant(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& d, const Params& p,
                           int grid, cudaStream_t s, bool cooperative) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(CF::NUM_THREADS);
    cfg.dynamicSmemBytes = CF::SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    if (cooperative) {
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, gemm_persistent<CF>, a, b, d, p);
}

template <class CF>
KernelInfo make_info() {
    return KernelInfo{CF::BN,     CF::FP8,        CF::A_MN,      CF::B_MN,
                      CF::MODE,   CF::STAGES,     CF::SMEM_BYTES, CF::TMEM_COLS,
                      reinterpret_cast<const void*>(&gemm_persistent<CF>), &launch_variant<CF>};
}

// Each instantiation unit exports its table.
const KernelInfo* kernels_bf16(int* count);
const KernelInfo* kernels_fp8(int* count);

}  // namespace dg
