// kernels.h -- registry of the compiled kernel variants, shared by the
// instantiation units and the host-side planner / launcher.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_kernel.cuh"

namespace dg {

struct KernelInfo;
// bh: B's tensor map for the loads of a tail half (K-major B: 64-row box).
// cluster: CTAs per cluster for kernels that are not CTA pairs (1 = none).
// smem: dynamic shared memory of this launch (the ring depth is p.stages).
using LaunchFn = cudaError_t (*)(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& bh,
                                 const CUtensorMap& d, const Params& p, int grid, cudaStream_t s, bool cooperative,
                                 int cluster, size_t smem);

struct KernelInfo {
    int bn, fp8, a_mn, b_mn, mode, pair, gs;
    int ks;            // K slices per pipeline stage (2: operands in 3-D TMA copies)
    int halves;        // can run tail tiles as two N halves
    int stages, smem_bytes, tmem_cols, threads, epi_warps;
    int launch_regs;   // register split (setmaxnreg): registers per thread the split assumes at launch; 0 = none
    // compact footprint (small-M form; otherwise the full one): ring depth and
    // shared memory that leave room for a second CTA on the SM
    int stages_compact, smem_compact;
    const void* func;  // host stub of the __global__ function (for attributes)
    LaunchFn launch;
};

template <class CF>
cudaError_t launch_variant(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& bh, const CUtensorMap& d,
                           const Params& p, int grid, cudaStream_t s, bool cooperative, int cluster, size_t smem) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(CF::NUM_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[3];
    unsigned n = 0;
    if (!cooperative) {
        // may start while the previous kernel in the stream finishes (the
        // kernel waits on griddepcontrol before touching global memory)
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (CF::PAIR || cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = CF::PAIR ? 2u : static_cast<unsigned>(cluster);
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (cooperative) {
        attr[n].id = cudaLaunchAttributeCooperative;
        attr[n].val.cooperative = 1;
        ++n;
    }
    cfg.attrs = n ? attr : nullptr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, gemm_persistent<CF>, a, b, bh, d, p);
}

template <class CF>
KernelInfo make_info() {
    return KernelInfo{CF::BN,     CF::FP8,    CF::A_MN,       CF::B_MN,      CF::MODE,
                      CF::PAIR ? 1 : 0, CF::GS ? 1 : 0, CF::KS, CF::HALVES ? 1 : 0, CF::STAGES, CF::SMEM_BYTES, CF::TMEM_COLS, CF::NUM_THREADS,
                      CF::EPI_WARPS, CF::REG_SPLIT ? CF::LAUNCH_REGS : 0,
                      CF::STAGES_COMPACT, CF::SMEM_FIXED + CF::STAGES_COMPACT * CF::STAGE_BYTES,
                      reinterpret_cast<const void*>(&gemm_persistent<CF>), &launch_variant<CF>};
}

// Each instantiation unit exports its table.
const KernelInfo* kernels_bf16(int* count);
const KernelInfo* kernels_fp8(int* count);
const KernelInfo* kernels_fp8_grouped(int* count);
const KernelInfo* kernels_two_slice(int* count);

}  // namespace dg
