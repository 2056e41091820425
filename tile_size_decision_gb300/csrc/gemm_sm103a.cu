// One compiled variant of the tcgen05 GEMM per translation unit: the build
// compiles this file once per tile width with -DTILES_GEMM_BN=<64|128|192|256>
// so the variants compile in parallel.
#include "gemm_sm103a.cuh"

#ifndef TILES_GEMM_BN
#error "TILES_GEMM_BN must be defined (64, 128, 192 or 256)"
#endif

namespace tiles {

template <>
int launch_gemm_variant<TILES_GEMM_BN>(const CUtensorMap& ta, const CUtensorMap& tb,
                                       const GemmArgs& args, int grid, cudaStream_t stream) {
    constexpr int BN = TILES_GEMM_BN;
    constexpr int STAGES = GemmStages<BN>::value;
    using L = GemmLayout<BN, STAGES>;
    auto kernel = gemm_tcgen05_kernel<BN, STAGES>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         L::SMEM_BYTES);
    if (e != cudaSuccess) return static_cast<int>(e);
    kernel<<<grid, kGemmThreads, L::SMEM_BYTES, stream>>>(ta, tb, args);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace tiles
