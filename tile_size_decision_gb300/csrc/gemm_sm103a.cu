// One compiled variant of the tcgen05 GEMM per translation unit: the build
// compiles this file once per (tile width, CTAs per MMA) with
// -DTILES_GEMM_BN=<64|128|192|256> -DTILES_GEMM_CG=<1|2>, so the variants
// compile in parallel.
#include <cuda_runtime.h>

#include "gemm_sm103a.cuh"

#ifndef TILES_GEMM_BN
#error "TILES_GEMM_BN must be defined (64, 128, 192 or 256)"
#endif
#ifndef TILES_GEMM_CG
#define TILES_GEMM_CG 1
#endif

namespace tiles {

namespace {

constexpr int BN = TILES_GEMM_BN;
constexpr int CG = TILES_GEMM_CG;
constexpr int STAGES = GemmStages<BN, CG>::value;
using Layout = GemmLayout<BN, STAGES, CG>;

void fill_launch(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, int groups,
                 cudaStream_t stream) {
    *cfg = cudaLaunchConfig_t{};
    cfg->gridDim = dim3(static_cast<unsigned>(groups * CG), 1, 1);
    cfg->blockDim = dim3(kGemmThreads, 1, 1);
    cfg->dynamicSmemBytes = Layout::SMEM_BYTES;
    cfg->stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg->attrs = attr;
    cfg->numAttrs = CG > 1 ? 1 : 0;
}

cudaError_t set_smem_attribute() {
    return cudaFuncSetAttribute(gemm_tcgen05_kernel<BN, STAGES, CG>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, Layout::SMEM_BYTES);
}

}  // namespace

template <>
int gemm_variant_max_groups<BN, CG>(int sm_count) {
    if (CG == 1) return sm_count;
    if (set_smem_attribute() != cudaSuccess) return sm_count / CG;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    fill_launch(&cfg, attr, sm_count / CG, nullptr);
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, gemm_tcgen05_kernel<BN, STAGES, CG>, &cfg) !=
            cudaSuccess || clusters <= 0) {
        cudaGetLastError();
        return sm_count / CG;
    }
    return clusters;
}

template <>
int gemm_variant_attributes<BN, CG>(int sm_count, VariantAttributes* out) {
    cudaError_t e = set_smem_attribute();
    if (e != cudaSuccess) return static_cast<int>(e);
    cudaFuncAttributes fa{};
    e = cudaFuncGetAttributes(&fa, gemm_tcgen05_kernel<BN, STAGES, CG>);
    if (e != cudaSuccess) return static_cast<int>(e);
    out->regs = fa.numRegs;
    out->local_bytes = static_cast<int>(fa.localSizeBytes);
    out->static_smem = static_cast<int>(fa.sharedSizeBytes);
    out->dynamic_smem = Layout::SMEM_BYTES;
    out->max_dynamic_smem = fa.maxDynamicSharedSizeBytes;
    int blocks = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, gemm_tcgen05_kernel<BN, STAGES, CG>,
                                                      kGemmThreads, Layout::SMEM_BYTES);
    if (e != cudaSuccess) return static_cast<int>(e);
    out->blocks_per_sm = blocks;
    if (CG == 1) {
        out->groups = blocks * sm_count;
        return static_cast<int>(cudaSuccess);
    }
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    fill_launch(&cfg, attr, sm_count / CG, nullptr);
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, gemm_tcgen05_kernel<BN, STAGES, CG>, &cfg);
    if (e != cudaSuccess) return static_cast<int>(e);
    out->groups = clusters;
    return static_cast<int>(cudaSuccess);
}

template <>
int launch_gemm_variant<BN, CG>(const CUtensorMap& ta, const CUtensorMap& tb,
                                const CUtensorMap& tc, const GemmArgs& args, int groups,
                                cudaStream_t stream) {
    cudaError_t e = set_smem_attribute();
    if (e != cudaSuccess) return static_cast<int>(e);
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    fill_launch(&cfg, attr, groups, stream);
    // Programmatic serialization: the blocks may start their set-up while
    // the previous kernel on the stream drains; they wait for it in-kernel
    // before touching global memory.
    attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
    ++cfg.numAttrs;
    e = cudaLaunchKernelEx(&cfg, gemm_tcgen05_kernel<BN, STAGES, CG>, ta, tb, tc, args);
    if (e != cudaSuccess) return static_cast<int>(e);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace tiles
