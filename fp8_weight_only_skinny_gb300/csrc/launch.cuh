// launch.cuh -- host-side launch of the skinny kernel variants.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include "kernel.cuh"
#include "internal.h"

namespace sk {

// pdl: programmatic dependent launch after the previous kernel on the stream;
// coop: a cooperative launch (all CTAs co-resident before any starts).
template <int FMT, int MP, bool F16OUT, bool ARGMAX, bool XWIDE>
cudaError_t launch_variant(const CUtensorMap &tm_codes, const CUtensorMap &tm_scales, const Params &p,
                           int grid, cudaStream_t stream, bool pdl, bool coop) {
    auto kfn = skinny_kernel<FMT, MP, F16OUT, ARGMAX, XWIDE>;
    constexpr size_t smem = smem_bytes<FMT, MP>();
    static bool attr_done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !attr_done[dev]) {
        e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(CTA_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = coop ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kfn, tm_codes, tm_scales, p);
}

template <int FMT, bool F16OUT, bool ARGMAX>
cudaError_t launch_by_m(int mp, bool xwide, const CUtensorMap &tm_codes, const CUtensorMap &tm_scales,
                        const Params &p, int grid, cudaStream_t stream, bool pdl, bool coop) {
    if (mp == 1) return launch_variant<FMT, 1, F16OUT, ARGMAX, false>(tm_codes, tm_scales, p, grid, stream, pdl, coop);
    if (xwide) return launch_variant<FMT, 8, F16OUT, ARGMAX, true>(tm_codes, tm_scales, p, grid, stream, pdl, coop);
    return launch_variant<FMT, 8, F16OUT, ARGMAX, false>(tm_codes, tm_scales, p, grid, stream, pdl, coop);
}

}  // namespace sk
