// k_nvfp4.cu -- instantiations of the NVFP4 kernel variants.
#include "launch.cuh"

namespace sk {

cudaError_t launch_nvfp4(int mp, bool xwide, bool f16out, bool argmax, const CUtensorMap &tm_codes,
                         const CUtensorMap &tm_scales, const Params &p, int grid,
                         cudaStream_t stream, bool pdl, bool coop) {
    if (argmax) return launch_by_m<NVFP4, false, true>(mp, xwide, tm_codes, tm_scales, p, grid, stream, pdl, coop);
    if (f16out) return launch_by_m<NVFP4, true, false>(mp, xwide, tm_codes, tm_scales, p, grid, stream, pdl, coop);
    return launch_by_m<NVFP4, false, false>(mp, xwide, tm_codes, tm_scales, p, grid, stream, pdl, coop);
}

}  // namespace sk
