// k_fp8.cu -- instantiations of the FP8 kernel variants.
#include "launch.cuh"

namespace sk {

cudaError_t launch_fp8(int mp, bool xwide, bool f16out, const CUtensorMap &tm_codes, const Params &p, int grid,
                       cudaStream_t stream, bool pdl, bool coop) {
    if (f16out) return launch_by_m<FP8, true, false>(mp, xwide, tm_codes, tm_codes, p, grid, stream, pdl, coop);
    return launch_by_m<FP8, false, false>(mp, xwide, tm_codes, tm_codes, p, grid, stream, pdl, coop);
}

}  // namespace sk
