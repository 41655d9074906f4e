// gemv_pp.cu -- the SIMT GEMV over the version-1 prepacked layout (INT4 and
// regrouped INT3; kernel and shapes in gemv_impl.cuh).  Each stage of the ring
// is one bulk copy of a block of whole prepacked rows (codes, scales and zero
// points together), for any K.
#include "gemv_impl.cuh"

namespace mnb {

cudaError_t gemv_pp_take_error(unsigned int* out) { return take_unit_error(out); }

cudaError_t launch_gemv_prepacked(const GemvArgs& a, int scale_dtype, int sm_count, bool pdl, cudaStream_t stream) {
    if (a.bits == 4) {
        if (scale_dtype == kF32) return launch_mt<4, kF32, true>(a, sm_count, pdl, stream);
        if (scale_dtype == kF16) return launch_mt<4, kF16, true>(a, sm_count, pdl, stream);
        return launch_mt<4, kBF16, true>(a, sm_count, pdl, stream);
    }
    if (scale_dtype == kF32) return launch_mt<3, kF32, true>(a, sm_count, pdl, stream);
    if (scale_dtype == kF16) return launch_mt<3, kF16, true>(a, sm_count, pdl, stream);
    return launch_mt<3, kBF16, true>(a, sm_count, pdl, stream);
}

}  // namespace mnb
