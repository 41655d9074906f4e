// gemv.cu -- the SIMT GEMV over the raw row-local LSB-first layout: every
// width 1..8, fp32 / fp16 / bf16 scales (kernel and shapes in gemv_impl.cuh).
#include "gemv_impl.cuh"

namespace mnb {

cudaError_t gemv_take_error(unsigned int* out) { return take_unit_error(out); }

size_t gemv_smem_bytes(int64_t M, int64_t K, int bits, int bs, int scale_dtype) {
    const int nb = static_cast<int>(cdiv<int64_t>(K, bs));
    const int C = nb * bs / 32;
    const int64_t row_bytes = int64_t(nb) * bs * bits / 8;
    const int ssize = ssize_of(scale_dtype);
    const int64_t RC = std::max<int64_t>(kConsumerWarps, row_align(row_bytes, nb, ssize));
    const Plan p = make_plan(pick_mt(M), C, static_cast<int>(RC), row_bytes, nb, ssize, 2);
    return p.total <= kSmemBudget ? static_cast<size_t>(p.total) : 0;
}

cudaError_t launch_gemv(const GemvArgs& a, int scale_dtype, int sm_count, bool pdl, cudaStream_t stream) {
    if (a.bits != 3 && a.bits != 4) {  // widths 1, 2, 5..8
        if (scale_dtype == kF32) return launch_mt<0, kF32>(a, sm_count, pdl, stream);
        if (scale_dtype == kF16) return launch_mt<0, kF16>(a, sm_count, pdl, stream);
        return launch_mt<0, kBF16>(a, sm_count, pdl, stream);
    }
    if (a.bits == 4) {
        if (scale_dtype == kF32) return launch_mt<4, kF32>(a, sm_count, pdl, stream);
        if (scale_dtype == kF16) return launch_mt<4, kF16>(a, sm_count, pdl, stream);
        return launch_mt<4, kBF16>(a, sm_count, pdl, stream);
    }
    if (scale_dtype == kF32) return launch_mt<3, kF32>(a, sm_count, pdl, stream);
    if (scale_dtype == kF16) return launch_mt<3, kF16>(a, sm_count, pdl, stream);
    return launch_mt<3, kBF16>(a, sm_count, pdl, stream);
}

}  // namespace mnb
