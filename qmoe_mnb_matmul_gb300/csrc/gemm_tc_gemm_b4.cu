// gemm_tc_gemm_b4.cu -- instantiations of the tensor-core GEMM (tile GEMM, INT4).
#include "gemm_tc_impl.cuh"

namespace mnb {
MNB_GEMM_TC_SLICE(gemm_tc_gemm_b4, kModeGemm, 4)
}  // namespace mnb
