// gemm_tc_gemm_b3.cu -- instantiations of the tensor-core GEMM (tile GEMM, INT3).
#include "gemm_tc_impl.cuh"

namespace mnb {
MNB_GEMM_TC_SLICE(gemm_tc_gemm_b3, kModeGemm, 3)
}  // namespace mnb
