// gemm_tc_fc1_b4.cu -- instantiations of the tensor-core GEMM (grouped FC1 + SwiGLU, INT4).
#include "gemm_tc_impl.cuh"

namespace mnb {
MNB_GEMM_TC_SLICE(gemm_tc_fc1_b4, kModeFc1, 4)
}  // namespace mnb
