// gemm_tc_fc1_b3.cu -- instantiations of the tensor-core GEMM (grouped FC1 + SwiGLU, INT3).
#include "gemm_tc_impl.cuh"

namespace mnb {
MNB_GEMM_TC_SLICE(gemm_tc_fc1_b3, kModeFc1, 3)
}  // namespace mnb
