// qmoe_static.cu -- qmoe_forward_static: one QMoE layer with no caller-provided
// workspace, for callers that cannot allocate device memory.
//
// Its scratch is a file-scope device array of kStaticScratchBytes.  Every GPU
// that loads this library holds one copy until the process exits.  Host code
// must not pass the array's name to a kernel (on the host it is only a
// stand-in for the symbol), so every call looks up the current device's
// address with cudaGetSymbolAddress.

#include "common.cuh"

namespace mnb {
namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;  // 8 MiB

static __device__ __align__(256) unsigned char g_qmoe_scratch[kStaticScratchBytes];

// Device address of the current device's copy of the scratch array.  Looked
// up on every call (a host-side symbol query, no allocation): a cached address
// would dangle after a device reset reloads the module.
cudaError_t scratch_address(void** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_qmoe_scratch);
    if (e != cudaSuccess) return e;
    *out = p;
    return cudaSuccess;
}

}  // namespace
}  // namespace mnb

extern "C" mnb_status qmoe_forward_static(const void* X, mnb_dtype act_dtype, int64_t T, int64_t H,
                                          const float* router_logits, int64_t E, int k, int normalize_topk,
                                          const uint8_t* fc1_w, const void* fc1_scales, const uint8_t* fc1_zp,
                                          int fc1_bits, const uint8_t* fc2_w, const void* fc2_scales,
                                          const uint8_t* fc2_zp, int fc2_bits, int64_t I, int block_size,
                                          mnb_fc1_layout fc1_layout, void* Y, mnb_stream_t stream) {
    size_t need = 0;
    const mnb_status st = qmoe_workspace_size(T, H, I, E, k, act_dtype, &need);
    if (st != MNB_OK) return st;
    if (need > mnb::kStaticScratchBytes) return MNB_ERR_WORKSPACE;  // beyond the fixed 8 MiB scratch
    void* scratch = nullptr;
    if (mnb::scratch_address(&scratch) != cudaSuccess) return MNB_ERR_CUDA;
    // Nothing in the scratch has to start at zero: every kernel of the layer
    // writes what it later reads within the same call.
    return qmoe_forward(X, act_dtype, T, H, router_logits, E, k, normalize_topk, fc1_w, fc1_scales, fc1_zp, fc1_bits,
                        fc2_w, fc2_scales, fc2_zp, fc2_bits, I, block_size, fc1_layout, Y, scratch,
                        mnb::kStaticScratchBytes, stream);
}
