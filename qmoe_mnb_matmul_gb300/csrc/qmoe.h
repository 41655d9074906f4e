// qmoe.h -- internal interface of the QMoE expert-FFN pipeline.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace mnb {

struct ProjGeom {
    int64_t nb;         // blocks per row
    int64_t row_bytes;  // packed bytes per row
    int64_t zp_row;     // packed zero-point bytes per row
};

struct QmoeArgs {
    const void* X;
    int act_dtype;
    int64_t T, H, I, E;
    int k, normalize;
    const void* logits;
    int logits_dtype;        // fp32, fp16 or bf16 router logits
    const void* fc1_bias;    // [E, 2I] in the activation dtype (rows in the FC1 layout) or null
    const void* fc2_bias;    // [E, H] in the activation dtype or null
    const void* agg;         // [T, E] aggregation weights (combine weights) or null
    int agg_dtype;
    const uint8_t* fc1_w;
    const void* fc1_s;
    const uint8_t* fc1_zp;
    int fc1_bits;
    const uint8_t* fc2_w;
    const void* fc2_s;
    const uint8_t* fc2_zp;
    int fc2_bits;
    int bs;
    int fc1_layout;
    int x_vec;  // X rows may be read with 16-byte loads
    void* Y;
    void* workspace;
    ProjGeom fc1, fc2;
};

// Workspace bytes for one qmoe_forward call; false on overflow.
bool qmoe_workspace_bytes(int64_t T, int64_t H, int64_t I, int64_t E, int k, int64_t* bytes);

cudaError_t launch_qmoe(const QmoeArgs& q, int sm_count, bool pdl, cudaStream_t stream);

// Workspace offsets of the SwiGLU activations h [T*k, I] (fp32) and of the
// 256-byte region the fused decode kernel uses for its grid barrier counter.
void qmoe_ws_decode_regions(int64_t T, int64_t H, int64_t I, int64_t E, int k, int64_t* h_off, int64_t* sync_off);

// One token (T = 1), k <= 8: the fused decode layer (qmoe_decode.cu).
// cudaErrorNotSupported when the shape is outside its rules (the caller then
// runs the two-kernel decode plan).
cudaError_t launch_qmoe_decode_fused(const QmoeArgs& q, int sm_count, bool pdl, cudaStream_t stream);
cudaError_t qmoe_decode_take_error(unsigned int* out);

}  // namespace mnb
