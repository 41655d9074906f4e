// kernels.h -- host-side launchers of the sm_103a kernels (internal to the library).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace mnb {

// Enqueues kern<<<grid, block, smem, stream>>>(args...), as a programmatic
// dependent of the work ahead on the stream when `pdl`: the kernel may then
// start while its predecessor finishes, so it must not read anything the
// predecessor writes before its own griddepcontrol.wait.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_ex(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
                             Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ------------------------------------------------------------- SIMT GEMV
// Y[M, N] = A[M, K] . W^T for small M, streaming packed rows through shared memory.
struct GemvArgs {
    const void* A;
    int a_dtype;
    int64_t M, K;
    const uint8_t* B;
    const void* scales;
    const uint8_t* zp;
    int64_t N;
    int bits, bs, nb;
    int64_t row_bytes;
    int zp_row_bytes;
    void* Y;
    int y_dtype;
    int64_t y_ld;          // row stride of Y in elements (N for a plain matmul)
    int rows_per_block;    // RC: rows of B staged per pipeline stage (8 warps x rows per warp)
    int stages;            // depth of the shared-memory ring
    int n_blocks;          // ceil(N / RC)
    int chunks;            // C = nb * bs / 32 (32 codes per chunk)
    int a_vec;             // activation rows may be read with 16-byte loads
    int prefetch_all;      // prefetch the CTA's whole row range into L2 before the dependency wait
    int int8a;             // int8 activation compute: A quantised per (row, block) to int8
    // dense gate/up with SwiGLU: N = 2 * pairs logical rows (gate i = 2i, up i =
    // 2i + 1), stored in B interleaved (fc1_inter) or as gate rows then up rows;
    // Y[m, i] = silu(gate_i) * up_i, y_ld = pairs
    int swiglu, fc1_inter;
    int64_t pairs;
    // prepacked weight (gemv_pp.cu): B = the first row, row_bytes = the row
    // stride; the header and the identity the kernel checks it against;
    // scales / zero points at these offsets within a row (zero points: -1 = none)
    const void* pp_header;
    uint64_t pp_identity;
    int64_t pp_scale_off, pp_zp_off;
    // grouped QMoE projection (gemv_grouped.cu): CTA row y takes m-tile y of
    // g_tiles ({expert e, first sorted row, rows, 0}; *g_ntiles of them), whose
    // weight, scales and zero points start e * w_estride / s_estride / z_estride
    // bytes into B / scales / zp; the activation of sorted row s is A row
    // g_perm[s] / g_k (g_perm set) or s; Y rows are sorted rows; bias [E, N]
    // in bias_dtype (FC1: rows in the weight's gate/up layout) or null
    const int4* g_tiles;
    const int* g_ntiles;
    const int* g_perm;
    int g_k;
    int64_t w_estride, s_estride, z_estride;
    const void* bias;
    int bias_dtype;
};

// Chooses the launch shape and enqueues the kernel.  scale_dtype selects the
// instantiation.  Returns cudaSuccess or the launch error; cudaErrorNotSupported
// when the shape does not fit the kernel's shared-memory plan.
cudaError_t launch_gemv(const GemvArgs& a, int scale_dtype, int sm_count, bool pdl,
                        cudaStream_t stream);

// The grouped QMoE projection (see the g_* fields): bits 3 or 4, fp16 / bf16
// scales, up to 4 rows per m-tile; grid_y m-tile slots (CTAs past *g_ntiles
// exit), est_tiles the expected tile count (sets the CTAs per tile).
// cudaErrorNotSupported when the shape does not fit the plan.
cudaError_t launch_gemv_grouped(const GemvArgs& a, int scale_dtype, int64_t grid_y, int64_t est_tiles, int sm_count,
                                bool pdl, cudaStream_t stream);
constexpr int kGroupedGemvRows = 4;  // rows of an m-tile of the grouped GEMV
// Whether the grouped plan takes this projection (bits, scale dtype, shared memory).
bool gemv_grouped_fits(const GemvArgs& a, int scale_dtype);

// The GEMV over a prepacked weight (a.B, a.row_bytes, a.pp_* set from its
// descriptor); bits 3 or 4.
cudaError_t launch_gemv_prepacked(const GemvArgs& a, int scale_dtype, int sm_count, bool pdl, cudaStream_t stream);
cudaError_t gemv_pp_take_error(unsigned int* out);

// The prepack kernel: the version-1 layout of a row-local weight (header included).
cudaError_t launch_prepack(const uint8_t* B, const void* scales, int scale_dtype, const uint8_t* zp, int64_t N,
                           int64_t K, int bits, int bs, const void* header, size_t header_bytes, uint8_t* dst,
                           int64_t row_stride, int64_t scale_off, int64_t zp_off, int sm_count, cudaStream_t stream);

// Shared memory the GEMV plan needs for (K, bits, bs, scale dtype, M); 0 if unsupported.
size_t gemv_smem_bytes(int64_t M, int64_t K, int bits, int bs, int scale_dtype);

// ------------------------------------------------ tensor-core GEMM (tcgen05)
// Y[M, N] = A[M, K] . W^T, A fp16/bf16 row-major with K % 8 == 0 and a 16-byte
// aligned base (TMA), swap-AB tiles of 128 weight rows.
struct GemmTcArgs {
    const void* A;
    int a_dtype;
    int64_t M, K;
    const uint8_t* B;
    const void* scales;
    const uint8_t* zp;
    int64_t N;
    int bits, bs, nb;
    int64_t row_bytes;
    int zp_row_bytes;
    void* Y;
    int y_dtype;
    void* workspace;        // split-K partial sums (may be null: no split)
    size_t workspace_bytes;
};
cudaError_t launch_gemm_tc(const GemmTcArgs& g, int scale_dtype, int sm_count, bool pdl, cudaStream_t stream);

// Workspace the tensor-core GEMM uses for this problem: fp32 partial sums when
// the output tiles alone cannot fill the GPU and K is split (0 otherwise).
size_t gemm_tc_workspace_bytes(int64_t M, int64_t K, int64_t N, int sm_count);

// Kernel-side arguments of the tensor-core GEMM, shared with the grouped QMoE
// launches.  Weight matrix of an expert: `rows` rows of K codes.
struct TcArgs {
    int64_t M, K, rows;
    const uint8_t* B;
    const void* scales;
    const uint8_t* zp;
    int64_t row_bytes;
    int nb, bs, zp_row_bytes;
    int64_t w_expert_stride, s_expert_stride, z_expert_stride;  // bytes between experts
    void* Y;
    int y_dtype;
    int64_t ld_y;          // row stride of the output in elements
    int tiles_n, tiles_m, k_steps;  // k_steps: K steps of one tile (of one split of K)
    int splits;                     // dense: K split in this many parts (partials, then a reduction)
    float* partials;                // [splits][M][N] fp32 when splits > 1
    int stages, stages_w;  // activation ring and dequantised-weight ring depths
    uint32_t tmem_cols;
    // grouped (QMoE) launches: activation-row tiles {expert, first sorted row, rows, 0}
    const int4* mtiles;
    const int* n_mtiles;
    const int* perm;       // FC1: sorted position -> flat (token, slot) index
    int k;
    int64_t I;
    int inter;             // FC1 rows interleaved gate/up
    const void* X;         // FC1: activations gathered by token
    int64_t experts;       // matrices stacked in B / scales (grouped launches; 0 or 1 otherwise)
    int w_tma, s_tma;      // set by the launcher: packed rows / scales come as tensor tiles
    // Second pass of an fp32 output from 16-bit activations: the weight
    // operand is the remainder s (q - z) - round16(s (q - z)) (rounded to the
    // activation type) and the epilogue adds to the fp32 output instead of
    // storing it.
    int remainder;
    // grouped (QMoE) launches: bias [experts, rows] in the activation dtype
    // added to each output row (FC1: to the gate and up rows before SwiGLU), or null
    const void* bias;
};

// Rows of activations per tile (32 .. 256) for `rows` activation rows spread
// over `matrices` weight matrices (experts) in a grouped launch.
int grouped_tile_m(int64_t rows, int64_t matrices);

// Dense H[M, I] = silu(A . Wg^T) * (A . Wu^T) on the tensor cores (B holds the
// 2I gate/up rows, interleaved or gate half then up half).
cudaError_t launch_gate_up_tc(const GemmTcArgs& g, int64_t I, bool inter, int scale_dtype, int sm_count, bool pdl,
                              cudaStream_t stream);

// Grouped per-expert tensor-core GEMM over the m-tiles in the workspace:
// fc1 gathers X rows by token and writes silu(gate)*up; otherwise a dense
// tile GEMM on A_rows [a_rows, a_cols] (TMA).
cudaError_t launch_grouped_tc(bool fc1, const TcArgs& a, int bits, int scale_dtype, int a_dtype, const void* A_rows,
                              int64_t a_rows, int64_t a_cols, int tile_m, int sm_count, bool pdl, cudaStream_t stream);

// --------------------------------------------------------------- unpack
cudaError_t launch_pack_codes(const uint8_t* codes, int64_t rows, int64_t K, int bits, int bs, uint8_t* packed,
                              cudaStream_t stream);
cudaError_t launch_unpack_codes(const uint8_t* packed, int64_t rows, int64_t K, int bits, int bs,
                                uint8_t* codes, cudaStream_t stream);

// ------------------------------------------------------------- routing
// logits [T, E] in dtype ldt; agg (or null): [T, E] aggregation weights in dtype
// adt, which replace the routing weights of the selected experts.
// `pdl`: these launches may start while the work ahead finishes (each kernel
// reads its inputs only after its dependency wait).
cudaError_t launch_route(const void* logits, int ldt, int64_t T, int64_t E, int k, int normalize,
                         int32_t* idx, float* w, const void* agg, int adt, cudaStream_t stream, bool pdl = false);
// One CTA; with mtiles set it also writes the grouped plan's m-tiles of <= tile_m
// sorted pairs per expert and their count.
cudaError_t launch_permute(const int32_t* idx, int64_t T, int k, int64_t E, int32_t* counts,
                           int32_t* offsets, int32_t* perm, int32_t* inv_perm, cudaStream_t stream,
                           int4* mtiles = nullptr, int* n_mtiles = nullptr, int tile_m = 0, bool pdl = false);

// The same stable permutation over many CTAs: chunk histograms (n_chunks x E
// ints of scratch in `chunkc`, n_chunks = permute_chunks(T * k)), a scan, and
// a scatter.  E <= 1024.
int64_t permute_chunks(int64_t P);
cudaError_t launch_permute_chunked(const int32_t* idx, int64_t T, int k, int64_t E, int32_t* chunkc, int32_t* counts,
                                   int32_t* offsets, int32_t* perm, int32_t* inv_perm, cudaStream_t stream,
                                   bool pdl = false);

// Per-translation-unit device error words (read and cleared; 0 = none).
cudaError_t gemv_take_error(unsigned int* out);
cudaError_t qmoe_take_error(unsigned int* out);
cudaError_t gemm_tc_take_error(unsigned int* out);
cudaError_t quant_take_error(unsigned int* out);
cudaError_t diag_take_error(unsigned int* out);

// ------------------------------------------------------------ diagnostics
// One CTA waits, with the library's bounded wait and a limit of limit_ns, on
// an mbarrier no thread arrives at; the wait records MNB_ERR_TIMEOUT.
cudaError_t launch_diag_wait_timeout(uint64_t limit_ns, cudaStream_t stream);

// --------------------------------------------------------------- quantizer
// Symmetric grouped INT3 round-to-nearest of W [N, K] (K % bs == 0) into
// packed codes B [N, K/bs, 3*bs/8] and scales S [N, K/bs].
cudaError_t launch_quantize_int3(const void* W, int w_dtype, int64_t N, int64_t K, int bs, uint8_t* B, void* S,
                                 int s_dtype, int sm_count, cudaStream_t stream);

}  // namespace mnb
