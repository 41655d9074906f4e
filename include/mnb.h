/*
 * mnb.h -- C ABI of the GB300 (sm_103a) library for block-quantized
 * weight-only matmul (MatMulNBits) and the QMoE expert FFN built on it.
 *
 * Shared conventions
 * ------------------
 * Pointers.  Every tensor argument is a device pointer owned by the caller,
 * except mnb_validate_host(), which reads host buffers.  The library keeps no
 * state between calls that affects results and never repacks weights on its
 * own: packed weights are consumed in the layout below on every call ("Qwen3
 * Missing-Kernel Implementation Plan", PR sequence rows K01/K02: reuse constant
 * packed weights, no repacking), unless the caller prepacks a weight once into
 * the opt-in private layout (mnb_prepack, below).
 *
 * Streams.  `stream` is a cudaStream_t (0 = the legacy default stream).  Calls
 * enqueue asynchronous work on it and return without synchronising, except
 * mnb_get_last_device_error(), which synchronises `stream`.
 *
 * Overlapped launches.  Kernels are launched as programmatic dependents of the
 * kernel ahead of them on the stream, so a call's prologue (barrier set-up,
 * tensor-memory allocation, L2 prefetches of its packed weights) may run while
 * the kernel ahead is still finishing.  No call reads any of its inputs before
 * the work ahead of it on the stream has completed (an L2 prefetch reads
 * nothing the call uses: L2 is coherent with every later write), so any
 * tensor may be the output of the immediately preceding kernel, whether it
 * belongs to this library or not.  Setting the environment variable
 * MNB_DISABLE_PDL turns the overlap off.
 *
 * Layouts (all dense, row-major, C order):
 *   bs = block_size, nb = ceil(K / bs), blob = bs * bits / 8 bytes.
 *   B_packed     uint8 [N, nb, blob].  Row n is one stream of K codes of width
 *                `bits`: code k occupies stream bits bits*k .. bits*k+bits-1,
 *                least significant bit first, stream bit i being bit i%8 of
 *                byte i/8 (so an INT4 byte holds column 2j in its low nibble and
 *                2j+1 in its high nibble, and 3-bit codes cross byte
 *                boundaries).  Codes at k >= K in the last blob are padding and
 *                are never read into a result ("INT3 QMoE CUDA correctness
 *                baseline and Qwen experimental results", section "P0: Portable
 *                Format and Numerical References": row-local LSB-first packing).
 *   scales       [N, nb], dtype `scale_dtype`.
 *   zero_points  uint8 [N, ceil(nb * bits / 8)]: one code of width `bits` per
 *                block, packed per row by the same LSB-first rule ("packed
 *                per-row block zero points", same section).  NULL selects the
 *                implicit zero point 2^(bits-1): 8 for INT4, 4 for INT3 (the
 *                offset-4 decoding (code - 4) * scale).
 *   Dequantised weight: w[n, k] = scale[n, k/bs] * (code[n, k] - zp[n, k/bs]).
 *
 * Supported set.  bits in {3, 4} (mnb_matmul and mnb_matmul_int8a: 1..8, the
 * widths other than 3 and 4 on CUDA cores); block_size in {32, 64, 128};
 * activation and output dtypes f32 / f16 / bf16 for mnb_matmul (f16 / bf16 for QMoE); scale
 * dtype f32 or equal to the activation dtype (QMoE: equal).  Alignment:
 * B_packed and the scales (mnb_matmul; QMoE: fc1_w, fc2_w, fc1_scales and
 * fc2_scales) must be 16-byte aligned, the QMoE workspace 256-byte aligned,
 * every other tensor aligned to its element size.  Anything else returns
 * MNB_ERR_UNSUPPORTED before any work is enqueued; no call ever falls back to
 * a CPU path or to a different kernel family silently.
 *
 * Errors.  Metadata is validated on the host before any launch (payloads are
 * never read on the host, except by mnb_validate_host).  Launch failures return
 * MNB_ERR_CUDA.  Kernels that wait on on-chip barriers give up after a bounded
 * time, record MNB_ERR_TIMEOUT in a device error word and return;
 * mnb_get_last_device_error() reports and clears that word.
 */
#ifndef MNB_H_
#define MNB_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MNB_OK = 0,
    MNB_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, k > E, ... */
    MNB_ERR_UNSUPPORTED = 2,   /* valid request outside the supported set */
    MNB_ERR_SIZE_OVERFLOW = 3, /* a byte count does not fit in 63 bits */
    MNB_ERR_WORKSPACE = 4,     /* workspace missing or smaller than required */
    MNB_ERR_CUDA = 5,          /* a CUDA runtime call failed */
    MNB_ERR_TIMEOUT = 6,       /* a bounded on-device wait gave up */
    MNB_ERR_CONTENT = 7        /* malformed content: mnb_validate_host, or a block
                                  mnb_quantize_int3 rejected (device error word) */
} mnb_status;

typedef enum { MNB_F32 = 0, MNB_F16 = 1, MNB_BF16 = 2 } mnb_dtype;

/* Row order of a fused FC1 weight of 2I rows: INTERLEAVED puts gate_i at row 2i
 * and up_i at row 2i+1 (the fused interleaved gate/up of "INT3 QMoE CUDA
 * correctness baseline...", "P1: Compatible QMoE v1 Extension"); CONCAT puts
 * gate_i at row i and up_i at row I+i. */
typedef enum { MNB_FC1_INTERLEAVED = 0, MNB_FC1_CONCAT = 1 } mnb_fc1_layout;

/* ABI-identical to cudaStream_t; declared here so that callers need no CUDA headers. */
typedef struct CUstream_st* mnb_stream_t;

/* ------------------------------------------------------------ MatMulNBits */

/* Bytes of device workspace mnb_matmul can use for this problem (0 = none, in
 * which case workspace may be NULL): the bounded workspace of "Qwen3
 * Missing-Kernel Implementation Plan", row K03.  The bound depends only on the arguments.
 * Non-zero for tensor-core problems whose output tiles cannot fill the GPU
 * (small M, few output columns): K is then split across CTAs and the fp32
 * partial sums go to the workspace before one reduction.  A call given less
 * (or NULL) splits K less, or not at all: same result, slower. */
mnb_status mnb_matmul_workspace_size(int64_t M, int64_t K, int64_t N, int bits, int block_size,
                                     mnb_dtype a_dtype, size_t* bytes);

/* Y[M, N] = A[M, K] . W^T with W[N, K] dequantised from B_packed/scales/
 * zero_points on the fly ("Qwen3 Missing-Kernel Implementation Plan", rows
 * K01 MatMulNBits contract, K02 M=1 decode GEMV, K03 small-M and prefill GEMM
 * with partial blocks and output tails).  Any M >= 1, K >= 1, N >= 1.
 * Accumulation is fp32; the dequantised weight is formed in fp32 (SIMT paths)
 * or rounded to bf16/fp16 in shared memory before a tensor-core contraction
 * (M >= 16 with f16/bf16 activations); an fp32 Y from f16/bf16 activations
 * adds, in a second tensor-core pass, the product with what that rounding
 * left (itself rounded to 16 bits), so its weights carry ~16 significant
 * bits.  Y is written in y_dtype with round-to-nearest-even.  `workspace` (16-byte aligned, see
 * mnb_matmul_workspace_size) holds split-K partial sums; the split changes the
 * order of the fp32 additions, not the rounding points. */
mnb_status mnb_matmul(const void* A, mnb_dtype a_dtype, int64_t M, int64_t K,
                      const uint8_t* B_packed, const void* scales, mnb_dtype scale_dtype,
                      const uint8_t* zero_points, int64_t N, int bits, int block_size, void* Y,
                      mnb_dtype y_dtype, void* workspace, size_t workspace_bytes,
                      mnb_stream_t stream);

/* MatMulNBits with int8 activation compute, the accuracy_level=4 mode of the
 * K01 contract ("Qwen3 Missing-Kernel Implementation Plan", row K01), as an
 * explicitly selected entry point (mnb_matmul never quantises activations).
 * Each block of block_size activations of a row of A is quantised
 * symmetrically: sa = max|a| / 127 (binary32 division; 0 for an all-zero
 * block), aq = rint(a / sa) (binary32 quotient, ties to even) clamped to
 * [-127, 127]; then Y[m, n] = sum_b sa_b * scale_b * sum_{k in b} aq_k
 * (code_k - zp_b), the inner sums exact in integers.  Same arguments, layouts
 * and errors as mnb_matmul (no workspace); runs on CUDA cores for any M. */
mnb_status mnb_matmul_int8a(const void* A, mnb_dtype a_dtype, int64_t M, int64_t K,
                            const uint8_t* B_packed, const void* scales, mnb_dtype scale_dtype,
                            const uint8_t* zero_points, int64_t N, int bits, int block_size, void* Y,
                            mnb_dtype y_dtype, mnb_stream_t stream);

/* The dense FFN's fused gate/up projection with SwiGLU, the dense
 * counterpart of the QMoE FC1 (the Qwen3 decoder MLP's gate and up
 * projections share their input): B_packed holds 2I rows [2I, nb, blob]
 * (scales [2I, nb], zero_points [2I, ...] or NULL, layouts as above), the gate
 * and up rows of pair i at rows 2i / 2i+1 (MNB_FC1_INTERLEAVED) or i / I+i
 * (MNB_FC1_CONCAT);
 *   Y[m, i] = silu(g) * up,  g = A[m] . Wgate_i^T,  up = A[m] . Wup_i^T,
 * Y [M, I] in y_dtype.  bits 3 or 4.  One launch: tensor cores for M >= 16
 * with f16/bf16 activations and y_dtype == a_dtype (K a multiple of 8, A
 * 16-byte aligned), CUDA cores otherwise (there the concatenated
 * layout needs rows and scale rows of whole 16-byte units, else
 * MNB_ERR_UNSUPPORTED).  Other arguments, alignment and errors as mnb_matmul. */
mnb_status mnb_gate_up_swiglu(const void* A, mnb_dtype a_dtype, int64_t M, int64_t K,
                              const uint8_t* B_packed, const void* scales, mnb_dtype scale_dtype,
                              const uint8_t* zero_points, int64_t I, int bits, int block_size,
                              mnb_fc1_layout layout, void* Y, mnb_dtype y_dtype, mnb_stream_t stream);

/* ------------------------------------------------------ private prepack */

/* A versioned private layout of one MatMulNBits weight (the "versioned
 * private prepack, cache identity/lifetime and prepack-cost qualification"
 * of "INT3 QMoE CUDA correctness baseline and Qwen experimental results", Not
 * PR2-PR4 Completion; a vectorised private layout, which the same page's
 * Review Fixes and Padding Experiment leaves open).  Version 1:
 *   bytes [0, 128): the header, this struct (the rest zero);
 *   row n at 128 + n * row_stride: the row's codes (C = nb * bs / 32 chunks of
 *   4 * bits bytes), its nb scales, its packed zero points (if any), zeros up
 *   to row_stride, a multiple of 16 bytes.
 * INT4 chunks are stored as in the row-local layout.  An INT3 chunk's 96 bits
 * are regrouped into three little-endian 32-bit words W0, W1, W2: byte b
 * (b = 0..3) of word g < 3 holds code 8g+2b in bits 0-2 and code 8g+2b+1 in
 * bits 3-5; bits 6-7 of byte b of W0 / W1 hold the low two bits of code 24+2b
 * / 25+2b, and bit 6 / 7 of byte b of W2 their third bits.  Scales keep their
 * dtype; zero points keep the row-local LSB-first packing.  Rows are then
 * whole 16-byte units whatever K is: one bulk copy moves a block of rows with
 * its scales and zero points.
 * identity is the caller's key for the source weight (an initializer id, a
 * content hash): mnb_matmul_prepacked checks the device copy of the header
 * against the descriptor it is given (magic, version, identity and shape), so
 * a buffer re-prepacked for another weight, or overwritten, is refused on the
 * device (MNB_ERR_INVALID_ARG in the device error word, Y left untouched)
 * instead of being read as codes.  The buffer stays valid while the caller
 * keeps it; nothing is cached inside the library. */
#define MNB_PREPACK_MAGIC 0x50424E4Du /* "MNBP" little-endian */
#define MNB_PREPACK_VERSION 1u
#define MNB_PREPACK_HEADER_BYTES 128

typedef struct {
    uint32_t magic;      /* MNB_PREPACK_MAGIC */
    uint32_t version;    /* MNB_PREPACK_VERSION */
    int64_t N, K;        /* weight rows and columns */
    int32_t bits;        /* 3 or 4 */
    int32_t block_size;  /* 32, 64 or 128 */
    int32_t scale_dtype; /* mnb_dtype of the scales */
    int32_t has_zp;      /* 1: packed zero points follow the scales */
    int64_t row_stride;  /* bytes per prepacked row, a multiple of 16 */
    int64_t scale_offset; /* bytes from a row's start to its scales */
    int64_t zp_offset;   /* bytes from a row's start to its zero points (-1: none) */
    int64_t bytes;       /* the whole buffer: header + N * row_stride */
    uint64_t identity;   /* the caller's key for the source weight */
} mnb_prepacked_desc;

/* Bytes of a version-1 prepacked buffer for these arguments. */
mnb_status mnb_prepack_size(int64_t N, int64_t K, int bits, int block_size, mnb_dtype scale_dtype,
                            int has_zero_points, size_t* bytes);

/* Rewrites a row-local weight (B_packed, scales, zero_points as in
 * mnb_matmul) into the version-1 layout at `dst` (device memory, 16-byte
 * aligned, dst_bytes >= mnb_prepack_size) with one kernel on `stream`, and
 * fills *desc (host memory) with the header it writes.  bits 3 or 4.  The
 * source is read, not changed; dst must not overlap it. */
mnb_status mnb_prepack(const uint8_t* B_packed, const void* scales, mnb_dtype scale_dtype,
                       const uint8_t* zero_points, int64_t N, int64_t K, int bits, int block_size,
                       uint64_t identity, void* dst, size_t dst_bytes, mnb_prepacked_desc* desc,
                       mnb_stream_t stream);

/* Y[M, N] = A[M, K] . W^T as mnb_matmul, W read from a prepacked buffer
 * described by *desc (host memory, as mnb_prepack filled it).  Runs the
 * CUDA-core GEMV for any M (the decode and small-M shapes the layout is made
 * for); fp32 accumulation, the same exact integer chunk sums as mnb_matmul's
 * CUDA-core path.  MNB_ERR_INVALID_ARG for a descriptor that is not version 1
 * or does not match K. */
mnb_status mnb_matmul_prepacked(const void* A, mnb_dtype a_dtype, int64_t M, int64_t K,
                                const mnb_prepacked_desc* desc, const void* prepacked, void* Y,
                                mnb_dtype y_dtype, mnb_stream_t stream);

/* ------------------------------------------------------------------- QMoE */

/* Bytes of device workspace qmoe_forward needs: the routing tables, the
 * SwiGLU activations between FC1 and FC2 and the FC2 outputs before the
 * combine (the bounded activation tiling of "INT3 QMoE CUDA correctness
 * baseline and Qwen experimental results", Summary).  Depends only on the
 * arguments; writes *bytes, touches no device memory. */
mnb_status qmoe_workspace_size(int64_t T, int64_t H, int64_t I, int64_t E, int k,
                               mnb_dtype act_dtype, size_t* bytes);

/* One QMoE expert-FFN layer ("INT3 QMoE CUDA correctness baseline and Qwen
 * experimental results", Summary and "P1: Compatible QMoE v1 Extension";
 * routing as in "feat(qwen4): component kernels extracted from the brick PRs"):
 *   route:   p = softmax(router_logits[t, :]) in fp32; the k experts with the
 *            largest logits, ties to the lower index; weights p[idx] divided
 *            by their sum when normalize_topk != 0, else p[idx].
 *   FC1:     g, u = the gate and up rows of expert e applied to X[t]
 *            (fc1_w [E, 2I, H/bs, bs*fc1_bits/8], fc1_scales [E, 2I, H/bs],
 *            fc1_zp [E, 2I, ceil((H/bs)*fc1_bits/8)] or NULL).
 *   SwiGLU:  h = silu(g) * u = g * sigmoid(g) * u.
 *   FC2:     o = expert e's down projection of h (fc2_w [E, H, I/bs, bs*fc2_bits/8],
 *            fc2_scales [E, H, I/bs], fc2_zp [E, H, ceil((I/bs)*fc2_bits/8)] or NULL).
 *   combine: Y[t] = sum_{j<k} w[t, j] * o[t, j], ascending j, fp32, then act_dtype.
 * X, Y and the scales have act_dtype (f16 or bf16); router_logits are fp32
 * [T, E].  H and I must be multiples of block_size; 1 <= k <= E <= 1024.
 * Never materialises a dequantised expert matrix in global memory. */
mnb_status qmoe_forward(const void* X, mnb_dtype act_dtype, int64_t T, int64_t H,
                        const float* router_logits, int64_t E, int k, int normalize_topk,
                        const uint8_t* fc1_w, const void* fc1_scales, const uint8_t* fc1_zp,
                        int fc1_bits, const uint8_t* fc2_w, const void* fc2_scales,
                        const uint8_t* fc2_zp, int fc2_bits, int64_t I, int block_size,
                        mnb_fc1_layout fc1_layout, void* Y, void* workspace,
                        size_t workspace_bytes, mnb_stream_t stream);

/* Optional inputs of a QMoE layer ("INT3 QMoE CUDA correctness baseline and
 * Qwen experimental results", Summary: optional biases / zero points /
 * aggregation weights).  Every NULL pointer is an absent input.
 *   fc1_bias     [E, 2I] in act_dtype, rows in the FC1 layout; added to the
 *                gate and up projections before SwiGLU.
 *   fc2_bias     [E, H] in act_dtype; added to each expert's FC2 output
 *                before the combine.
 *   agg_weights  [T, E] in agg_dtype: the combine weight of slot j becomes
 *                agg_weights[t, idx[j]] (the experts are still selected by the
 *                router logits; normalize_topk then has no effect).
 *   logits_dtype dtype of router_logits: MNB_F32, MNB_F16 or MNB_BF16 (the
 *                selection and the softmax use the exactly widened values). */
typedef struct {
    const void* fc1_bias;
    const void* fc2_bias;
    const void* agg_weights;
    mnb_dtype agg_dtype;
    mnb_dtype logits_dtype;
} qmoe_options;

/* qmoe_forward with the optional inputs above (options == NULL: none, fp32
 * logits; the result is then that of qmoe_forward).  router_logits is
 * [T, E] in options->logits_dtype, aligned to its element size; the biases
 * are aligned to 2 bytes, agg_weights to its element size.  Same workspace,
 * layouts, errors and asynchrony as qmoe_forward. */
mnb_status qmoe_forward_ex(const void* X, mnb_dtype act_dtype, int64_t T, int64_t H, const void* router_logits,
                           int64_t E, int k, int normalize_topk, const uint8_t* fc1_w, const void* fc1_scales,
                           const uint8_t* fc1_zp, int fc1_bits, const uint8_t* fc2_w, const void* fc2_scales,
                           const uint8_t* fc2_zp, int fc2_bits, int64_t I, int block_size,
                           mnb_fc1_layout fc1_layout, void* Y, void* workspace, size_t workspace_bytes,
                           const qmoe_options* options, mnb_stream_t stream);

/* qmoe_forward without a workspace argument, for callers that cannot allocate
 * device memory: code that receives only input and output pointers (a plugin
 * or an operator inside another runtime that owns every allocation), code
 * running under a fixed device-memory budget that forbids new allocations,
 * and code that must not call cudaMalloc/cudaFree on its path (they
 * synchronise the device and cannot be recorded in a CUDA graph).  The pages
 * have no counterpart to this entry point; it exists for those callers.
 *
 * Scratch: a fixed 8 MiB array inside the library, one copy on every GPU
 * that loads the library, held until the process exits.  Problems whose
 * qmoe_workspace_size() exceeds 8 MiB return MNB_ERR_WORKSPACE (with the
 * Qwen3-30B-A3B layer, H 2048, I 768, E 128, k 8, that is T <= 92 tokens;
 * T = 1 needs 91 KiB).
 * The first call on a device looks up the array's device address on the
 * current device; make that first call before any stream capture.  Every
 * call uses the same array and leaves its contents behind; nothing in it has
 * to start at zero, but calls that overlap on the GPU (other streams, other
 * host threads) race on it and must be serialised by the caller.  Allocates
 * nothing (no cudaMalloc, cudaFree or allocating library call).  All other
 * arguments, layouts and errors are those of qmoe_forward. */
mnb_status qmoe_forward_static(const void* X, mnb_dtype act_dtype, int64_t T, int64_t H,
                               const float* router_logits, int64_t E, int k, int normalize_topk,
                               const uint8_t* fc1_w, const void* fc1_scales, const uint8_t* fc1_zp,
                               int fc1_bits, const uint8_t* fc2_w, const void* fc2_scales,
                               const uint8_t* fc2_zp, int fc2_bits, int64_t I, int block_size,
                               mnb_fc1_layout fc1_layout, void* Y, mnb_stream_t stream);

/* The routing step alone ("feat(qwen4): component kernels extracted from the
 * brick PRs", MoE routing: softmax over the router logits in fp32, canonical
 * top-k, optional renormalisation; the top-k of QMoE's Summary in "INT3 QMoE
 * CUDA correctness baseline and Qwen experimental results"): logits fp32
 * [T, E] in, topk_idx int32 [T, k] and topk_w fp32 [T, k] out, all device
 * buffers owned by the caller.  Indices are the k largest logits in
 * descending order, ties to the lower expert index; weights as in
 * qmoe_forward.  1 <= k <= E, E <= 1024 (else MNB_ERR_UNSUPPORTED); NaN
 * logits are not supported. */
mnb_status qmoe_route(const float* logits, int64_t T, int64_t E, int k, int normalize_topk,
                      int32_t* topk_idx, float* topk_w, mnb_stream_t stream);

/* Expert-sorted order of routed (token, slot) pairs, the step that lets the
 * prefill run one grouped GEMM per selected expert ("INT3 QMoE CUDA
 * correctness baseline and Qwen experimental results", Not PR2-PR4
 * Completion: the selected-expert prefill): topk_idx int32 [T, k] in (values
 * in [0, E)); counts int32 [E]; offsets int32 [E+1] = exclusive prefix sum of
 * counts; perm int32 [T*k] lists the flat pair index t*k + j grouped by
 * expert, ascending inside an expert (a stable sort).  Device buffers owned by
 * the caller; E <= 1024, T*k < 2^31. */
mnb_status qmoe_permute(const int32_t* topk_idx, int64_t T, int k, int64_t E, int32_t* counts,
                        int32_t* offsets, int32_t* perm, mnb_stream_t stream);

/* ------------------------------------------------------ diagnostics, tools */

/* Row-local LSB-first packing for any width 1..8 ("INT3 QMoE CUDA correctness
 * baseline and Qwen experimental results", "P0: Portable Format and Numerical
 * References": generic pack/unpack for widths 1..8).  Device buffers, caller
 * owned; bits in 1..8 and block_size in {32, 64, 128}, else MNB_ERR_UNSUPPORTED.
 * mnb_unpack_codes: codes uint8 [rows, K] = the raw codes of B_packed [rows,
 * nb, block_size*bits/8] (layout above), bit-exact.
 * mnb_pack_codes: B_packed from codes uint8 [rows, K], each code's low `bits`
 * bits; the padding bits of a partial last block are written as zeros. */
mnb_status mnb_unpack_codes(const uint8_t* B_packed, int64_t rows, int64_t K, int bits,
                            int block_size, uint8_t* codes, mnb_stream_t stream);
mnb_status mnb_pack_codes(const uint8_t* codes, int64_t rows, int64_t K, int bits, int block_size,
                          uint8_t* B_packed, mnb_stream_t stream);

/* Symmetric grouped INT3 round-to-nearest quantisation, the producer policy
 * quoted in "INT3 QMoE CUDA correctness baseline and Qwen experimental
 * results" (Olive summary): for every block of block_size weights of a row,
 * scale = max|w| / 3.5 (binary32) rounded to scale_dtype (nearest, ties to
 * even), code = round(w / stored scale) + 4 (binary32 quotient, ties to even)
 * clamped to 0..7, packed like B_packed above (implicit zero point 4, so
 * (code - 4) * scale reconstructs w); an all-zero block stores scale 1/3.5
 * and code 4.
 *   W          device, [N, K] in w_dtype (f32, f16 or bf16), 16-byte aligned.
 *   B_packed   device, out, [N, K/block_size, 3*block_size/8], 4-byte aligned.
 *   scales     device, out, [N, K/block_size] in scale_dtype, aligned to its
 *              element size.
 * K must be a multiple of block_size (32, 64 or 128), else
 * MNB_ERR_UNSUPPORTED.  Content errors are found on the device: a block with
 * a non-finite weight or stored scale, or a nonzero block whose stored scale
 * rounds to zero (subnormal stored scales are kept), gets codes 4 and sets
 * the device error word to MNB_ERR_CONTENT (read it with
 * mnb_get_last_device_error); the other blocks are unaffected.  Asynchronous
 * on `stream`; the caller owns every buffer. */
mnb_status mnb_quantize_int3(const void* W, mnb_dtype w_dtype, int64_t N, int64_t K, int block_size,
                             uint8_t* B_packed, void* scales, mnb_dtype scale_dtype, mnb_stream_t stream);

/* Host-side content check of one packed projection (host buffers): exact
 * sizes are implied by the arguments; scales must be finite and >= 0; every
 * padding bit of the weights and of the zero points must be zero ("canonical
 * padding" of "INT3 QMoE CUDA correctness baseline...", P0 and P1 sections).
 * Returns MNB_OK or MNB_ERR_CONTENT.  Never called by the compute entry points. */
mnb_status mnb_validate_host(const uint8_t* B_packed, const void* scales, mnb_dtype scale_dtype,
                             const uint8_t* zero_points, int64_t N, int64_t K, int bits,
                             int block_size);

/* Synchronises `stream`, then returns and clears the device error word
 * (MNB_OK when no kernel recorded an error). */
mnb_status mnb_get_last_device_error(mnb_stream_t stream);

/* Diagnostic: enqueues one small kernel that runs the library's bounded
 * on-chip wait on a barrier nothing ever completes, giving up after limit_ns
 * nanoseconds (1e3 .. 1e9, else MNB_ERR_INVALID_ARG).  No copy, tensor-core
 * operation or tensor-memory allocation is in flight while it waits.  The
 * kernel records MNB_ERR_TIMEOUT in the device error word and returns
 * normally, so the context stays usable: it exercises the failure path every
 * pipelined kernel takes when a wait runs out.  The pages have no
 * counterpart; this entry point exists for failure-detection tests. */
mnb_status mnb_diag_wait_timeout(uint64_t limit_ns, mnb_stream_t stream);

/* Static, human-readable name of a status code. */
const char* mnb_status_string(mnb_status s);

#ifdef __cplusplus
}
#endif
#endif /* MNB_H_ */
