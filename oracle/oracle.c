/*
 * oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-purpose CPU restatement of block-quantized weight-only
 * matmul (MatMulNBits) and of the QMoE expert FFN, written in fp64 so that it
 * can serve as the independent reference for the CUDA library.  Only the test
 * suite, __graft_entry__.smoke() and bench.py's CPU-baseline leg may load it.
 * It shares no code, header, table or constant with the CUDA library: formats
 * are decoded bit by bit from their definitions, and every sum runs in
 * ascending index order with no blocking or reordering.
 *
 * Sources restated here (page title, then section):
 *  - "Qwen3 Missing-Kernel Implementation Plan", PR sequence, rows K01-K03:
 *    FP32 A / UINT8 packed B / FP32 per-block scales, bits=4, block_size=32,
 *    implicit zero points, partial last blocks and output tails.
 *  - "INT3 QMoE CUDA correctness baseline and Qwen experimental results"
 *    (onnxruntime PR 33519), Summary and "P0: Portable Format and Numerical
 *    References": row-local LSB-first packing for widths 1..8 (3-bit codes
 *    cross byte boundaries), packed per-row block zero points, offset-4 INT3
 *    decoding; "P1: Compatible QMoE v1 Extension": fused interleaved gate/up
 *    FC1 with SwiGLU, FC2 down projection, routing, weighted combine.  The
 *    quoted Olive summary in the same page gives the INT3 mapping
 *    (code - 4) * scale.
 *  - "feat(qwen4): component kernels extracted from the brick PRs"
 *    (pegainfer PR 1242): MoE routing is an fp32 softmax, a canonical top-k and
 *    an optional renormalisation of the selected probabilities.
 *  - The same page's quoted Olive producer summary (symmetric grouped INT3
 *    round-to-nearest): scale max|w| / 3.5, implicit zero point 4, all-zero
 *    block scale 1/3.5 with code 4, stored-scale rounding, rejection of
 *    non-finite weights or scales and of nonzero blocks whose stored scale
 *    rounds to zero, subnormal stored scales kept.
 *
 * Readings taken where the pages are silent (each one is listed in the design
 * notes): nibble order low-first (even k in the low nibble); implicit zero point
 * 2^(bits-1) for every width; SwiGLU is silu(gate) * up with no bias, clamp or
 * alpha (parity unpinned beyond that definition); top-k ranks the fp32 logits
 * with ties going to the lower expert index.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F32 0
#define ORC_F16 1
#define ORC_BF16 2

#define ORC_FC1_INTERLEAVED 0
#define ORC_FC1_CONCAT 1

/* ---------------------------------------------------------------- scalars */

/* IEEE 754 binary16 -> double, exact: sign, 5-bit exponent (bias 15), 10-bit
 * fraction; exponent 0 is the subnormal range m * 2^-24. */
static double f16_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m + 1024), e - 25);
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32: widen by appending 16 zero
 * bits, then widen the binary32 exactly. */
static double bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load_elem(const void* p, int dtype, int64_t i) {
    if (dtype == ORC_F32) return (double)((const float*)p)[i];
    if (dtype == ORC_F16) return f16_to_double(((const uint16_t*)p)[i]);
    return bf16_to_double(((const uint16_t*)p)[i]);
}

/* ------------------------------------------------------ packed bit streams */

/* Bit i of a row-local LSB-first stream lives in byte i/8 at bit i%8. */
static int stream_bit(const uint8_t* stream, int64_t i) {
    return (stream[i >> 3] >> (i & 7)) & 1;
}

/* Code j of width `bits`: stream bits bits*j .. bits*j+bits-1, least
 * significant bit first.  A 3-bit code may straddle two bytes. */
static int stream_code(const uint8_t* stream, int64_t j, int bits) {
    int q = 0;
    for (int t = 0; t < bits; ++t) q |= stream_bit(stream, (int64_t)bits * j + t) << t;
    return q;
}

static void stream_put(uint8_t* stream, int64_t j, int bits, int q) {
    for (int t = 0; t < bits; ++t) {
        int64_t i = (int64_t)bits * j + t;
        if ((q >> t) & 1) stream[i >> 3] |= (uint8_t)(1u << (i & 7));
    }
}

/* Layout of one packed weight row: nb = ceil(K/bs) blobs of bs*bits/8 bytes.
 * Code k is entry k % bs of blob k / bs. */
static int64_t n_blocks(int64_t K, int bs) { return (K + bs - 1) / bs; }
static int64_t blob_bytes(int bits, int bs) { return (int64_t)bs * bits / 8; }
static int64_t zp_row_bytes(int64_t nb, int bits) { return (nb * bits + 7) / 8; }

static int weight_code(const uint8_t* row, int64_t k, int bits, int bs) {
    const uint8_t* blob = row + (k / bs) * blob_bytes(bits, bs);
    return stream_code(blob, k % bs, bits);
}

static int check_format(int bits, int bs) {
    if (bits < 1 || bits > 8) return 1;
    if (bs < 8 || (bs * bits) % 8 != 0) return 1;
    return 0;
}

/* codes[n*K + k] = raw code of row n, column k (k < K). */
int orc_unpack_codes(const uint8_t* packed, int64_t rows, int64_t K, int bits, int bs,
                     uint8_t* codes) {
    if (check_format(bits, bs) || rows < 0 || K < 0) return 1;
    int64_t rb = n_blocks(K, bs) * blob_bytes(bits, bs);
    for (int64_t n = 0; n < rows; ++n)
        for (int64_t k = 0; k < K; ++k)
            codes[n * K + k] = (uint8_t)weight_code(packed + n * rb, k, bits, bs);
    return 0;
}

/* Canonical packing: every padding bit is zero. */
int orc_pack_codes(const uint8_t* codes, int64_t rows, int64_t K, int bits, int bs,
                   uint8_t* packed) {
    if (check_format(bits, bs) || rows < 0 || K < 0) return 1;
    int64_t bb = blob_bytes(bits, bs);
    int64_t rb = n_blocks(K, bs) * bb;
    memset(packed, 0, (size_t)(rows * rb));
    for (int64_t n = 0; n < rows; ++n)
        for (int64_t k = 0; k < K; ++k) {
            int q = codes[n * K + k];
            if (q < 0 || q >= (1 << bits)) return 1;
            stream_put(packed + n * rb + (k / bs) * bb, k % bs, bits, q);
        }
    return 0;
}

/* Zero points: one code per block, row-local LSB-first with the weight width,
 * ceil(nb*bits/8) bytes per row. */
int orc_unpack_zero_points(const uint8_t* zp, int64_t rows, int64_t nb, int bits,
                           uint8_t* zcodes) {
    if (bits < 1 || bits > 8) return 1;
    int64_t zb = zp_row_bytes(nb, bits);
    for (int64_t n = 0; n < rows; ++n)
        for (int64_t b = 0; b < nb; ++b) zcodes[n * nb + b] = (uint8_t)stream_code(zp + n * zb, b, bits);
    return 0;
}

int orc_pack_zero_points(const uint8_t* zcodes, int64_t rows, int64_t nb, int bits, uint8_t* zp) {
    if (bits < 1 || bits > 8) return 1;
    int64_t zb = zp_row_bytes(nb, bits);
    memset(zp, 0, (size_t)(rows * zb));
    for (int64_t n = 0; n < rows; ++n)
        for (int64_t b = 0; b < nb; ++b) {
            int q = zcodes[n * nb + b];
            if (q < 0 || q >= (1 << bits)) return 1;
            stream_put(zp + n * zb, b, bits, q);
        }
    return 0;
}

/* --------------------------------------------------------------- dequant */

/* w[k] = scale[n, k/bs] * (code[n, k] - z[n, k/bs]) for k < K, with z the
 * explicit zero-point code when zp != NULL and 2^(bits-1) otherwise (8 for
 * INT4, 4 for INT3: the offset-4 decoding (code - 4) * scale). */
static void dequant_row(const uint8_t* packed, const void* scales, int s_dtype,
                        const uint8_t* zp, int64_t n, int64_t K, int bits, int bs,
                        double* w) {
    int64_t nb = n_blocks(K, bs);
    const uint8_t* row = packed + n * nb * blob_bytes(bits, bs);
    const uint8_t* zrow = zp ? zp + n * zp_row_bytes(nb, bits) : NULL;
    for (int64_t k = 0; k < K; ++k) {
        int64_t b = k / bs;
        double s = load_elem(scales, s_dtype, n * nb + b);
        double z = zrow ? (double)stream_code(zrow, b, bits) : (double)(1 << (bits - 1));
        double q = (double)weight_code(row, k, bits, bs);
        w[k] = s * (q - z);
    }
}

int orc_dequantize(const uint8_t* packed, const void* scales, int s_dtype, const uint8_t* zp,
                   int64_t N, int64_t K, int bits, int bs, double* W) {
    if (check_format(bits, bs) || N < 0 || K < 0) return 1;
    for (int64_t n = 0; n < N; ++n) dequant_row(packed, scales, s_dtype, zp, n, K, bits, bs, W + n * K);
    return 0;
}

/* ------------------------------------------------------------ matmul */

/* Y[m, n] = sum_{k<K} A[m, k] * w[n, k], ascending k, fp64.
 * Only the rows listed in `mrows` (all M rows when mrows == NULL) are computed;
 * Y has one row per computed A row.  Output rows are independent, so the work
 * is split over threads by output column n with no change to any sum. */
int orc_mnb_matmul(const void* A, int a_dtype, int64_t M, int64_t K,
                   const uint8_t* packed, const void* scales, int s_dtype, const uint8_t* zp,
                   int64_t N, int bits, int bs, const int64_t* mrows, int64_t n_mrows,
                   double* Y, int threads) {
    if (check_format(bits, bs) || M < 0 || K < 0 || N < 0) return 1;
    int64_t rows = mrows ? n_mrows : M;
    int bad = 0;
    if (threads < 1) threads = 1;
#pragma omp parallel num_threads(threads)
    {
        double* w = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
        if (!w) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(static)
            for (int64_t n = 0; n < N; ++n) {
                dequant_row(packed, scales, s_dtype, zp, n, K, bits, bs, w);
                for (int64_t i = 0; i < rows; ++i) {
                    int64_t m = mrows ? mrows[i] : i;
                    double acc = 0.0;
                    for (int64_t k = 0; k < K; ++k) acc += load_elem(A, a_dtype, m * K + k) * w[k];
                    Y[i * N + n] = acc;
                }
            }
            free(w);
        }
    }
    return bad;
}

/* MatMulNBits with accuracy_level=4 ("Qwen3 Missing-Kernel Implementation
 * Plan", row K01: the audited contract carries accuracy_level=4, which ONNX
 * Runtime takes as int8 activation compute).  Each block of bs activations of
 * a row (the weight's K blocks) is quantised symmetrically:
 *   amax = max |a| over the block's K entries (binary32),
 *   sa   = amax / 127 (binary32 division; 0 when amax is 0),
 *   aq   = rint(a / sa) clamped to [-127, 127] (binary32 quotient, ties to
 *          even; 0 when sa is 0),
 * and Y[m, n] = sum_b sa_b * sw_b * sum_{k in b} aq_k (q_k - z_b), the inner
 * sums exact integers, the rest in fp64, ascending b. */
void orc_quantize_a_int8(const void* A, int a_dtype, int64_t M, int64_t K, int bs, int8_t* aq, float* sa) {
    int64_t nb = n_blocks(K, bs);
    for (int64_t m = 0; m < M; ++m)
        for (int64_t b = 0; b < nb; ++b) {
            float amax = 0.0f;
            for (int64_t k = b * bs; k < (b + 1) * bs && k < K; ++k) {
                float v = (float)load_elem(A, a_dtype, m * K + k);
                float av = v < 0.0f ? -v : v;
                if (av > amax) amax = av;
            }
            float s = amax / 127.0f;
            sa[m * nb + b] = s;
            for (int64_t k = b * bs; k < (b + 1) * bs; ++k) {
                int8_t q = 0;
                if (k < K && s != 0.0f) {
                    float r = rintf((float)load_elem(A, a_dtype, m * K + k) / s);
                    if (r > 127.0f) r = 127.0f;
                    if (r < -127.0f) r = -127.0f;
                    q = (int8_t)r;
                }
                if (k < K) aq[m * K + k] = q;
            }
        }
}

int orc_mnb_matmul_int8a(const void* A, int a_dtype, int64_t M, int64_t K, const uint8_t* packed,
                         const void* scales, int s_dtype, const uint8_t* zp, int64_t N, int bits, int bs,
                         double* Y, int threads) {
    if (check_format(bits, bs) || M < 0 || K < 0 || N < 0) return 1;
    int64_t nb = n_blocks(K, bs);
    int8_t* aq = (int8_t*)malloc((size_t)(M * K > 0 ? M * K : 1));
    float* sa = (float*)malloc(sizeof(float) * (size_t)(M * nb > 0 ? M * nb : 1));
    if (!aq || !sa) { free(aq); free(sa); return 1; }
    orc_quantize_a_int8(A, a_dtype, M, K, bs, aq, sa);
    int64_t rb = nb * blob_bytes(bits, bs), zr = zp_row_bytes(nb, bits);
    if (threads < 1) threads = 1;
#pragma omp parallel for num_threads(threads) schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        const uint8_t* row = packed + n * rb;
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                int64_t z = zp ? stream_code(zp + n * zr, b, bits) : (1 << (bits - 1));
                int64_t isum = 0;
                for (int64_t k = b * bs; k < (b + 1) * bs && k < K; ++k)
                    isum += (int64_t)aq[m * K + k] * (stream_code(row, k, bits) - z);
                acc += (double)sa[m * nb + b] * load_elem(scales, s_dtype, n * nb + b) * (double)isum;
            }
            Y[m * N + n] = acc;
        }
    }
    free(aq);
    free(sa);
    return 0;
}

/* ------------------------------------------------------------ routing */

/* Top-k by fp32 logit value: repeatedly take the largest unselected logit; a
 * later index replaces the current choice only when strictly greater, so ties
 * go to the lower expert index.  Probabilities are the softmax of the row in
 * fp64; with `normalize` the k selected probabilities are divided by their own
 * sum (the renormalised top-k of the routing page), else they are returned as
 * softmax probabilities over all E experts. */
static void route_token(const float* row, int64_t E, int k, int normalize, int32_t* idx,
                        double* w, unsigned char* taken) {
    memset(taken, 0, (size_t)E);
    for (int j = 0; j < k; ++j) {
        int64_t best = -1;
        for (int64_t e = 0; e < E; ++e) {
            if (taken[e]) continue;
            if (best < 0 || row[e] > row[best]) best = e;
        }
        taken[best] = 1;
        idx[j] = (int32_t)best;
    }
    double lmax = row[0];
    for (int64_t e = 1; e < E; ++e)
        if (row[e] > lmax) lmax = row[e];
    double denom = 0.0;
    if (normalize) {
        for (int j = 0; j < k; ++j) denom += exp((double)row[idx[j]] - lmax);
    } else {
        for (int64_t e = 0; e < E; ++e) denom += exp((double)row[e] - lmax);
    }
    for (int j = 0; j < k; ++j) w[j] = exp((double)row[idx[j]] - lmax) / denom;
}

int orc_route(const float* logits, int64_t T, int64_t E, int k, int normalize, int32_t* idx,
              double* w) {
    if (T < 0 || E < 1 || k < 1 || k > E) return 1;
    unsigned char* taken = (unsigned char*)malloc((size_t)E);
    if (!taken) return 1;
    for (int64_t t = 0; t < T; ++t) route_token(logits + t * E, E, k, normalize, idx + t * k, w + t * k, taken);
    free(taken);
    return 0;
}

/* Expert-sorted order of the (token, slot) pairs: counts[e] pairs go to expert
 * e, offsets is the exclusive prefix sum (E+1 entries), and perm lists the
 * flattened pair index t*k+j grouped by expert, ascending within an expert. */
int orc_permute(const int32_t* idx, int64_t T, int k, int64_t E, int32_t* counts,
                int32_t* offsets, int32_t* perm) {
    for (int64_t e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t p = 0; p < T * k; ++p) {
        if (idx[p] < 0 || idx[p] >= E) return 1;
        counts[idx[p]] += 1;
    }
    offsets[0] = 0;
    for (int64_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int64_t pos = 0;
    for (int64_t e = 0; e < E; ++e)
        for (int64_t p = 0; p < T * k; ++p)
            if (idx[p] == e) perm[pos++] = (int32_t)p;
    return 0;
}

/* --------------------------------------------------------------- QMoE */

/* silu(g) * u = g * sigmoid(g) * u */
static double swiglu(double g, double u) { return g / (1.0 + exp(-g)) * u; }

/* The dense FFN's fused gate/up projection with SwiGLU (the gate+up GEMV of a
 * Qwen3 decoder layer, the dense counterpart of the QMoE FC1): packed
 * [2I, K] with the gate and up rows of pair p at rows 2p / 2p+1 (interleaved)
 * or p / I+p (concatenated); Y[m, p] = swiglu(g, u) with g, u the two rows'
 * products with A[m] (steps 1-4 of the matmul above, fp64, ascending k). */
int orc_gate_up_swiglu(const void* A, int a_dtype, int64_t M, int64_t K, const uint8_t* packed,
                       const void* scales, int s_dtype, const uint8_t* zp, int64_t I, int bits, int bs,
                       int layout, double* Y, int threads) {
    if (check_format(bits, bs) || M < 0 || K < 0 || I < 1) return 1;
    if (layout != ORC_FC1_INTERLEAVED && layout != ORC_FC1_CONCAT) return 1;
    int bad = 0;
    if (threads < 1) threads = 1;
#pragma omp parallel num_threads(threads)
    {
        double* wg = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
        double* wu = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
        if (!wg || !wu) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(static)
            for (int64_t p = 0; p < I; ++p) {
                int64_t rg = layout == ORC_FC1_INTERLEAVED ? 2 * p : p;
                int64_t ru = layout == ORC_FC1_INTERLEAVED ? 2 * p + 1 : I + p;
                dequant_row(packed, scales, s_dtype, zp, rg, K, bits, bs, wg);
                dequant_row(packed, scales, s_dtype, zp, ru, K, bits, bs, wu);
                for (int64_t m = 0; m < M; ++m) {
                    double g = 0.0, u = 0.0;
                    for (int64_t k = 0; k < K; ++k) g += load_elem(A, a_dtype, m * K + k) * wg[k];
                    for (int64_t k = 0; k < K; ++k) u += load_elem(A, a_dtype, m * K + k) * wu[k];
                    Y[m * I + p] = g / (1.0 + exp(-g)) * u;
                }
            }
        }
        free(wg);
        free(wu);
    }
    return bad;
}

/* One QMoE FFN layer for the listed tokens (all T when tokens == NULL).
 * Expert tensors are stacked on a leading expert axis:
 *   fc1_w [E, 2I, H/bs, bs*fc1_bits/8], fc1_scales [E, 2I, H/bs], fc1_zp [E, 2I, ceil((H/bs)*fc1_bits/8)]
 *   fc2_w [E, H, I/bs, bs*fc2_bits/8],  fc2_scales [E, H, I/bs],  fc2_zp [E, H, ceil((I/bs)*fc2_bits/8)]
 * Scales have the activation dtype.  FC1 row pairs: interleaved layout puts
 * gate_i at row 2i and up_i at row 2i+1; the concatenated layout puts gate_i at
 * row i and up_i at row I+i.  Y[t] = sum_j w[t,j] * FC2_e(swiglu(FC1_e(x_t))),
 * ascending slot j, everything in fp64. */
/* One QMoE layer with the optional inputs of the QMoE contract ("INT3 QMoE CUDA
 * correctness baseline and Qwen experimental results", Summary: routing, fused
 * gate/up SwiGLU, the down projection, optional biases / zero points /
 * aggregation weights).  logits [T, E] in logits_dtype, widened exactly;
 * fc1_bias [E, 2I] (rows in the FC1 layout) and fc2_bias [E, H] in act_dtype,
 * added to the projections before SwiGLU and before the combine; agg [T, E] in
 * agg_dtype: when given, the combine weight of slot j is agg[t, idx[j]]
 * (selection still by the logits), else the routing weight.  Every NULL
 * optional input is absent. */
int orc_qmoe_ex(const void* X, int act_dtype, int64_t T, int64_t H, const void* logits, int logits_dtype,
                int64_t E, int k, int normalize, const uint8_t* fc1_w, const void* fc1_s, const uint8_t* fc1_zp,
                const void* fc1_bias, int fc1_bits, const uint8_t* fc2_w, const void* fc2_s, const uint8_t* fc2_zp,
                const void* fc2_bias, int fc2_bits, const void* agg, int agg_dtype, int64_t I, int bs,
                int fc1_layout, const int64_t* tokens, int64_t n_tokens, double* Y, int threads) {
    if (check_format(fc1_bits, bs) || check_format(fc2_bits, bs)) return 1;
    if (T < 0 || H < 1 || I < 1 || E < 1 || k < 1 || k > E) return 1;
    if (fc1_layout != ORC_FC1_INTERLEAVED && fc1_layout != ORC_FC1_CONCAT) return 1;
    int64_t rows = tokens ? n_tokens : T;
    int64_t nb1 = n_blocks(H, bs), nb2 = n_blocks(I, bs);
    int64_t w1_stride = 2 * I * nb1 * blob_bytes(fc1_bits, bs);
    int64_t s1_stride = 2 * I * nb1;
    int64_t z1_stride = 2 * I * zp_row_bytes(nb1, fc1_bits);
    int64_t w2_stride = H * nb2 * blob_bytes(fc2_bits, bs);
    int64_t s2_stride = H * nb2;
    int64_t z2_stride = H * zp_row_bytes(nb2, fc2_bits);
    int64_t s_elem = act_dtype == ORC_F32 ? 4 : 2;
    int bad = 0;
    if (threads < 1) threads = 1;
#pragma omp parallel num_threads(threads)
    {
        double* x = (double*)malloc(sizeof(double) * (size_t)H);
        double* wg = (double*)malloc(sizeof(double) * (size_t)H);
        double* wu = (double*)malloc(sizeof(double) * (size_t)H);
        double* h = (double*)malloc(sizeof(double) * (size_t)I);
        double* w2 = (double*)malloc(sizeof(double) * (size_t)I);
        float* lrow = (float*)malloc(sizeof(float) * (size_t)E);
        int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)k);
        double* rw = (double*)malloc(sizeof(double) * (size_t)k);
        unsigned char* taken = (unsigned char*)malloc((size_t)E);
        if (!x || !wg || !wu || !h || !w2 || !lrow || !idx || !rw || !taken) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t i = 0; i < rows; ++i) {
                int64_t t = tokens ? tokens[i] : i;
                double* y = Y + i * H;
                for (int64_t c = 0; c < H; ++c) {
                    x[c] = load_elem(X, act_dtype, t * H + c);
                    y[c] = 0.0;
                }
                for (int64_t e = 0; e < E; ++e) lrow[e] = (float)load_elem(logits, logits_dtype, t * E + e);
                route_token(lrow, E, k, normalize, idx, rw, taken);
                if (agg)
                    for (int j = 0; j < k; ++j) rw[j] = load_elem(agg, agg_dtype, t * E + idx[j]);
                for (int j = 0; j < k; ++j) {
                    int64_t e = idx[j];
                    const uint8_t* W1 = fc1_w + e * w1_stride;
                    const char* S1 = (const char*)fc1_s + e * s1_stride * s_elem;
                    const uint8_t* Z1 = fc1_zp ? fc1_zp + e * z1_stride : NULL;
                    const uint8_t* W2 = fc2_w + e * w2_stride;
                    const char* S2 = (const char*)fc2_s + e * s2_stride * s_elem;
                    const uint8_t* Z2 = fc2_zp ? fc2_zp + e * z2_stride : NULL;
                    for (int64_t c = 0; c < I; ++c) {
                        int64_t rg = fc1_layout == ORC_FC1_INTERLEAVED ? 2 * c : c;
                        int64_t ru = fc1_layout == ORC_FC1_INTERLEAVED ? 2 * c + 1 : I + c;
                        dequant_row(W1, S1, act_dtype, Z1, rg, H, fc1_bits, bs, wg);
                        dequant_row(W1, S1, act_dtype, Z1, ru, H, fc1_bits, bs, wu);
                        double g = 0.0, u = 0.0;
                        for (int64_t q = 0; q < H; ++q) g += x[q] * wg[q];
                        for (int64_t q = 0; q < H; ++q) u += x[q] * wu[q];
                        if (fc1_bias) {
                            g += load_elem(fc1_bias, act_dtype, e * 2 * I + rg);
                            u += load_elem(fc1_bias, act_dtype, e * 2 * I + ru);
                        }
                        h[c] = swiglu(g, u);
                    }
                    for (int64_t r = 0; r < H; ++r) {
                        dequant_row(W2, S2, act_dtype, Z2, r, I, fc2_bits, bs, w2);
                        double o = 0.0;
                        for (int64_t q = 0; q < I; ++q) o += h[q] * w2[q];
                        if (fc2_bias) o += load_elem(fc2_bias, act_dtype, e * H + r);
                        y[r] += rw[j] * o;
                    }
                }
            }
        }
        free(x); free(wg); free(wu); free(h); free(w2); free(lrow); free(idx); free(rw); free(taken);
    }
    return bad;
}

int orc_qmoe(const void* X, int act_dtype, int64_t T, int64_t H, const float* logits, int64_t E,
             int k, int normalize, const uint8_t* fc1_w, const void* fc1_s, const uint8_t* fc1_zp,
             int fc1_bits, const uint8_t* fc2_w, const void* fc2_s, const uint8_t* fc2_zp,
             int fc2_bits, int64_t I, int bs, int fc1_layout, const int64_t* tokens, int64_t n_tokens,
             double* Y, int threads) {
    return orc_qmoe_ex(X, act_dtype, T, H, logits, ORC_F32, E, k, normalize, fc1_w, fc1_s, fc1_zp, NULL,
                       fc1_bits, fc2_w, fc2_s, fc2_zp, NULL, fc2_bits, NULL, ORC_F32, I, bs, fc1_layout, tokens,
                       n_tokens, Y, threads);
}

/* --------------------------------------------- INT3 producer (quantizer) */

/* binary32 -> binary16 bit pattern, rounded to nearest with ties to even (the
 * IEEE 754 default): normal values 2^-14 .. 65504 keep 10 fraction bits,
 * smaller ones become subnormals m * 2^-24, values that round past 65504
 * become infinity.  A subnormal that rounds up to m = 1024 is exactly the
 * smallest normal, whose encoding is the same integer. */
static uint16_t float_to_f16_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    const uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    const double a = fabs((double)f);
    if (f != f) return (uint16_t)(sign | 0x7E00u);
    if (isinf(a)) return (uint16_t)(sign | 0x7C00u);
    if (a < ldexp(1.0, -14)) return (uint16_t)(sign | (uint16_t)nearbyint(ldexp(a, 24)));
    int e;
    frexp(a, &e); /* a in [2^(e-1), 2^e) */
    int E = e - 1;
    double m = nearbyint(ldexp(a, 10 - E)); /* 1024 .. 2048 */
    if (m == 2048.0) {
        m = 1024.0;
        ++E;
    }
    if (E > 15) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(m - 1024.0));
}

/* binary32 -> bfloat16 bit pattern: the upper 16 bits, the dropped 16 rounded
 * to nearest with ties to even (a carry may reach the exponent, and past the
 * largest finite value gives infinity); NaN stays NaN. */
static uint16_t float_to_bf16_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if (f != f) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t hi = u >> 16;
    const uint32_t low = u & 0xFFFFu;
    if (low > 0x8000u || (low == 0x8000u && (hi & 1u))) ++hi;
    return (uint16_t)hi;
}

/* Exported for the pins: the rounding helpers above over arrays. */
int orc_round_to_half_bits(const float* x, int64_t n, int bf16, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = bf16 ? float_to_bf16_bits(x[i]) : float_to_f16_bits(x[i]);
    return 0;
}

/* Symmetric grouped INT3 round-to-nearest, as the Olive producer summary
 * quoted in "INT3 QMoE CUDA correctness baseline and Qwen experimental
 * results" states it: for each block of bs weights of a row, scale = max|w| / 3.5,
 * rounded to the stored scale dtype; code = round(w / stored scale) + 4,
 * clamped to 0..7, so that (code - 4) * scale reconstructs w; an all-zero
 * block stores scale 1/3.5 and code 4.  A block with a non-finite weight, a
 * non-finite stored scale, or a nonzero block whose stored scale rounds to
 * zero is rejected: bad[n * nb + b] = 1, its codes are then 4.  Subnormal
 * stored scales are kept.  The arithmetic is binary32 (max|w| exact, each
 * division correctly rounded, rounding to an integer with ties to even).
 * Requires K % bs == 0; W is [N, K] in w_dtype, packed [N, nb, 3*bs/8],
 * scales [N, nb] in s_dtype. */
int orc_quantize_int3(const void* W, int w_dtype, int64_t N, int64_t K, int bs, int s_dtype,
                      uint8_t* packed, void* scales, uint8_t* bad) {
    if (check_format(3, bs) || K % bs != 0) return 1;
    const int64_t nb = K / bs, blob = blob_bytes(3, bs), rb = nb * blob;
    memset(packed, 0, (size_t)(N * rb));
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t b = 0; b < nb; ++b) {
            const int64_t w0 = n * K + b * bs;
            float amax = 0.0f;
            int nonfinite = 0;
            for (int i = 0; i < bs; ++i) {
                const float w = (float)load_elem(W, w_dtype, w0 + i);
                if (!isfinite(w))
                    nonfinite = 1;
                else if (fabsf(w) > amax)
                    amax = fabsf(w);
            }
            const float s = amax > 0.0f ? amax / 3.5f : 1.0f / 3.5f;
            float stored;
            if (s_dtype == ORC_F32) {
                ((float*)scales)[n * nb + b] = s;
                stored = s;
            } else if (s_dtype == ORC_F16) {
                const uint16_t h = float_to_f16_bits(s);
                ((uint16_t*)scales)[n * nb + b] = h;
                stored = (float)f16_to_double(h);
            } else {
                const uint16_t h = float_to_bf16_bits(s);
                ((uint16_t*)scales)[n * nb + b] = h;
                stored = (float)bf16_to_double(h);
            }
            const int rejected = nonfinite || !isfinite(stored) || (amax > 0.0f && stored == 0.0f);
            bad[n * nb + b] = (uint8_t)rejected;
            uint8_t* blk = packed + n * rb + b * blob;
            for (int i = 0; i < bs; ++i) {
                int q = 4;
                if (!rejected) {
                    const float w = (float)load_elem(W, w_dtype, w0 + i);
                    const float r = rintf(w / stored);
                    q = r < -4.0f ? 0 : r > 3.0f ? 7 : (int)r + 4;
                }
                stream_put(blk, i, 3, q);
            }
        }
    }
    return 0;
}

/* ------------------------------------------------- version-1 prepacked layout
 *
 * The library's private prepacked form of a weight (its own format, restated
 * here from its definition so the tests can check the bytes the library
 * writes): a 128-byte little-endian header {u32 magic "MNBP", u32 version 1,
 * i64 N, i64 K, i32 bits, i32 block_size, i32 scale dtype, i32 has_zp,
 * i64 row_stride, i64 scale_offset, i64 zp_offset (-1: none), i64 bytes,
 * u64 identity, zeros}, then N rows of row_stride bytes: the row's 32-code
 * chunks (INT4: the stored bytes; INT3: regrouped, below), its scale bytes,
 * its zero-point bytes, zeros up to a multiple of 16 bytes.
 * INT3 chunk (codes c_0 .. c_31), three 32-bit little-endian words W_0..W_2:
 * in byte b of W_g (g < 3), bits 0-2 = c_{8g+2b}, bits 3-5 = c_{8g+2b+1};
 * bits 6-7 of byte b of W_0 = low two bits of c_{24+2b}, of W_1 = low two bits
 * of c_{25+2b}; bit 6 of byte b of W_2 = bit 2 of c_{24+2b}, bit 7 = bit 2 of
 * c_{25+2b}.  Parity unpinned against the pages: the layout is the library's
 * own; the tests pin it by decoding it back to the row-local codes. */
static void put_le(uint8_t* p, uint64_t v, int n) {
    for (int i = 0; i < n; ++i) p[i] = (uint8_t)(v >> (8 * i));
}

int64_t orc_prepack_size(int64_t N, int64_t K, int bits, int bs, int s_dtype, int has_zp) {
    const int64_t nb = n_blocks(K, bs);
    const int64_t raw = nb * blob_bytes(bits, bs) + nb * (s_dtype == ORC_F32 ? 4 : 2) +
                        (has_zp ? zp_row_bytes(nb, bits) : 0);
    const int64_t stride = (raw + 15) / 16 * 16;
    return 128 + N * stride;
}

int orc_prepack(const uint8_t* packed, const void* scales, int s_dtype, const uint8_t* zp, int64_t N,
                int64_t K, int bits, int bs, uint64_t identity, uint8_t* out) {
    if ((bits != 3 && bits != 4) || (bs != 32 && bs != 64 && bs != 128)) return 1;
    const int64_t nb = n_blocks(K, bs);
    const int64_t rb = nb * blob_bytes(bits, bs);
    const int64_t ss = s_dtype == ORC_F32 ? 4 : 2;
    const int64_t zr = zp_row_bytes(nb, bits);
    const int64_t total = orc_prepack_size(N, K, bits, bs, s_dtype, zp != NULL);
    const int64_t stride = (total - 128) / N;
    const int64_t scale_off = rb;
    const int64_t zp_off = zp ? scale_off + nb * ss : -1;
    memset(out, 0, (size_t)total);
    put_le(out + 0, 0x50424E4Du, 4);
    put_le(out + 4, 1, 4);
    put_le(out + 8, (uint64_t)N, 8);
    put_le(out + 16, (uint64_t)K, 8);
    put_le(out + 24, (uint64_t)bits, 4);
    put_le(out + 28, (uint64_t)bs, 4);
    put_le(out + 32, (uint64_t)s_dtype, 4);
    put_le(out + 36, zp != NULL, 4);
    put_le(out + 40, (uint64_t)stride, 8);
    put_le(out + 48, (uint64_t)scale_off, 8);
    put_le(out + 56, (uint64_t)zp_off, 8);
    put_le(out + 64, (uint64_t)total, 8);
    put_le(out + 72, identity, 8);
    for (int64_t n = 0; n < N; ++n) {
        const uint8_t* src = packed + n * rb;
        uint8_t* row = out + 128 + n * stride;
        for (int64_t c = 0; c < nb * bs / 32; ++c) {
            uint8_t* ch = row + c * 4 * bits;
            if (bits == 4) {
                memcpy(ch, src + c * 16, 16);
                continue;
            }
            /* code j of the chunk: stream position 32c + j of the row */
            int q[32];
            for (int j = 0; j < 32; ++j) q[j] = stream_code(src, 32 * c + j, 3);
            for (int g = 0; g < 3; ++g)
                for (int b = 0; b < 4; ++b) ch[4 * g + b] = (uint8_t)(q[8 * g + 2 * b] | (q[8 * g + 2 * b + 1] << 3));
            for (int b = 0; b < 4; ++b) {
                const int e = q[24 + 2 * b], d = q[25 + 2 * b];
                ch[0 + b] |= (uint8_t)((e & 3) << 6);
                ch[4 + b] |= (uint8_t)((d & 3) << 6);
                ch[8 + b] |= (uint8_t)(((e >> 2) & 1) << 6 | ((d >> 2) & 1) << 7);
            }
        }
        memcpy(row + scale_off, (const uint8_t*)scales + n * nb * ss, (size_t)(nb * ss));
        if (zp) memcpy(row + zp_off, zp + n * zr, (size_t)zr);
    }
    return 0;
}
