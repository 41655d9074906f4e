// quant.cu -- the producer side of the INT3 format: symmetric grouped
// round-to-nearest quantisation of a dense weight matrix W [N, K] into packed
// INT3 codes [N, nb, 3*bs/8] and per-block scales [N, nb].  The policy is the
// Olive producer summary quoted in "INT3 QMoE CUDA correctness baseline and
// Qwen experimental results": per block of bs weights, scale = max|w| / 3.5
// rounded to the stored scale dtype, code = round(w / stored scale) + 4
// clamped to 0..7, an all-zero block storing scale 1/3.5 with code 4; blocks
// with a non-finite weight or stored scale, or a nonzero block whose stored
// scale rounds to zero, are rejected.  Codes are packed row-local LSB-first
// (the same page, "P0: Portable Format and Numerical References").
//
// One thread per 32-code chunk: 32 codes are 96 bits = 12 bytes, so every
// chunk starts on a byte and the chunks of a row are independent.  The bs/32
// threads of one block are adjacent lanes and combine max|w| and the rejection
// flag with shuffles.  The kernel streams W once (16-byte loads) and writes
// 3/8 byte per weight plus the scales: it is bound by HBM.
#include "common.cuh"
#include "kernels.h"

namespace mnb {

namespace {

constexpr int kQuantThreads = 256;

// The raw bytes of chunk c (elements 32c .. 32c+31 of W's flat storage) as
// 16-byte words, and the same 32 weights widened to binary32.
template <int WD>
constexpr int chunk_words() { return WD == kF32 ? 8 : 4; }

// Weight j of a chunk held as raw 16-byte words, widened to binary32 (exact).
template <int WD>
__device__ __forceinline__ float weight_at(const uint4 (&raw)[chunk_words<WD>()], int j) {
    if constexpr (WD == kF32) {
        const uint4 v = raw[j >> 2];
        const uint32_t u = (j & 3) == 0 ? v.x : (j & 3) == 1 ? v.y : (j & 3) == 2 ? v.z : v.w;
        return __uint_as_float(u);
    } else {
        const uint4 v = raw[j >> 3];
        const int k = (j >> 1) & 3;
        const uint32_t u = k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
        const uint32_t h = (j & 1) ? (u >> 16) : (u & 0xFFFFu);
        if constexpr (WD == kF16) return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
        return __uint_as_float(h << 16);  // bfloat16 is the upper half of a binary32
    }
}

// max |w| over the finite weights of the chunk, and whether any weight is not finite.
template <int WD>
__device__ __forceinline__ float chunk_amax(const uint4 (&raw)[chunk_words<WD>()], bool& nonfinite) {
    if constexpr (WD == kF32) {
        // w * 0 is NaN exactly when w is infinite or NaN
        float amax = 0.f, probe = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const float w = weight_at<WD>(raw, j);
            amax = fmaxf(amax, fabsf(w));
            probe = fmaf(w, 0.f, probe);
        }
        nonfinite = probe != probe;
        if (!nonfinite) return amax;
    } else {
        // |x| of a 16-bit float orders like its bit pattern with the sign
        // cleared, and a pattern at or above the exponent-all-ones one is an
        // infinity or a NaN: one integer max per pair of weights.
        uint32_t m = 0u;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 v = raw[j];
            m = __vmaxu2(m, __vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu));
            m = __vmaxu2(m, __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
        }
        const uint32_t top = max(m & 0xFFFFu, m >> 16);
        constexpr uint32_t kInfBits = WD == kF16 ? 0x7C00u : 0x7F80u;
        nonfinite = top >= kInfBits;
        if (!nonfinite) {
            if constexpr (WD == kF16) return __half2float(__ushort_as_half(static_cast<unsigned short>(top)));
            return __uint_as_float(top << 16);
        }
    }
    float amax = 0.f;  // a chunk with a non-finite weight: max over the finite ones
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const float w = weight_at<WD>(raw, j);
        if (isfinite(w)) amax = fmaxf(amax, fabsf(w));
    }
    return amax;
}

template <int WD>
__device__ __forceinline__ void fetch_chunk(const void* W, int64_t c, uint4 (&raw)[chunk_words<WD>()]) {
    const uint4* p = reinterpret_cast<const uint4*>(W) + c * chunk_words<WD>();
#pragma unroll
    for (int j = 0; j < chunk_words<WD>(); ++j) raw[j] = p[j];
}

// The scale as stored (its bit pattern, widened to 32 bits) and its value.
template <int SD>
__device__ __forceinline__ float stored_scale(float s) {
    if constexpr (SD == kF32) return s;
    else if constexpr (SD == kF16) return __half2float(__float2half_rn(s));
    else return __bfloat162float(__float2bfloat16_rn(s));
}

template <int SD>
__device__ __forceinline__ void store_scale(void* S, int64_t i, float s) {
    if constexpr (SD == kF32) static_cast<float*>(S)[i] = s;
    else if constexpr (SD == kF16) static_cast<__half*>(S)[i] = __float2half_rn(s);
    else static_cast<__nv_bfloat16*>(S)[i] = __float2bfloat16_rn(s);
}

__device__ __forceinline__ void put_code(uint32_t (&word)[3], int j, uint32_t q) {
    const int bit = 3 * j, wi = bit >> 5, sh = bit & 31;  // stream bits 3j .. 3j+2 of the chunk
    word[wi] |= q << sh;
    if (sh > 29) word[wi + 1] |= q >> (32 - sh);
}

template <int WD, int SD>
__global__ void __launch_bounds__(kQuantThreads) quantize_int3_kernel(const void* __restrict__ W, int64_t chunks,
                                                                      int cpb, void* __restrict__ S,
                                                                      uint8_t* __restrict__ B) {
    grid_dependency_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (int64_t(blockIdx.x) * kQuantThreads + threadIdx.x - lane);
    const int64_t stride = int64_t(gridDim.x) * kQuantThreads;
    // Chunk c of the flat storage is chunk c % cpb of block c / cpb; since cpb
    // divides 32 and the warp's chunks start on a multiple of 32, a block's
    // chunks sit in adjacent lanes of one warp.
    for (int64_t base = warp0; base < chunks; base += stride) {
        const int64_t c = base + lane;
        const bool live = c < chunks;
        uint4 raw[chunk_words<WD>()];
        float amax = 0.f;
        bool nonfinite = false;
        if (live) {
            fetch_chunk<WD>(W, c, raw);
            amax = chunk_amax<WD>(raw, nonfinite);
        }
        for (int o = 1; o < cpb; o <<= 1) {
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            nonfinite |= __shfl_xor_sync(0xffffffffu, nonfinite ? 1 : 0, o) != 0;
        }
        if (!live) continue;
        const float s = amax > 0.f ? amax / 3.5f : 1.0f / 3.5f;
        const float stored = stored_scale<SD>(s);
        if ((lane & (cpb - 1)) == 0) store_scale<SD>(S, c / cpb, s);
        const bool rejected = nonfinite || !isfinite(stored) || (amax > 0.f && stored == 0.f);
        if (rejected && (lane & (cpb - 1)) == 0) record_error(MNB_ERR_CONTENT);
        // The code is rint of the correctly rounded quotient w / stored.  It is
        // formed without a division by Markstein's correction step (Markstein,
        // "Computation of elementary functions on the IBM RISC System/6000
        // processor", 1990; Muller et al., "Handbook of Floating-Point
        // Arithmetic", division with an fma): when y = RN(1/stored) and q is
        // within one ulp of w / stored, the residual r = w - stored * q is
        // exact in one fma and RN(q + r y) is the correctly rounded quotient.
        // q0 = RN(w y) can be up to two ulps off near the top of a binade, so
        // the step is applied twice: the first brings q within one ulp, the
        // second rounds correctly.  Scales whose reciprocal is not a normal
        // number, or whose significand is all ones, keep the IEEE division.
        // Adding 1.5 * 2^23 then rounds the quotient (|q| < 6 for an accepted
        // block) to an integer in the low mantissa bits, ties to even.
        constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
        const float y = 1.0f / stored;
        const bool direct = rejected || !(fabsf(y) < 0x1p100f && fabsf(y) > 0x1p-100f) ||
                            (__float_as_uint(stored) & 0x7FFFFFu) == 0x7FFFFFu;
        const int kBias = __float_as_int(kMagic) - 4;
        uint32_t word[3] = {0u, 0u, 0u};
        if (!direct) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float w = weight_at<WD>(raw, j);
                const float q0 = w * y;
                const float q1 = fmaf(fmaf(-q0, stored, w), y, q0);
                const float q = fmaf(fmaf(-q1, stored, w), y, q1);
                const float m = q + kMagic;
                put_code(word, j, static_cast<uint32_t>(min(max(__float_as_int(m) - kBias, 0), 7)));
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float r = fminf(fmaxf(rintf(weight_at<WD>(raw, j) / stored), -8.f), 8.f);
                put_code(word, j, rejected ? 4u : static_cast<uint32_t>(min(max(static_cast<int>(r) + 4, 0), 7)));
            }
        }
        uint32_t* dst = reinterpret_cast<uint32_t*>(B + c * 12);
        dst[0] = word[0];
        dst[1] = word[1];
        dst[2] = word[2];
    }
    grid_launch_dependents();
}

template <int WD>
cudaError_t launch_wd(const void* W, int64_t chunks, int cpb, int s_dtype, void* S, uint8_t* B, int sm_count,
                      cudaStream_t stream) {
    const int64_t blocks = std::min<int64_t>(cdiv<int64_t>(chunks, kQuantThreads), int64_t(sm_count) * 8);
    const dim3 grid(static_cast<unsigned>(std::max<int64_t>(blocks, 1)));
    cudaError_t e;
    if (s_dtype == kF32) {
        if ((e = set_max_carveout(quantize_int3_kernel<WD, kF32>)) != cudaSuccess) return e;
        quantize_int3_kernel<WD, kF32><<<grid, kQuantThreads, 0, stream>>>(W, chunks, cpb, S, B);
    } else if (s_dtype == kF16) {
        if ((e = set_max_carveout(quantize_int3_kernel<WD, kF16>)) != cudaSuccess) return e;
        quantize_int3_kernel<WD, kF16><<<grid, kQuantThreads, 0, stream>>>(W, chunks, cpb, S, B);
    } else {
        if ((e = set_max_carveout(quantize_int3_kernel<WD, kBF16>)) != cudaSuccess) return e;
        quantize_int3_kernel<WD, kBF16><<<grid, kQuantThreads, 0, stream>>>(W, chunks, cpb, S, B);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t quant_take_error(unsigned int* out) { return take_unit_error(out); }

// W [N, K] (K % bs == 0, so the flat storage is whole chunks and whole blocks):
// the packed rows are the chunks' 12-byte groups in order, and the scales the
// blocks' in order.
cudaError_t launch_quantize_int3(const void* W, int w_dtype, int64_t N, int64_t K, int bs, uint8_t* B, void* S,
                                 int s_dtype, int sm_count, cudaStream_t stream) {
    const int64_t chunks = N * (K / 32);
    const int cpb = bs / 32;
    if (w_dtype == kF32) return launch_wd<kF32>(W, chunks, cpb, s_dtype, S, B, sm_count, stream);
    if (w_dtype == kF16) return launch_wd<kF16>(W, chunks, cpb, s_dtype, S, B, sm_count, stream);
    return launch_wd<kBF16>(W, chunks, cpb, s_dtype, S, B, sm_count, stream);
}

}  // namespace mnb
