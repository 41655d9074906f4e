// gemv_core.cuh -- building blocks of the SIMT weight-only GEMV kernels
// (dense mnb_matmul and the QMoE expert projections).
//
// A chunk is 32 consecutive codes of one packed row: 16 bytes of INT4 or 12
// bytes of INT3 (3-bit codes cross byte boundaries inside the chunk).  A code q
// becomes a float with one byte-permute (INT4) or one shift + one mask (INT3)
// by placing it in mantissa bits 16.. under exponent 126, f = 0.5 + q/256.
// Activations are staged pre-multiplied by 256 (exact), A' = 256 A, so
//     A' f = 128 A + A q   and over a chunk   sum A (q - z) = sum A' f - (128 + z) sum A.
// The scale of the chunk's block then multiplies that once.  Integer inputs
// stay exact: every partial sum is an integer below 2^24.
#pragma once

#include "common.cuh"

namespace mnb {
namespace gemv {

constexpr uint32_t kCodeExp = 0x3F000000u;  // exponent 126 in bits 23..30
constexpr float kAScale = 256.0f;

__host__ __device__ constexpr int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// Float images (0.5 + q/256) of the 4 codes 4g .. 4g+3 of a 32-code chunk.
template <int BITS>
__device__ __forceinline__ void chunk_codes4(const uint32_t (&w)[BITS], int g, float2& f01, float2& f23) {
    if constexpr (BITS == 4) {
        // word g/2 holds codes 8(g/2) .. 8(g/2)+7, low nibble first: its low
        // nibbles are the even codes, its high nibbles the odd ones.
        const uint32_t x = w[g >> 1];
        const uint32_t lo = x & 0x0F0F0F0Fu;
        const uint32_t hi = (x >> 4) & 0x0F0F0F0Fu;
        const uint32_t sub = (g & 1) * 2;
        f01.x = __uint_as_float(__byte_perm(lo, kCodeExp, 0x7044u | (sub << 8)));
        f01.y = __uint_as_float(__byte_perm(hi, kCodeExp, 0x7044u | (sub << 8)));
        f23.x = __uint_as_float(__byte_perm(lo, kCodeExp, 0x7044u | ((sub + 1) << 8)));
        f23.y = __uint_as_float(__byte_perm(hi, kCodeExp, 0x7044u | ((sub + 1) << 8)));
    } else {
        // 3-bit code j sits at stream bit 3j of the 96-bit chunk (w[0] first).
        uint32_t f[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int p = 3 * (4 * g + i);
            const int wi = p >> 5, off = p & 31;
            uint32_t x;
            if (off >= 16)
                x = (off + 3 <= 32) ? (w[wi] >> (off - 16))
                                    : __funnelshift_r(w[wi], w[wi + 1 < BITS ? wi + 1 : wi], off - 16);
            else
                x = w[wi] << (16 - off);
            f[i] = (x & 0x00070000u) | kCodeExp;
        }
        f01 = make_float2(__uint_as_float(f[0]), __uint_as_float(f[1]));
        f23 = make_float2(__uint_as_float(f[2]), __uint_as_float(f[3]));
    }
}

// Words of chunk c of a packed row held in shared memory.
template <int BITS>
__device__ __forceinline__ void load_chunk(const uint8_t* row, int c, uint32_t (&w)[BITS]) {
    if constexpr (BITS == 4) {
        const uint4 v = *reinterpret_cast<const uint4*>(row + 16 * c);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else {
        const uint32_t* p = reinterpret_cast<const uint32_t*>(row + 12 * c);
        w[0] = p[0]; w[1] = p[1]; w[2] = p[2];
    }
}

// Zero-point code of block b in a packed zero-point row (LSB-first, width BITS).
template <int BITS>
__device__ __forceinline__ int zero_point_code(const uint8_t* zrow, int b) {
    const int bit = b * BITS, byte = bit >> 3, sh = bit & 7;
    uint32_t v = zrow[byte];
    if (sh + BITS > 8) v |= static_cast<uint32_t>(zrow[byte + 1]) << 8;
    return (v >> sh) & ((1u << BITS) - 1u);
}

// Shared-memory image of MT activation rows for the chunk loop: float4 i4 of
// chunk c of row m (codes 32c + 4 i4 .. +3) lives at A4[(m*8 + i4)*C + c], so
// consecutive lanes (consecutive c) read consecutive 16-byte words.
// fetch(m, k) returns the activation (0 when out of range); the image holds
// 256 * fetch, and Asum[m*C + c] the plain sum of the chunk's 32 activations.
template <int MT, typename Fetch>
__device__ __forceinline__ void stage_activations(float4* A4, float* Asum, int C, Fetch fetch, int tid, int nthreads) {
    const int64_t Kpad = int64_t(C) * 32;
    for (int64_t i = tid; i < int64_t(MT) * Kpad; i += nthreads) {
        const int m = static_cast<int>(i / Kpad);
        const int64_t k = i - int64_t(m) * Kpad;
        const float v = kAScale * fetch(m, k);
        const int c = static_cast<int>(k >> 5), i4 = static_cast<int>((k >> 2) & 7), e = static_cast<int>(k & 3);
        reinterpret_cast<float*>(&A4[(int64_t(m) * 8 + i4) * C + c])[e] = v;
    }
    __syncthreads();
    for (int i = tid; i < MT * C; i += nthreads) {
        const int m = i / C, c = i - m * C;
        float s = 0.f;
        for (int j = 0; j < 32; ++j) s += reinterpret_cast<const float*>(&A4[(m * 8 + (j >> 2)) * C + c])[j & 3];
        Asum[m * C + c] = s * (1.0f / kAScale);
    }
    __syncthreads();
}

// One lane, chunk c of R packed rows: out[r][m] += scale[r] * sum_k A[m, k] (q[r, k] - z[r]).
template <int BITS, int R, int MT>
__device__ __forceinline__ void chunk_accumulate(const uint32_t (&w)[R][BITS], const float (&sc)[R], const float (&zz)[R],
                                                 const float4* __restrict__ A4, const float* __restrict__ Asum, int C,
                                                 int c, float (&out)[R][MT]) {
    float2 P[R][MT];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) P[r][m] = make_float2(0.f, 0.f);
#pragma unroll
    for (int i4 = 0; i4 < 8; ++i4) {
        float4 av[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) av[m] = A4[(m * 8 + i4) * C + c];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float2 f01, f23;
            chunk_codes4<BITS>(w[r], i4, f01, f23);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                P[r][m] = ffma2(make_float2(av[m].x, av[m].y), f01, P[r][m]);
                P[r][m] = ffma2(make_float2(av[m].z, av[m].w), f23, P[r][m]);
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const float as = Asum[m * C + c];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float t = fmaf(-(128.0f + zz[r]), as, P[r][m].x + P[r][m].y);
            out[r][m] = fmaf(sc[r], t, out[r][m]);
        }
    }
}

}  // namespace gemv
}  // namespace mnb
