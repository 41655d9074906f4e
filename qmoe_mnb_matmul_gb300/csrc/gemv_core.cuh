// gemv_core.cuh -- building blocks of the SIMT weight-only GEMV kernels
// (dense mnb_matmul and the QMoE expert projections).
//
// A chunk is 32 consecutive codes of one packed row: 16 bytes of INT4 or 12
// bytes of INT3 (3-bit codes cross byte boundaries inside the chunk).  A code
// q becomes a float by a single bit operation that drops it into mantissa
// bits p .. p+bits-1 under exponent 126:  f = 0.5 + q * 2^(p-24).
//   INT4: one byte-permute per code, p = 16 (even codes) and 12 (odd codes).
//   INT3: one funnel shift per three codes, then one mask per code,
//         p = 13, 16, 19 for codes 3i, 3i+1, 3i+2 of the chunk.
// Activations are staged pre-multiplied by the matching power of two,
// A'_j = A_j * 2^(24 - p_j) (exact), so A'_j f_j = A'_j / 2 + A_j q_j and
//     sum_j A_j (q_j - z) = sum_j A'_j f_j - Csum - z * Asum
// with Csum = sum_j A'_j / 2 and Asum = sum_j A_j per chunk, computed once
// per staged activation row.  The block scale then multiplies the chunk
// result once.  Integer inputs stay exact: every partial sum is an integer
// below 2^24.
#pragma once

#include "common.cuh"

namespace mnb {
namespace gemv {

constexpr uint32_t kCodeExp = 0x3F000000u;  // exponent 126 in bits 23..30

__host__ __device__ constexpr int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// Mantissa position of code j (0..31) of a chunk.  INT4: the even codes
// (low nibbles) go to bits 16..19 and the odd codes (high nibbles, masked in
// place) to bits 12..15.
template <int BITS>
__host__ __device__ constexpr int code_pos(int j) {
    return BITS == 4 ? (j % 2 == 0 ? 16 : 12) : 13 + 3 * (j % 3);
}

// Power-of-two pre-scale of the activation that meets code j.
template <int BITS>
__host__ __device__ constexpr float code_scale(int j) {
    return static_cast<float>(1u << (24 - code_pos<BITS>(j)));
}

// INT3: the 32-bit window of the chunk's 96-bit stream that holds code j at
// bit code_pos(j).  j is a compile-time constant after unrolling.
__device__ __forceinline__ uint32_t int3_window(const uint32_t (&w)[3], int j) {
    const int first = j - j % 3;                  // first code of j's triplet
    const int b = 3 * first - 13;                 // stream bit that lands on bit 0
    if (b < 0) return w[0] << (-b);
    const int i = b >> 5, o = b & 31;
    if (o == 0) return w[i];
    return __funnelshift_r(w[i], w[i + 1 < 3 ? i + 1 : 2], o);  // bits past the chunk are never used
}

// Float images of the 4 codes 4g .. 4g+3 of a 32-code chunk.
template <int BITS>
__device__ __forceinline__ void chunk_codes4(const uint32_t (&w)[BITS], int g, float2& f01, float2& f23) {
    if constexpr (BITS == 4) {
        // word g/2 holds codes 8(g/2) .. 8(g/2)+7, low nibble first.  Byte b of
        // lo is the even code 2b (placed at bits 16..19 of the image), byte b of
        // hi is the odd code 2b+1 already shifted up by 4 (placed at bits 8..15,
        // i.e. the code lands on bits 12..15).
        const uint32_t x = w[g >> 1];
        const uint32_t lo = x & 0x0F0F0F0Fu;
        const uint32_t hi = x & 0xF0F0F0F0u;
        const uint32_t sub = (g & 1) * 2;
        f01.x = __uint_as_float(__byte_perm(lo, kCodeExp, 0x7044u | (sub << 8)));
        f01.y = __uint_as_float(__byte_perm(hi, kCodeExp, 0x7404u | (sub << 4)));
        f23.x = __uint_as_float(__byte_perm(lo, kCodeExp, 0x7044u | ((sub + 1) << 8)));
        f23.y = __uint_as_float(__byte_perm(hi, kCodeExp, 0x7404u | ((sub + 1) << 4)));
    } else {
        uint32_t f[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int j = 4 * g + i;
            const int p = code_pos<3>(j);
            f[i] = and_or(int3_window(w, j), 7u << p, kCodeExp);
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

// 32 activations starting at k0 one by one (zeros past K or for a null row):
// the path for unaligned rows and a ragged last chunk, kept out of line so the
// vector path stays compact in the instruction cache.
static __device__ __noinline__ void load_chunk_slow(const void* src, int dt, int64_t k0, int64_t K, float* v) {
#pragma unroll 1
    for (int j = 0; j < 32; ++j) v[j] = (src != nullptr && k0 + j < K) ? load_as_f32(src, dt, k0 + j) : 0.f;
}

// Shared-memory image of MT activation rows for the chunk loop.  Chunks are
// grouped by 32 (one per lane of a warp step): float4 i4 (codes 4 i4 .. +3 of
// the chunk) of chunk c of row m lives at
//   A4[(m * CB + c / 32) * 256 + i4 * 32 + c % 32],   CB = ceil(C / 32),
// so a lane's eight float4 of one chunk sit at fixed 512-byte steps from one
// base and the 32 lanes of a step read 32 consecutive 16-byte words.
__host__ __device__ inline int a4_groups(int C) { return (C + 31) / 32; }
__host__ __device__ inline int64_t a4_bytes(int MT, int C) { return int64_t(MT) * a4_groups(C) * 256 * 16; }
__device__ __forceinline__ int a4_base(int m, int c, int C) { return (m * a4_groups(C) + (c >> 5)) * 256 + (c & 31); }

// One thread stages one (row, chunk): it loads the chunk's 32 activations
// (vectorised when `vec`), writes A'_j = A_j * code_scale(j), and the chunk's
// correction Corr[m*C + c] = {-(Csum + z0 Asum) over even j, the same over odd
// j, Asum over even j, Asum over odd j}, with Csum = sum A'_j / 2, Asum =
// sum A_j and z0 = 2^(BITS-1) the implicit zero point, summed in ascending j.
// (The f32x2 products keep even codes in .x and odd codes in .y.)
// row(m) returns activation row m (dtype `dt_arg`, or FIXED_DT when that is
// given at compile time; K valid entries) or nullptr for a row of zeros.
template <int BITS, int MT, int FIXED_DT = -1, typename RowFn>
__device__ __forceinline__ void stage_chunks(float4* A4, float4* Corr, int C, int64_t K, int dt_arg, bool vec, RowFn row,
                                             int tid, int nthreads) {
    const int dt = FIXED_DT >= 0 ? FIXED_DT : dt_arg;  // a compile-time dtype drops the other paths
    constexpr float z0 = float(1 << (BITS - 1));
    for (int i = tid; i < MT * C; i += nthreads) {
        const int m = i / C, c = i - m * C;
        const void* src = row(m);
        const int64_t k0 = int64_t(c) * 32;
        float v[32];
        if (src != nullptr && vec && k0 + 32 <= K) {
            if (dt == kF32) {
                const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(src) + k0);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 x = p[q];
                    v[4 * q] = x.x; v[4 * q + 1] = x.y; v[4 * q + 2] = x.z; v[4 * q + 3] = x.w;
                }
            } else {
                const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(src) + k0);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 x = p[q];
                    const uint32_t u[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        if (dt == kF16) {
                            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&u[h]));
                            v[8 * q + 2 * h] = f.x; v[8 * q + 2 * h + 1] = f.y;
                        } else {
                            v[8 * q + 2 * h] = __uint_as_float(u[h] << 16);
                            v[8 * q + 2 * h + 1] = __uint_as_float(u[h] & 0xFFFF0000u);
                        }
                    }
                }
            }
        } else {
            float t[32];
            load_chunk_slow(src, dt, k0, K, t);
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = t[j];
        }
        float as[2] = {0.f, 0.f}, cs[2] = {0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            as[j & 1] += v[j];
            v[j] *= code_scale<BITS>(j);
            cs[j & 1] += 0.5f * v[j];
        }
        float4* dst = A4 + a4_base(m, c, C);
#pragma unroll
        for (int q = 0; q < 8; ++q) dst[q * 32] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        Corr[m * C + c] = make_float4(-fmaf(z0, as[0], cs[0]), -fmaf(z0, as[1], cs[1]), as[0], as[1]);
    }
}

// One lane, chunk c of R packed rows:
//   out[r][m] += scale[r] * sum_k A[m, k] (q[r, k] - z[r])      (as an even/odd pair)
// dz[r] = z0 - z[r] is the row's zero-point shift from the implicit one (0
// without zero points: one code path serves both, which keeps the kernels
// small).
//
// a4c = A4 + a4_base(0, c, C); row m's float4 i4 is a4c[m * mstride + 32 i4]
// with mstride = a4_groups(C) * 256.  corr = Corr + c; row m's correction is
// corr[m * C].
template <int BITS, int R, int MT>
__device__ __forceinline__ void chunk_accumulate(const uint32_t (&w)[R][BITS], const float (&sc)[R], const float (&dz)[R],
                                                 const float4* __restrict__ a4c, int mstride,
                                                 const float4* __restrict__ corr, int C, float2 (&out)[R][MT]) {
    float2 P[R][MT];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) P[r][m] = make_float2(0.f, 0.f);
#pragma unroll
    for (int i4 = 0; i4 < 8; ++i4) {
        float4 av[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) av[m] = a4c[m * mstride + i4 * 32];
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
        const float4 cr = corr[m * C];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float2 t = __fadd2_rn(P[r][m], make_float2(cr.x, cr.y));
            t = ffma2(make_float2(dz[r], dz[r]), make_float2(cr.z, cr.w), t);
            out[r][m] = ffma2(make_float2(sc[r], sc[r]), t, out[r][m]);
        }
    }
}

}  // namespace gemv
}  // namespace mnb
