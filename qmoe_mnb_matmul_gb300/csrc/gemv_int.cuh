// gemv_int.cuh -- exact integer dot products of packed INT4 / INT3 codes with
// fixed-point activations (dp4a): the arithmetic core of the SIMT GEMV.
//
// Activation image.  Every 32-code chunk c of an activation row gets its own
// power-of-two scale 2^s, s = min(140 - e, 126) with e the exponent field of
// the chunk's largest |a|, so that v_k = rint(a_k 2^s) is an integer with
// |v_k| <= 2^14.  v_k is split into two signed 8-bit digits,
// v = 256 d1 + d0 (d0 in [-128, 127], d1 in [-64, 64]).  The rounding of v_k
// is the only approximation: 2^-15 of the chunk's largest |a| at most.
//
// Code words.  Word i of an INT4 chunk holds codes 8i .. 8i+7, the even codes
// in the low nibbles of its bytes and the odd codes in the high nibbles, so
//   lo = w & 0x0F0F0F0F   has codes 8i, 8i+2, 8i+4, 8i+6, one per byte,
//   hi = w & 0xF0F0F0F0   has 16 x codes 8i+1, 8i+3, 8i+5, 8i+7,
// and one dp4a multiplies four codes by four digits and adds the products.
// INT3: the 24-bit group g (codes 8g .. 8g+7) of the chunk's 96-bit stream is
// spread so that byte b holds code 8g+2b in bits 0-2 and code 8g+2b+1 in
// bits 3-5; the masks 0x07070707 and 0x38383838 then give the even codes and
// 8 x the odd codes.
//
// Regrouped INT3 (the prepacked layout): the chunk's three words hold codes
// 0-7, 8-15 and 16-23 already spread (byte b: code 8g+2b in bits 0-2, code
// 8g+2b+1 in bits 3-5), and codes 24-31 in the spare top two bits of each
// byte: bits 6-7 of word 0 / word 1 byte b hold the low two bits of code
// 24+2b / 25+2b, bits 6 / 7 of word 2 byte b their third bits.  Groups 0-2
// then need only the two masks, and group 3 two shifts and a mask per half.
//
// A chunk's result T = sum_k v_k (q_k - z) = S_even + S_odd / 16 (INT4; / 8
// for INT3) - z V with V = sum_k v_k is an exact int32 (|T| < 2^23), and the
// chunk contributes block_scale * 2^-s * T (one conversion, one multiply and
// one fp32 add).  Integer inputs stay exact: with integer activations and a
// unit scale, every chunk term and every partial sum is an integer below 2^24.
#pragma once

#include "common.cuh"

namespace mnb {
namespace gemv_int {

// Activation image of one (row, chunk): four 16-byte quads of digits, quad q =
// {low digits of the even codes, high digits of the even codes, low digits of
// the odd codes, high digits of the odd codes}; word i of a quad covers the
// code word i (codes 8i .. 8i+7).  Quads of 32 consecutive chunks are
// interleaved so that the 32 lanes of a warp read 32 consecutive 16-byte words:
//   Q[((m * CB + c / 32) * 4 + q) * 32 + c % 32],  CB = ceil(C / 32).
__host__ __device__ inline int qgroups(int C) { return (C + 31) / 32; }
__host__ __device__ inline int64_t qimg_bytes(int MT, int C) { return int64_t(MT) * qgroups(C) * 4 * 32 * 16; }
__device__ __forceinline__ int qbase(int m, int c, int C) { return (m * qgroups(C) + (c >> 5)) * 128 + (c & 31); }

// Per-(row, chunk) constants: {V = sum of the chunk's v_k, bits of 2^-s}.
__host__ __device__ inline int64_t corr_bytes(int MT, int C) { return (int64_t(MT) * C * 8 + 127) / 128 * 128; }

// d += sum over the four byte lanes of a (signed digits) * b (unsigned codes).
__device__ __forceinline__ int dp4a_su(uint32_t a, uint32_t b, int d) {
    int r;
    asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(d));
    return r;
}

// (a & m) | (b & ~m) in one logic instruction.
__device__ __forceinline__ uint32_t bit_select(uint32_t m, uint32_t a, uint32_t b) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xE4;" : "=r"(d) : "r"(a), "r"(b), "r"(m));
    return d;
}

// Even / odd code bytes of code word g of a chunk (see the file comment);
// RG: the chunk is in the regrouped INT3 form.
template <int BITS, bool RG = false>
__device__ __forceinline__ void code_bytes(const uint32_t (&w)[BITS], int g, uint32_t& lo, uint32_t& hi) {
    if constexpr (BITS == 3 && RG) {
        if (g < 3) {
            lo = w[g] & 0x07070707u;
            hi = w[g] & 0x38383838u;
        } else {
            lo = ((w[0] >> 6) & 0x03030303u) | ((w[2] >> 4) & 0x04040404u);
            hi = ((w[1] >> 3) & 0x18181818u) | ((w[2] >> 2) & 0x20202020u);
        }
    } else if constexpr (BITS == 4) {
        lo = w[g] & 0x0F0F0F0Fu;
        hi = w[g] & 0xF0F0F0F0u;
    } else {
        // the 24-bit group g of the 96-bit stream w[0..2] at bit 0
        const uint32_t x = g == 0 ? w[0] : g == 1 ? __funnelshift_r(w[0], w[1], 24)
                                     : g == 2 ? __funnelshift_r(w[1], w[2], 16) : (w[2] >> 8);
        // 12-bit halves to 16-bit halves, then 6-bit quarters to bytes (bits
        // above the fields are never read by the masks below)
        const uint32_t x1 = bit_select(0x00000FFFu, x, x << 4);
        const uint32_t x2 = bit_select(0x003F003Fu, x1, x1 << 2);
        lo = x2 & 0x07070707u;
        hi = x2 & 0x38383838u;
    }
}

// sum over the chunk of v_k q_k for one code chunk w and one activation image q.
template <int BITS, bool RG = false>
__device__ __forceinline__ int chunk_dot(const uint32_t (&w)[BITS], const uint4 (&q)[4]) {
    const uint32_t q0[4] = {q[0].x, q[0].y, q[0].z, q[0].w};
    const uint32_t q1[4] = {q[1].x, q[1].y, q[1].z, q[1].w};
    const uint32_t q2[4] = {q[2].x, q[2].y, q[2].z, q[2].w};
    const uint32_t q3[4] = {q[3].x, q[3].y, q[3].z, q[3].w};
    int se0 = 0, se1 = 0, so0 = 0, so1 = 0;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        uint32_t lo, hi;
        code_bytes<BITS, RG>(w, g, lo, hi);
        se0 = dp4a_su(q0[g], lo, se0);
        se1 = dp4a_su(q1[g], lo, se1);
        so0 = dp4a_su(q2[g], hi, so0);
        so1 = dp4a_su(q3[g], hi, so1);
    }
    // the odd sums carry the codes' 16x (INT4) or 8x (INT3) byte position exactly
    return (se1 * 256 + se0) + ((so1 * 256 + so0) >> (BITS == 4 ? 4 : 3));
}

// Any width 1..8 (the row-local LSB-first format beyond 3 and 4 bits): code j
// of the chunk whose 4 * bits bytes start at `chunk` (4-byte aligned, shared
// memory), read through at most two aligned words.
__device__ __forceinline__ uint32_t code_any(const uint8_t* chunk, int j, int bits) {
    const uint32_t bit = static_cast<uint32_t>(j * bits);
    const uint32_t* wp = reinterpret_cast<const uint32_t*>(chunk) + (bit >> 5);
    const uint32_t off = bit & 31;
    const uint32_t hi = off + bits > 32 ? wp[1] : 0u;  // only a code that crosses a word reads the next one
    return __funnelshift_r(wp[0], hi, off) & ((1u << bits) - 1u);
}

// Any width: the chunk's codes as plain bytes, code word g's even codes in
// lo[g] and its odd codes in hi[g] (no position factor).
__device__ __forceinline__ void codes_any(const uint8_t* chunk, int bits, uint32_t (&lo)[4], uint32_t (&hi)[4]) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        lo[g] = 0;
        hi[g] = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            lo[g] |= code_any(chunk, 8 * g + 2 * b, bits) << (8 * b);
            hi[g] |= code_any(chunk, 8 * g + 2 * b + 1, bits) << (8 * b);
        }
    }
}

// chunk_dot on code bytes from codes_any.
__device__ __forceinline__ int chunk_dot_bytes(const uint32_t (&lo)[4], const uint32_t (&hi)[4], const uint4 (&q)[4]) {
    const uint32_t q0[4] = {q[0].x, q[0].y, q[0].z, q[0].w};
    const uint32_t q1[4] = {q[1].x, q[1].y, q[1].z, q[1].w};
    const uint32_t q2[4] = {q[2].x, q[2].y, q[2].z, q[2].w};
    const uint32_t q3[4] = {q[3].x, q[3].y, q[3].z, q[3].w};
    int se0 = 0, se1 = 0, so0 = 0, so1 = 0;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        se0 = dp4a_su(q0[g], lo[g], se0);
        se1 = dp4a_su(q1[g], lo[g], se1);
        so0 = dp4a_su(q2[g], hi[g], so0);
        so1 = dp4a_su(q3[g], hi[g], so1);
    }
    return (se1 * 256 + se0) + (so1 * 256 + so0);
}

// Zero-point code of block b in a packed zero-point row of any width.
__device__ __forceinline__ int zero_point_any(const uint8_t* zrow, int b, int bits) {
    const int bit = b * bits, byte = bit >> 3, sh = bit & 7;
    uint32_t v = zrow[byte];
    if (sh + bits > 8) v |= static_cast<uint32_t>(zrow[byte + 1]) << 8;
    return static_cast<int>((v >> sh) & ((1u << bits) - 1u));
}

// Signed 8-bit digit d as the byte of lane `lane` (0..3).
__device__ __forceinline__ uint32_t digit_byte(int d, int lane) { return (static_cast<uint32_t>(d) & 0xFFu) << (8 * lane); }

// One thread per (row m, chunk c, code word i): the eight activations of codes
// 32c + 8i .. +7 of row m -> the image words and, from lane i == 0 of the four
// adjacent lanes that share the chunk, the chunk's {V, 2^-s}.  With more items
// than threads, a thread loads kStageBatch items before it converts any (one
// memory round trip per batch, not per item).  Every lane of a warp runs the
// same number of iterations (the shuffles need all of them); row(m) returns
// activation row m (K valid entries, dtype `dt`) or nullptr for a row of
// zeros; `vec`: rows may be read with 16-byte loads.
constexpr int kStageBatch = 4;

// int8 activation image (the int8-activation compute mode): lanes of one
// weight block (4 * bs / 32 adjacent items) share the block's amax; the
// quantised codes rint(a / (amax / 127)) (binary32 division) go to the low
// digits, the high digits stay zero, and the chunk factor is amax / 127.
__device__ __forceinline__ void int8a_item(const float (&a)[8], int block_lanes, uint32_t (&wd)[4], int& vsum,
                                           float& factor) {
    uint32_t mx = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) mx = max(mx, __float_as_uint(a[j]) & 0x7FFFFFFFu);
    for (int o = 1; o < block_lanes; o <<= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float sa = __uint_as_float(mx) / 127.0f;
#pragma unroll
    for (int q = 0; q < 4; ++q) wd[q] = 0u;
    vsum = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int v = sa != 0.0f ? static_cast<int>(fminf(fmaxf(rintf(a[j] / sa), -127.0f), 127.0f)) : 0;
        wd[2 * (j & 1)] |= digit_byte(v, j >> 1);
        vsum += v;
    }
    factor = sa;
}

template <int BATCH, typename RowFn>
__device__ __forceinline__ void stage_image_b(uint4* Q, int2* Corr, int MT, int C, int64_t K, int dt, bool vec,
                                              RowFn row, int tid, int nthreads, int int8a_block_lanes = 0) {
    constexpr int kStageBatch = BATCH;
    const int total = MT * C * 4;
    for (int base = 0; base < total; base += nthreads * kStageBatch) {
        float a[kStageBatch][8];
#pragma unroll
        for (int u = 0; u < kStageBatch; ++u) {
            const int item = base + u * nthreads + tid;
            const bool live = item < total;
            const int i = item & 3, mc = item >> 2;
            const int m = live ? mc / C : 0, c = live ? mc - m * C : 0;
            const void* src = live ? row(m) : nullptr;
            const int64_t k0 = int64_t(c) * 32 + 8 * i;
            if (src != nullptr && vec && k0 + 8 <= K) {
                if (dt == kF32) {
                    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(src) + k0);
                    const float4 x = p[0], y = p[1];
                    a[u][0] = x.x; a[u][1] = x.y; a[u][2] = x.z; a[u][3] = x.w;
                    a[u][4] = y.x; a[u][5] = y.y; a[u][6] = y.z; a[u][7] = y.w;
                } else {
                    const uint4 x = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(src) + k0);
                    const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        if (dt == kF16) {
                            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w4[h]));
                            a[u][2 * h] = f.x; a[u][2 * h + 1] = f.y;
                        } else {
                            a[u][2 * h] = __uint_as_float(w4[h] << 16);
                            a[u][2 * h + 1] = __uint_as_float(w4[h] & 0xFFFF0000u);
                        }
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) a[u][j] = (src != nullptr && k0 + j < K) ? load_as_f32(src, dt, k0 + j) : 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < kStageBatch; ++u) {
            if (base + u * nthreads >= total) break;  // uniform: no lane of the CTA has items from here on
            const int item = base + u * nthreads + tid;
            const bool live = item < total;
            const int i = item & 3, mc = item >> 2;
            const int m = live ? mc / C : 0, c = live ? mc - m * C : 0;
            uint32_t wd[4] = {0u, 0u, 0u, 0u};  // even low, even high, odd low, odd high
            int vsum = 0;
            float factor;
            if (int8a_block_lanes) {
                int8a_item(a[u], int8a_block_lanes, wd, vsum, factor);
            } else {
                uint32_t mx = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) mx = max(mx, __float_as_uint(a[u][j]) & 0x7FFFFFFFu);
                mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const int s = min(140 - static_cast<int>(mx >> 23), 126);  // |a| 2^s < 2^14 for the whole chunk
                const float up = __uint_as_float(static_cast<uint32_t>(s + 127) << 23);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int v = __float2int_rn(a[u][j] * up);  // exact scaling, one rounding
                    const int d1 = (v + 128) >> 8;
                    const int d0 = v - d1 * 256;
                    const int odd = j & 1, lane = j >> 1;
                    wd[2 * odd] |= digit_byte(d0, lane);
                    wd[2 * odd + 1] |= digit_byte(d1, lane);
                    vsum += v;
                }
                factor = __uint_as_float(static_cast<uint32_t>(127 - s) << 23);
            }
            vsum += __shfl_xor_sync(0xffffffffu, vsum, 1);
            vsum += __shfl_xor_sync(0xffffffffu, vsum, 2);
            if (live) {
                uint32_t* q = reinterpret_cast<uint32_t*>(Q + qbase(m, c, C));
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) q[qq * 32 * 4 + i] = wd[qq];
                if (i == 0) Corr[m * C + c] = make_int2(vsum, __float_as_int(factor));
            }
        }
    }
}

// One item per thread when they all fit (the common decode case: a batch
// would only add dead slots), else batches of kStageBatch.
// int8a_block_lanes: 0 for the exact 15-bit image, else 4 * block_size / 32
// (the int8 activation compute mode).
template <typename RowFn>
__device__ __forceinline__ void stage_image(uint4* Q, int2* Corr, int MT, int C, int64_t K, int dt, bool vec, RowFn row,
                                            int tid, int nthreads, int int8a_block_lanes = 0) {
    if (MT * C * 4 <= nthreads)
        stage_image_b<1>(Q, Corr, MT, C, K, dt, vec, row, tid, nthreads, int8a_block_lanes);
    else
        stage_image_b<kStageBatch>(Q, Corr, MT, C, K, dt, vec, row, tid, nthreads, int8a_block_lanes);
}

}  // namespace gemv_int
}  // namespace mnb
