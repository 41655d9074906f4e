// prepack.cu -- the version-1 private prepacked layout of a MatMulNBits weight
// (the versioned private prepack left open by "INT3 QMoE CUDA correctness
// baseline and Qwen experimental results", Not PR2-PR4 Completion).
//
// One pass over the source: one thread per (row, 32-code chunk) writes the
// chunk's code words (INT3 regrouped, INT4 as stored), one thread per (row,
// 4-byte word of the row's tail) writes its scales, zero points and zero
// padding; thread 0 of block 0 writes the header.  The layout is described in
// include/mnb.h.
#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "kernels.h"

namespace mnb {

namespace {

struct Header {
    uint32_t w[MNB_PREPACK_HEADER_BYTES / 4];
};

// The 32 codes of an INT3 chunk (96-bit LSB-first stream s0..s2) regrouped
// into the three words of the prepacked form.
__device__ __forceinline__ void regroup_int3(const uint32_t (&s)[3], uint32_t (&o)[3]) {
    auto code = [&](int j) -> uint32_t {
        const int bit = 3 * j, wd = bit >> 5, sh = bit & 31;
        uint32_t v = s[wd] >> sh;
        if (sh > 29) v |= s[wd + 1] << (32 - sh);
        return v & 7u;
    };
    o[0] = o[1] = o[2] = 0u;
#pragma unroll
    for (int g = 0; g < 3; ++g)
#pragma unroll
        for (int b = 0; b < 4; ++b) o[g] |= (code(8 * g + 2 * b) | (code(8 * g + 2 * b + 1) << 3)) << (8 * b);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const uint32_t e = code(24 + 2 * b), d = code(25 + 2 * b);
        o[0] |= (e & 3u) << (8 * b + 6);
        o[1] |= (d & 3u) << (8 * b + 6);
        o[2] |= ((e >> 2) << (8 * b + 6)) | ((d >> 2) << (8 * b + 7));
    }
}

__global__ void prepack_kernel(const uint8_t* __restrict__ B, const uint8_t* __restrict__ S,
                               const uint8_t* __restrict__ Z, int64_t N, int C, int bits, int64_t row_bytes,
                               int64_t s_row, int64_t z_row, uint8_t* __restrict__ dst, int64_t stride,
                               int64_t scale_off, int64_t zp_off, const Header hdr) {
    if (blockIdx.x == 0 && threadIdx.x < MNB_PREPACK_HEADER_BYTES / 4)
        reinterpret_cast<uint32_t*>(dst)[threadIdx.x] = hdr.w[threadIdx.x];
    uint8_t* rows = dst + MNB_PREPACK_HEADER_BYTES;
    const int64_t code_bytes = int64_t(C) * 4 * bits;
    const int tail_words = static_cast<int>((stride - code_bytes) / 4);
    const int per_row = C + tail_words;
    const int64_t total = N * per_row;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t n = i / per_row;
        const int item = static_cast<int>(i - n * per_row);
        uint8_t* out = rows + n * stride;
        if (item < C) {
            // code chunk: 4 * bits bytes, 4-byte aligned on both sides
            const uint32_t* src = reinterpret_cast<const uint32_t*>(B + n * row_bytes + int64_t(item) * 4 * bits);
            uint32_t* o = reinterpret_cast<uint32_t*>(out + int64_t(item) * 4 * bits);
            if (bits == 3) {
                const uint32_t s[3] = {src[0], src[1], src[2]};
                uint32_t r[3];
                regroup_int3(s, r);
                o[0] = r[0];
                o[1] = r[1];
                o[2] = r[2];
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) o[q] = src[q];
            }
        } else {
            // tail word: scale bytes, then zero-point bytes, then zeros
            const int64_t off = code_bytes + int64_t(item - C) * 4;
            uint32_t v = 0;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int64_t o = off + b;
                uint32_t byte = 0;
                if (o < scale_off + s_row)
                    byte = S[n * s_row + (o - scale_off)];
                else if (zp_off >= 0 && o < zp_off + z_row)
                    byte = Z[n * z_row + (o - zp_off)];
                v |= byte << (8 * b);
            }
            *reinterpret_cast<uint32_t*>(out + off) = v;
        }
    }
}

}  // namespace

cudaError_t launch_prepack(const uint8_t* B, const void* scales, int scale_dtype, const uint8_t* zp, int64_t N,
                           int64_t K, int bits, int bs, const void* header, size_t header_bytes, uint8_t* dst,
                           int64_t row_stride, int64_t scale_off, int64_t zp_off, int sm_count, cudaStream_t stream) {
    if (header_bytes > sizeof(Header)) return cudaErrorInvalidValue;
    Header h = {};
    std::memcpy(h.w, header, header_bytes);
    const int64_t nb = cdiv<int64_t>(K, bs);
    const int C = static_cast<int>(nb * bs / 32);
    const int64_t row_bytes = nb * bs * bits / 8;
    const int64_t s_row = nb * (scale_dtype == kF32 ? 4 : 2);
    const int64_t z_row = zp ? cdiv<int64_t>(nb * bits, 8) : 0;
    const int64_t items = N * (C + (row_stride - int64_t(C) * 4 * bits) / 4);
    const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>(cdiv<int64_t>(items, 256), int64_t(sm_count) * 8));
    const cudaError_t e = set_max_carveout(prepack_kernel);
    if (e != cudaSuccess) return e;
    prepack_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        B, static_cast<const uint8_t*>(scales), zp, N, C, bits, row_bytes, s_row, z_row, dst, row_stride, scale_off,
        zp_off, h);
    return cudaGetLastError();
}

}  // namespace mnb
