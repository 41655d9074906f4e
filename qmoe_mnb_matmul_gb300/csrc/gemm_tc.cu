// gemm_tc.cu -- small-M / prefill MatMulNBits on the 5th-generation tensor
// cores (tcgen05, sm_103a): Y[M, N] = A[M, K] . W^T with W dequantised from
// packed INT4 / INT3 codes, per-block scales and optional zero points, tile by
// tile in shared memory ("Qwen3 Missing-Kernel Implementation Plan", row K03:
// small-M and prefill GEMM on the same compressed weights with bounded
// workspace, partial blocks and output tails; the "tiled dequantisation plus
// GEMM" the QMoE CUDA page names as the missing prefill path).
//
// One persistent CTA per SM walks output tiles of 128 weight rows x BN
// activation rows.  The MMA is "swap-AB": the dequantised weight tile is
// operand A (M = 128), the activation tile operand B (N = BN <= 256), so the
// fp32 accumulator in tensor memory holds Y^T (lane = weight row, column =
// activation row) and small M costs no padding of the weight side.
//
// Warp roles (320 threads):
//   warp 0     TMA producer: activation tiles [BN x 64] (128-byte swizzle)
//   warp 1     TMEM owner; one lane issues tcgen05.mma (K = 16 each, 4 per stage)
//   warps 2-5  dequant: one thread per weight row; cp.async ring of packed
//              bytes and scales, codes -> fp32 (gemv_core.cuh images) ->
//              s (q - z) by FMA -> bf16/fp16 -> swizzled 16-byte stores
//   warps 6-9  epilogue: tcgen05.ld of the accumulator (double buffered in
//              TMEM) -> output dtype -> coalesced stores with M/N masking
// Stage s of the shared ring holds the activation tile and the dequantised
// weight tile of one K step; it is released by a tcgen05.commit once the MMAs
// that read it have completed.  Every wait is bounded.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "gemv_core.cuh"
#include "kernels.h"

namespace mnb {

namespace {

using namespace gemv;

constexpr int kBK = 64;          // K elements per stage: one 128-byte swizzle atom of 16-bit values
constexpr int kBW = 128;         // weight rows per tile (MMA M)
constexpr int kPack = 4;         // depth of each dequant thread's cp.async ring
constexpr int kThreadsTC = 320;
constexpr int kDequantWarp0 = 2, kEpilogueWarp0 = 6;

struct TcArgs {
    int64_t M, K, N;
    const uint8_t* B;
    const void* scales;
    const uint8_t* zp;
    int64_t row_bytes;
    int nb, bs, zp_row_bytes;
    int a_dtype;   // kF16 or kBF16
    void* Y;
    int y_dtype;
    int tiles_n, tiles_m, k_steps;
    int stages;
    uint32_t tmem_cols;
};

struct TcPlan {
    int64_t bars, act, w, pack, scl, total;
};

__host__ __device__ inline TcPlan tc_plan(int BN, int stages, int bits) {
    TcPlan p;
    p.bars = 1024;                                   // barriers + TMEM address, padded to the 1024-byte atom
    p.act = int64_t(BN) * 128;                       // one stage of activations
    p.w = int64_t(kBW) * 128;                        // one stage of dequantised weights
    p.pack = int64_t(kPack) * kBW * (bits == 4 ? 32 : 24);
    p.scl = int64_t(kPack) * kBW * 8;
    p.total = p.bars + int64_t(stages) * (p.act + p.w) + p.pack + p.scl;
    return p;
}

// Byte offset of 16-byte chunk c (k elements 8c .. 8c+7) of row r inside a
// 128-byte-swizzled tile: atoms of 8 rows x 128 bytes, chunk index XOR row % 8.
__device__ __forceinline__ uint32_t sw128(int r, int c) {
    return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

template <int ST>
__device__ __forceinline__ float scale_from_word(uint32_t word, int64_t idx) {
    if constexpr (ST == kF32) {
        return __uint_as_float(word);
    } else {
        const uint32_t h = (idx & 1) ? (word >> 16) : (word & 0xFFFFu);
        if constexpr (ST == kF16) return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
        return __uint_as_float(h << 16);
    }
}

__device__ __forceinline__ uint32_t pack2(float a, float b, bool bf16) {
    if (bf16) {
        const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<const uint32_t*>(&v);
    }
    const __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
}

template <int BITS, int ST, int BN>
__global__ void __launch_bounds__(kThreadsTC, 1) gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_a,
                                                                const __grid_constant__ TcArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int S = a.stages;
    const TcPlan plan = tc_plan(BN, S, BITS);
    uint64_t* full_a = reinterpret_cast<uint64_t*>(smem);
    uint64_t* full_w = full_a + 8;
    uint64_t* empty = full_a + 16;
    uint64_t* acc_full = full_a + 24;
    uint64_t* acc_empty = full_a + 26;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(full_a + 28);
    uint8_t* act = smem + plan.bars;
    uint8_t* wt = act + S * plan.act;
    uint8_t* pack = wt + S * plan.w;
    uint8_t* scl = pack + plan.pack;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (smem_u32(smem) & 1023) {  // the swizzled tiles need 1024-byte alignment
        if (tid == 0) record_error(MNB_ERR_UNSUPPORTED);
        return;
    }
    const int n_tiles = a.tiles_n * a.tiles_m;
    const int ksteps = a.k_steps;
    const bool bf16 = a.a_dtype == kBF16;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full_a[s], 1);
            mbar_init(&full_w[s], 4);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4);
        }
        fence_barrier_init();
        prefetch_tmap(&tmap_a);
    }
    if (warp == 1) tmem_alloc(tmem_holder, a.tmem_cols);
    grid_dependency_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    bool failed = false;

    if (warp == 0) {
        // ----------------------------------------------------- TMA producer
        if (lane == 0) {
            int step = 0;
            for (int t = blockIdx.x; t < n_tiles && !failed; t += gridDim.x) {
                const int m0 = (t % a.tiles_m) * BN;
                for (int ks = 0; ks < ksteps; ++ks, ++step) {
                    const int s = step % S;
                    if (step >= S && !mbar_wait(&empty[s], ((step / S) - 1) & 1)) { failed = true; break; }
                    mbar_arrive_expect_tx(&full_a[s], BN * 128);
                    tma_load_2d(act + s * plan.act, &tmap_a, ks * kBK, m0, &full_a[s]);
                }
            }
        }
    } else if (warp == 1) {
        // --------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_bf = idesc_f16(kBW, BN, true), idesc_h = idesc_f16(kBW, BN, false);
            const uint32_t idesc = bf16 ? idesc_bf : idesc_h;
            int step = 0, tl = 0;
            for (int t = blockIdx.x; t < n_tiles && !failed; t += gridDim.x, ++tl) {
                const int buf = tl & 1;
                if (tl >= 2 && !mbar_wait(&acc_empty[buf], ((tl >> 1) - 1) & 1)) { failed = true; break; }
                tc_fence_after();
                const uint32_t d = tmem + buf * BN;
                for (int ks = 0; ks < ksteps; ++ks, ++step) {
                    const int s = step % S;
                    const uint32_t par = (step / S) & 1;
                    if (!mbar_wait(&full_a[s], par) || !mbar_wait(&full_w[s], par)) { failed = true; break; }
                    tc_fence_after();
                    const uint64_t da = smem_desc_sw128(wt + s * plan.w);
                    const uint64_t db = smem_desc_sw128(act + s * plan.act);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        tc_mma_f16(d, da + 2 * kk, db + 2 * kk, idesc, (ks | kk) != 0);
                    tc_commit(&empty[s]);
                }
                if (failed) break;
                tc_commit(&acc_full[buf]);
            }
        }
    } else if (warp < kEpilogueWarp0) {
        // ------------------------------------------------------------ dequant
        const int r = tid - kDequantWarp0 * 32;  // weight row of the tile
        constexpr int kPB = BITS == 4 ? 32 : 24;  // packed bytes per row per K step
        constexpr int kZ = 1 << (BITS - 1);
        const int nb = a.nb, bs_shift = __ffs(a.bs) - 1;
        const int64_t kcodes = int64_t(nb) * a.bs;  // codes stored per row (K rounded up to a block)
        // the (tile, K step) pairs of this CTA, in order: issue(i) prefetches pair i into ring slot i % kPack
        int64_t total = 0;
        for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) total += ksteps;
        auto pair_at = [&](int64_t i, int& n0, int& ks) {
            const int tl = static_cast<int>(i / ksteps);
            ks = static_cast<int>(i - int64_t(tl) * ksteps);
            const int t = blockIdx.x + tl * gridDim.x;
            n0 = (t / a.tiles_m) * kBW;
        };
        auto issue = [&](int64_t i) {
            if (i < total) {
                int n0, ks;
                pair_at(i, n0, ks);
                const int64_t n = n0 + r;
                uint8_t* dst = pack + ((i % kPack) * kBW + r) * kPB;
                uint32_t* sdst = reinterpret_cast<uint32_t*>(scl + ((i % kPack) * kBW + r) * 8);
                if (n < a.N) {
                    const uint8_t* row = a.B + n * a.row_bytes;
#pragma unroll
                    for (int ch = 0; ch < 2; ++ch) {
                        const int64_t k = int64_t(ks) * kBK + 32 * ch;
                        if (k < kcodes) {
                            if constexpr (BITS == 4) {
                                cp_async16(dst + 16 * ch, row + k / 2);
                            } else {
#pragma unroll
                                for (int q = 0; q < 3; ++q) cp_async4(dst + 12 * ch + 4 * q, row + 3 * k / 8 + 4 * q);
                            }
                            const int64_t si = n * nb + (k >> bs_shift);
                            if (ST == kF32 || (si | 1) < a.N * nb) {
                                cp_async4(sdst + ch, static_cast<const uint32_t*>(a.scales) + (ST == kF32 ? si : (si >> 1)));
                            } else {  // the last half-precision scale: its 4-byte word would run past the array
                                sdst[ch] = static_cast<const uint16_t*>(a.scales)[si];
                            }
                        }
                    }
                }
            }
            cp_async_commit();
        };
        for (int64_t i = 0; i < kPack - 1; ++i) issue(i);
        int64_t i = 0;
        for (int t = blockIdx.x; t < n_tiles && !failed; t += gridDim.x) {
            const int n0 = (t / a.tiles_m) * kBW;
            const int64_t n = n0 + r;
            for (int ks = 0; ks < ksteps; ++ks, ++i) {
                issue(i + kPack - 1);
                cp_async_wait<kPack - 1>();
                const int s = static_cast<int>(i % S);
                if (i >= S && !warp_wait(&empty[s], ((i / S) - 1) & 1)) { failed = true; break; }
                const uint8_t* src = pack + ((i % kPack) * kBW + r) * kPB;
                const uint32_t* ssrc = reinterpret_cast<const uint32_t*>(scl + ((i % kPack) * kBW + r) * 8);
                uint8_t* wdst = wt + s * plan.w;
#pragma unroll
                for (int ch = 0; ch < 2; ++ch) {
                    const int64_t k = int64_t(ks) * kBK + 32 * ch;
                    const bool live = n < a.N && k < kcodes;
                    uint32_t w[BITS];
                    float sc = 0.f, z = float(kZ);
                    if (live) {
#pragma unroll
                        for (int q = 0; q < BITS; ++q) w[q] = reinterpret_cast<const uint32_t*>(src + ch * 4 * BITS)[q];
                        const int b = static_cast<int>(k >> bs_shift);
                        sc = scale_from_word<ST>(ssrc[ch], n * nb + b);
                        if (a.zp) z = float(zero_point_code<BITS>(a.zp + n * a.zp_row_bytes, b));
                    } else {
#pragma unroll
                        for (int q = 0; q < BITS; ++q) w[q] = 0;
                    }
                    // w = s (q - z) = f * s 2^(24-p) - s (2^(23-p) + z), one rounding per value;
                    // the pre-scale depends only on the code's position class p (2 for INT4, 3 for INT3)
                    float mc[3], ac[3];
#pragma unroll
                    for (int c = 0; c < 3; ++c) {
                        const int p = code_pos<BITS>(c);
                        mc[c] = sc * float(1u << (24 - p));
                        ac[c] = -sc * (float(1u << (23 - p)) + z);
                    }
                    constexpr int kCls = BITS == 4 ? 2 : 3;
                    uint32_t outw[16];
#pragma unroll
                    for (int g = 0; g < 8; ++g) {
                        float2 f01, f23;
                        chunk_codes4<BITS>(w, g, f01, f23);
                        const int j = 4 * g;
                        const float2 m01 = make_float2(mc[j % kCls], mc[(j + 1) % kCls]);
                        const float2 a01 = make_float2(ac[j % kCls], ac[(j + 1) % kCls]);
                        const float2 m23 = make_float2(mc[(j + 2) % kCls], mc[(j + 3) % kCls]);
                        const float2 a23 = make_float2(ac[(j + 2) % kCls], ac[(j + 3) % kCls]);
                        const float2 v01 = ffma2(f01, m01, a01);
                        const float2 v23 = ffma2(f23, m23, a23);
                        outw[2 * g] = pack2(v01.x, v01.y, bf16);
                        outw[2 * g + 1] = pack2(v23.x, v23.y, bf16);
                    }
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *reinterpret_cast<uint4*>(wdst + sw128(r, 4 * ch + c)) =
                            make_uint4(outw[4 * c], outw[4 * c + 1], outw[4 * c + 2], outw[4 * c + 3]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&full_w[s]);
            }
        }
        cp_async_wait<0>();
    } else {
        // ----------------------------------------------------------- epilogue
        const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
        int tl = 0;
        for (int t = blockIdx.x; t < n_tiles && !failed; t += gridDim.x, ++tl) {
            const int buf = tl & 1;
            const int n0 = (t / a.tiles_m) * kBW, m0 = (t % a.tiles_m) * BN;
            if (!warp_wait(&acc_full[buf], (tl >> 1) & 1)) { failed = true; break; }
            tc_fence_after();
            const int64_t n = n0 + quarter * 32 + lane;
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(tmem + (uint32_t(quarter * 32) << 16) + buf * BN + c0, v);
                tmem_ld_wait();
                if (n < a.N) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int64_t m = m0 + c0 + j;
                        // a 16-column tile loads 32 columns: the upper 16 belong to the other accumulator
                        if (c0 + j < BN && m < a.M) store_from_f32(a.Y, a.y_dtype, m * a.N + n, __uint_as_float(v[j]));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
        }
    }
    if (failed) record_error(MNB_ERR_TIMEOUT);
    grid_launch_dependents();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, a.tmem_cols);
    }
}

// ------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

template <int BITS, int ST, int BN>
cudaError_t launch_bn(const GemmTcArgs& g, int sm_count, bool pdl, cudaStream_t stream) {
    auto encode = encode_fn();
    if (!encode) return cudaErrorNotSupported;
    CUtensorMap tmap;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(g.K), static_cast<cuuint64_t>(g.M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(g.K * 2)};
    const cuuint32_t box[2] = {kBK, BN};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult cr = encode(&tmap, g.a_dtype == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                               2, const_cast<void*>(g.A), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
    TcArgs a = {};
    a.M = g.M;
    a.K = g.K;
    a.N = g.N;
    a.B = g.B;
    a.scales = g.scales;
    a.zp = g.zp;
    a.row_bytes = g.row_bytes;
    a.nb = g.nb;
    a.bs = g.bs;
    a.zp_row_bytes = g.zp_row_bytes;
    a.a_dtype = g.a_dtype;
    a.Y = g.Y;
    a.y_dtype = g.y_dtype;
    a.tiles_n = static_cast<int>(cdiv<int64_t>(g.N, kBW));
    a.tiles_m = static_cast<int>(cdiv<int64_t>(g.M, BN));
    a.k_steps = static_cast<int>(cdiv<int64_t>(g.K, kBK));
    uint32_t cols = 32;
    while (cols < 2u * BN) cols <<= 1;
    a.tmem_cols = cols;
    int stages = 6;
    while (stages > 2 && tc_plan(BN, stages, BITS).total > 227 * 1024) --stages;
    a.stages = stages;
    const int64_t smem = tc_plan(BN, stages, BITS).total;
    auto kern = gemm_tc_kernel<BITS, ST, BN>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int tiles = a.tiles_n * a.tiles_m;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(std::min(tiles, sm_count)), 1, 1);
    cfg.blockDim = dim3(kThreadsTC, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, tmap, a);
}

// Activation rows per tile: fewest waves of persistent CTAs, weighing the
// lower per-FLOP efficiency of narrow tiles.
int pick_bn(int64_t M, int64_t N, int sm_count) {
    int best = 256;
    double best_cost = 1e300;
    for (int bn : {256, 128, 64, 32, 16}) {
        if (bn > 16 && bn / 2 >= M) continue;  // a narrower tile covers M already
        const int64_t tiles = cdiv<int64_t>(N, kBW) * cdiv<int64_t>(M, bn);
        const double waves = double(cdiv<int64_t>(tiles, sm_count));
        const double eff = bn >= 256 ? 1.0 : bn >= 128 ? 0.9 : bn >= 64 ? 0.7 : 0.5;
        const double cost = waves * bn / eff;
        if (cost < best_cost) { best_cost = cost; best = bn; }
    }
    return best;
}

template <int BITS, int ST>
cudaError_t launch_bits_st(const GemmTcArgs& g, int sm_count, bool pdl, cudaStream_t stream) {
    switch (pick_bn(g.M, g.N, sm_count)) {
        case 256: return launch_bn<BITS, ST, 256>(g, sm_count, pdl, stream);
        case 128: return launch_bn<BITS, ST, 128>(g, sm_count, pdl, stream);
        case 64: return launch_bn<BITS, ST, 64>(g, sm_count, pdl, stream);
        case 32: return launch_bn<BITS, ST, 32>(g, sm_count, pdl, stream);
        default: return launch_bn<BITS, ST, 16>(g, sm_count, pdl, stream);
    }
}

}  // namespace

cudaError_t gemm_tc_take_error(unsigned int* out) { return take_unit_error(out); }

cudaError_t launch_gemm_tc(const GemmTcArgs& g, int scale_dtype, int sm_count, bool pdl, cudaStream_t stream) {
    if (g.bits == 4) {
        if (scale_dtype == kF32) return launch_bits_st<4, kF32>(g, sm_count, pdl, stream);
        if (scale_dtype == kF16) return launch_bits_st<4, kF16>(g, sm_count, pdl, stream);
        return launch_bits_st<4, kBF16>(g, sm_count, pdl, stream);
    }
    if (scale_dtype == kF32) return launch_bits_st<3, kF32>(g, sm_count, pdl, stream);
    if (scale_dtype == kF16) return launch_bits_st<3, kF16>(g, sm_count, pdl, stream);
    return launch_bits_st<3, kBF16>(g, sm_count, pdl, stream);
}

}  // namespace mnb
