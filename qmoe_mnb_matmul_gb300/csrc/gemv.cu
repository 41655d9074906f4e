// gemv.cu -- packed INT4 / INT3 weight-only GEMV (M = 1 decode) and small-M
// matmul on CUDA cores, sm_103a.
//
// Follows "Qwen3 Missing-Kernel Implementation Plan", rows K02/K03: scales and
// zero points are applied while bounded panels of the packed weights are
// consumed; no dequantised weight matrix is ever written to global memory.
//
// Design (HBM-bound: the packed weights and scales are the traffic):
//  * A CTA owns contiguous blocks of RC weight rows.  Because rows are
//    contiguous in the [N, nb, blob] layout, a block's packed bytes and its
//    scales are two contiguous ranges; one thread moves each with a single
//    bulk (TMA) copy into a 2-stage shared-memory ring tracked by mbarriers.
//    The grid is persistent (<= resident CTAs), so the copy of block i+2 is in
//    flight while block i is consumed.
//  * The activations are staged once per CTA, pre-multiplied by 256 (exact),
//    in a chunk-interleaved float4 layout that makes every lane's read
//    conflict-free, together with per-chunk activation sums.
//  * A chunk is 32 consecutive codes of one row (16 bytes of INT4, 12 of INT3).
//    A code q is turned into a float with one byte-permute (INT4) or one
//    shift + one mask (INT3) by placing it in mantissa bits 16.. under
//    exponent 126: f = 0.5 + q/256.  With A' = 256 A this gives
//    A' f = 128 A + A q, so over a chunk
//        sum A (q - z) = sum A' f - (128 + z) sum A,
//    and the scale of the chunk's block multiplies that once.  The products
//    run as packed f32x2 FMAs.  Integer inputs stay exact (all partial sums
//    are integers below 2^24).
//  * A warp owns R rows at a time and walks their chunks with one chunk per
//    lane; the R x MT sums are reduced with shuffles in a fixed order, so
//    results are deterministic.
#include <algorithm>

#include "common.cuh"
#include "gemv_core.cuh"
#include "kernels.h"

namespace mnb {

namespace {

using namespace gemv;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kStages = 2;
constexpr int kRowsPerWarp = 4;                 // R
struct Plan {
    int64_t a4_bytes, asum_bytes, w_stage, s_stage, total;
};

__host__ __device__ inline Plan make_plan(int MT, int C, int RC, int64_t row_bytes, int nb, int ssize) {
    Plan p;
    p.a4_bytes = int64_t(MT) * 8 * C * 16;
    p.asum_bytes = round_up(int64_t(MT) * C * 4, 128);
    p.w_stage = round_up(int64_t(RC) * row_bytes, 128);
    p.s_stage = round_up(int64_t(RC) * nb * ssize, 128);
    p.total = 128 + p.a4_bytes + p.asum_bytes + kStages * (p.w_stage + p.s_stage);
    return p;
}

template <int BITS, int ST, int MT>
__global__ void __launch_bounds__(kThreads) gemv_kernel(const __grid_constant__ GemvArgs a) {
    using S = typename DType<ST>::T;
    constexpr int R = kRowsPerWarp;
    extern __shared__ __align__(128) uint8_t smem[];

    const int C = a.chunks, RC = a.rows_per_block, nb = a.nb;
    const Plan plan = make_plan(MT, C, RC, a.row_bytes, nb, sizeof(S));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
    float4* A4 = reinterpret_cast<float4*>(smem + 128);
    float* Asum = reinterpret_cast<float*>(smem + 128 + plan.a4_bytes);
    uint8_t* Wst = smem + 128 + plan.a4_bytes + plan.asum_bytes;
    uint8_t* Sst = Wst + kStages * plan.w_stage;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t m0 = int64_t(blockIdx.y) * MT;

    auto block_rows = [&](int blk) -> int {
        const int64_t n0 = int64_t(blk) * RC;
        return static_cast<int>(a.N - n0 < RC ? a.N - n0 : int64_t(RC));
    };
    auto issue = [&](int blk, int st) {
        const int64_t n0 = int64_t(blk) * RC;
        const int rc = block_rows(blk);
        const uint32_t wb = static_cast<uint32_t>(rc * a.row_bytes) & ~15u;
        const uint32_t sb = static_cast<uint32_t>(int64_t(rc) * nb * sizeof(S)) & ~15u;
        mbar_arrive_expect_tx(&bars[st], wb + sb);
        if (wb) bulk_g2s(Wst + st * plan.w_stage, a.B + n0 * a.row_bytes, wb, &bars[st]);
        if (sb)
            bulk_g2s(Sst + st * plan.s_stage, static_cast<const S*>(a.scales) + n0 * nb, sb, &bars[st]);
    };

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
        fence_barrier_init();
        // Warm L2 with this CTA's first blocks while the previous kernel drains.
        for (int i = 0; i < kStages; ++i) {
            const int blk = blockIdx.x + i * gridDim.x;
            if (blk >= a.n_blocks) break;
            const uint32_t wb = static_cast<uint32_t>(block_rows(blk) * a.row_bytes) & ~15u;
            if (wb) bulk_prefetch_l2(a.B + int64_t(blk) * RC * a.row_bytes, wb);
        }
    }
    grid_dependency_wait();
    __syncthreads();
    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            const int blk = blockIdx.x + i * gridDim.x;
            if (blk < a.n_blocks) issue(blk, i);
        }
    }

    // Stage A' = 256 A (zero beyond K and beyond M) and the per-chunk sums.
    stage_activations<MT>(
        A4, Asum, C,
        [&](int m, int64_t k) -> float {
            return (m0 + m < a.M && k < a.K) ? load_as_f32(a.A, a.a_dtype, (m0 + m) * a.K + k) : 0.f;
        },
        tid, kThreads);
    grid_launch_dependents();

    const int bs_shift = __ffs(a.bs) - 1;
    constexpr int kZImplicit = 1 << (BITS - 1);

    for (int it = 0;; ++it) {
        const int blk = blockIdx.x + it * gridDim.x;
        if (blk >= a.n_blocks) break;
        const int st = it % kStages;
        const uint32_t parity = (it / kStages) & 1;
        const bool ok = mbar_wait(&bars[st], parity);
        if (__syncthreads_or(!ok)) {
            // A bulk copy never completed; leave after giving in-flight copies a bounded chance.
            mbar_wait(&bars[st], parity);
            return;
        }
        const int64_t n0 = int64_t(blk) * RC;
        const int rc = block_rows(blk);
        uint8_t* W = Wst + st * plan.w_stage;
        const S* Sc = reinterpret_cast<const S*>(Sst + st * plan.s_stage);
        {   // bytes past the last 16-byte multiple of a partial block come in with plain loads
            const int64_t wtot = rc * a.row_bytes, stot = int64_t(rc) * nb * sizeof(S);
            const int64_t wb = wtot & ~int64_t(15), sb = stot & ~int64_t(15);
            if (wtot != wb || stot != sb) {
                for (int64_t i = wb + tid; i < wtot; i += kThreads) W[i] = a.B[n0 * a.row_bytes + i];
                const uint8_t* sg = reinterpret_cast<const uint8_t*>(static_cast<const S*>(a.scales) + n0 * nb);
                for (int64_t i = sb + tid; i < stot; i += kThreads) Sst[st * plan.s_stage + i] = sg[i];
                __syncthreads();
            }
        }

        for (int g = warp; g * R < rc; g += kWarps) {
            float out[R][MT];
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int m = 0; m < MT; ++m) out[r][m] = 0.f;

            for (int c = lane; c < C; c += 32) {
                const int b = (c * 32) >> bs_shift;
                uint32_t w[R][BITS];
                float sc[R], zz[R];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int rl = min(g * R + r, rc - 1);   // rows past the block end recompute the last row
                    load_chunk<BITS>(W + int64_t(rl) * a.row_bytes, c, w[r]);
                    sc[r] = to_f32(Sc[rl * nb + b]);
                    zz[r] = float(a.zp ? zero_point_code<BITS>(a.zp + (n0 + rl) * a.zp_row_bytes, b) : kZImplicit);
                }
                chunk_accumulate<BITS, R, MT>(w, sc, zz, A4, Asum, C, c, out);
            }
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int m = 0; m < MT; ++m) out[r][m] = warp_sum(out[r][m]);
            if (lane == 0) {
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int rl = g * R + r;
                    if (rl >= rc) break;
#pragma unroll
                    for (int m = 0; m < MT; ++m)
                        if (m0 + m < a.M) store_from_f32(a.Y, a.y_dtype, (m0 + m) * a.y_ld + n0 + rl, out[r][m]);
                }
            }
        }
        __syncthreads();  // every warp is done with stage st
        if (tid == 0) {
            const int nxt = blk + kStages * gridDim.x;
            if (nxt < a.n_blocks) {
                fence_proxy_async_smem();
                issue(nxt, st);
            }
        }
    }
}

template <int BITS, int ST, int MT>
cudaError_t launch_typed(const GemvArgs& a, int sm_count, bool pdl, cudaStream_t stream, int64_t smem) {
    auto kern = gemv_kernel<BITS, ST, MT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, static_cast<size_t>(smem));
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorNotSupported;
    const int64_t mgroups = cdiv<int64_t>(a.M, MT);
    int64_t gx = std::min<int64_t>(a.n_blocks, std::max<int64_t>(1, int64_t(sm_count) * per_sm / mgroups));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(gx), static_cast<unsigned>(mgroups), 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

int pick_mt(int64_t M) { return M <= 1 ? 1 : (M <= 2 ? 2 : 4); }

int ssize_of(int dt) { return dt == kF32 ? 4 : 2; }

// Alignment unit of a row block: the smallest row count (a multiple of the
// warp row group) for which every block's packed bytes and scales start on a
// 16-byte boundary.
int64_t row_unit(int64_t row_bytes, int nb, int ssize) {
    auto g16 = [](int64_t x) { int64_t g = 16; while (x % g) g >>= 1; return 16 / g; };
    return std::max<int64_t>(kRowsPerWarp, std::max(g16(row_bytes), g16(int64_t(nb) * ssize)));
}

// Rows per stage: about 16 KB of packed weights, a multiple of the alignment
// unit, shrunk while the grid would leave SMs idle.
int pick_rows(int64_t N, int64_t row_bytes, int nb, int ssize, int sm_count) {
    const int64_t unit = row_unit(row_bytes, nb, ssize);
    int64_t rc = std::max<int64_t>(unit, (16384 / std::max<int64_t>(row_bytes, 1)) / unit * unit);
    rc = std::max<int64_t>(unit, std::min<int64_t>(rc, 64) / unit * unit);
    while (rc > unit && cdiv<int64_t>(N, rc) < 2 * sm_count) rc -= unit;
    return static_cast<int>(rc);
}

}  // namespace

cudaError_t gemv_take_error(unsigned int* out) { return take_unit_error(out); }

size_t gemv_smem_bytes(int64_t M, int64_t K, int bits, int bs, int scale_dtype) {
    const int nb = static_cast<int>(cdiv<int64_t>(K, bs));
    const int C = nb * bs / 32;
    const int64_t row_bytes = int64_t(nb) * bs * bits / 8;
    const Plan p = make_plan(pick_mt(M), C, static_cast<int>(row_unit(row_bytes, nb, ssize_of(scale_dtype))),
                             row_bytes, nb, ssize_of(scale_dtype));
    return p.total <= 227 * 1024 ? static_cast<size_t>(p.total) : 0;
}

cudaError_t launch_gemv(const GemvArgs& in, int scale_dtype, int sm_count, bool pdl, cudaStream_t stream) {
    GemvArgs a = in;
    const int ssize = ssize_of(scale_dtype);
    const int MT = pick_mt(a.M);
    a.rows_per_block = pick_rows(a.N, a.row_bytes, a.nb, ssize, sm_count);
    Plan p = make_plan(MT, a.chunks, a.rows_per_block, a.row_bytes, a.nb, ssize);
    const int unit = static_cast<int>(row_unit(a.row_bytes, a.nb, ssize));
    while (p.total > 227 * 1024 && a.rows_per_block > unit) {
        a.rows_per_block = std::max(unit, a.rows_per_block / 2 / unit * unit);
        p = make_plan(MT, a.chunks, a.rows_per_block, a.row_bytes, a.nb, ssize);
    }
    if (p.total > 227 * 1024) return cudaErrorNotSupported;
    a.n_blocks = static_cast<int>(cdiv<int64_t>(a.N, a.rows_per_block));

#define MNB_GEMV_DISPATCH(BITS, ST)                                                   \
    switch (MT) {                                                                     \
        case 1: return launch_typed<BITS, ST, 1>(a, sm_count, pdl, stream, p.total); \
        case 2: return launch_typed<BITS, ST, 2>(a, sm_count, pdl, stream, p.total); \
        default: return launch_typed<BITS, ST, 4>(a, sm_count, pdl, stream, p.total); \
    }
    if (a.bits == 4) {
        if (scale_dtype == kF32) { MNB_GEMV_DISPATCH(4, kF32) }
        if (scale_dtype == kF16) { MNB_GEMV_DISPATCH(4, kF16) }
        MNB_GEMV_DISPATCH(4, kBF16)
    } else {
        if (scale_dtype == kF32) { MNB_GEMV_DISPATCH(3, kF32) }
        if (scale_dtype == kF16) { MNB_GEMV_DISPATCH(3, kF16) }
        MNB_GEMV_DISPATCH(3, kBF16)
    }
#undef MNB_GEMV_DISPATCH
}

}  // namespace mnb
