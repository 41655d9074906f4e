// gemv.cu -- packed INT4 / INT3 weight-only GEMV (M = 1 decode) and small-M
// matmul on CUDA cores, sm_103a.
//
// Follows "Qwen3 Missing-Kernel Implementation Plan", rows K02/K03: scales and
// zero points are applied while bounded panels of the packed weights are
// consumed; no dequantised weight matrix is ever written to global memory.
//
// Design (HBM-bound: the packed weights and scales are the traffic):
//  * A CTA owns contiguous blocks of RC = 8 * R weight rows.  Rows are
//    contiguous in the [N, nb, blob] layout, so a block's packed bytes and its
//    scales are two contiguous ranges, each moved by one bulk (TMA) copy.
//  * Warp 8 is the producer: one lane keeps a ring of NST stages filled,
//    waiting on per-stage "empty" mbarriers; the 8 consumer warps wait on the
//    per-stage "full" mbarriers.  There is no block-wide barrier in the loop.
//    The grid is persistent (<= resident CTAs).
//  * The activations are staged once per CTA (gemv_core.cuh); each consumer
//    warp owns R rows of a block and walks their 32-code chunks, one chunk
//    per lane; the R x MT sums are reduced together with shuffles that hand
//    half of the values to the partner lane at each step (fixed order, so
//    results are deterministic).
//  * Before the grid-dependency wait each CTA only warms L2 with its first
//    blocks (a prefetch cannot observe stale data), so a programmatic
//    dependent launch overlaps that traffic with the previous kernel.
#include <algorithm>

#include "common.cuh"
#include "gemv_core.cuh"
#include "kernels.h"

namespace mnb {

namespace {

using namespace gemv;

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxStages = 8;
constexpr int64_t kSmemBudget = 227 * 1024;

struct Plan {
    int64_t a4, sums, w_stage, s_stage, fixed;
    int stages;
    int64_t total;
};

__host__ __device__ inline Plan make_plan(int MT, int C, int RC, int64_t row_bytes, int nb, int ssize, int stages) {
    Plan p;
    p.a4 = a4_bytes(MT, C);
    p.sums = round_up(int64_t(MT) * C * 16, 128);  // one float4 correction per (row, chunk)
    p.w_stage = round_up(int64_t(RC) * row_bytes, 128);
    p.s_stage = round_up(int64_t(RC) * nb * ssize, 128);
    p.fixed = 256 + p.a4 + p.sums;
    p.stages = stages;
    p.total = p.fixed + int64_t(stages) * (p.w_stage + p.s_stage);
    return p;
}

// dst[i] = src[i] for i in [from, to): the sub-16-byte tail of a block, out of line.
static __device__ __noinline__ void copy_bytes(uint8_t* dst, const uint8_t* src, int64_t from, int64_t to) {
    for (int64_t i = from; i < to; ++i) dst[i] = src[i];
}

// Named barrier over the consumer warps only.
__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

template <int BITS, int ST, int MT, int R>
__global__ void __launch_bounds__(kThreads) gemv_kernel(const __grid_constant__ GemvArgs a) {
    using S = typename DType<ST>::T;
    constexpr int RC = kConsumerWarps * R;
    extern __shared__ __align__(128) uint8_t smem[];

    const int C = a.chunks, nb = a.nb;
    const Plan plan = make_plan(MT, C, RC, a.row_bytes, nb, sizeof(S), a.stages);
    const int NST = plan.stages;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kMaxStages;
    float4* A4 = reinterpret_cast<float4*>(smem + 256);
    float4* Corr = reinterpret_cast<float4*>(smem + 256 + plan.a4);
    uint8_t* Wst = smem + plan.fixed;
    uint8_t* Sst = Wst + NST * plan.w_stage;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t m0 = int64_t(blockIdx.y) * MT;
    const int nblk = a.n_blocks;
    auto block_rows = [&](int blk) -> int {
        const int64_t left = a.N - int64_t(blk) * RC;
        return static_cast<int>(left < RC ? left : int64_t(RC));
    };

    if (tid == kConsumerWarps * 32) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        fence_barrier_init();
        for (int i = 0; i < NST; ++i) {
            const int blk = blockIdx.x + i * gridDim.x;
            if (blk >= nblk) break;
            const uint32_t wb = static_cast<uint32_t>(block_rows(blk) * a.row_bytes) & ~15u;
            if (wb) bulk_prefetch_l2(a.B + int64_t(blk) * RC * a.row_bytes, wb);
        }
    }
    grid_dependency_wait();
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------- producer
        if (lane != 0) return;
        int st = 0;
        uint32_t round = 0;  // times the ring has wrapped
        for (int blk = blockIdx.x; blk < nblk; blk += gridDim.x) {
            if (round && !mbar_wait(&empty[st], (round - 1) & 1)) {
                for (int j = 0; j < NST; ++j) mbar_wait(&full[j], 0);  // give in-flight copies a bounded chance
                return;
            }
            const int64_t n0 = int64_t(blk) * RC;
            const int rc = block_rows(blk);
            uint8_t* W = Wst + st * plan.w_stage;
            uint8_t* Sd = Sst + st * plan.s_stage;
            const int64_t wtot = rc * a.row_bytes, stot = int64_t(rc) * nb * sizeof(S);
            const uint32_t wb = static_cast<uint32_t>(wtot) & ~15u, sb = static_cast<uint32_t>(stot) & ~15u;
            const uint8_t* wsrc = a.B + n0 * a.row_bytes;
            const uint8_t* ssrc = reinterpret_cast<const uint8_t*>(static_cast<const S*>(a.scales) + n0 * nb);
            // bytes past the last 16-byte multiple of a partial block: plain copies, published by the arrive below
            if (wb < wtot) copy_bytes(W, wsrc, wb, wtot);
            if (sb < stot) copy_bytes(Sd, ssrc, sb, stot);
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&full[st], wb + sb);
            if (wb) bulk_g2s(W, wsrc, wb, &full[st]);
            if (sb) bulk_g2s(Sd, ssrc, sb, &full[st]);
            if (++st == NST) { st = 0; ++round; }
        }
        return;
    }

    // ------------------------------------------------------------ consumers
    stage_chunks<BITS, MT>(
        A4, Corr, C, a.K, a.a_dtype, a.a_vec != 0,
        [&](int m) -> const void* {
            return m0 + m < a.M ? static_cast<const char*>(a.A) + (m0 + m) * a.K * (a.a_dtype == kF32 ? 4 : 2)
                                : nullptr;
        },
        tid, kConsumerWarps * 32);
    consumer_sync();
    grid_launch_dependents();

    const int bs_shift = __ffs(a.bs) - 1;
    const int mstride = a4_groups(C) * 256;
    constexpr int kZImplicit = 1 << (BITS - 1);
    int st = 0;
    uint32_t phase = 0;
    for (int blk = blockIdx.x; blk < nblk; blk += gridDim.x) {
        if (!warp_wait(&full[st], phase)) return;
        const int64_t n0 = int64_t(blk) * RC;
        const int rc = block_rows(blk);
        const uint8_t* W = Wst + st * plan.w_stage;
        const S* Sc = reinterpret_cast<const S*>(Sst + st * plan.s_stage);
        const int r0 = warp * R;
        if (r0 < rc) {
            float2 acc[R][MT];
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int m = 0; m < MT; ++m) acc[r][m] = make_float2(0.f, 0.f);
            const uint8_t* wrow[R];
            const S* srow[R];
            const uint8_t* zrow[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int rl = min(r0 + r, rc - 1);  // rows past the block end recompute the last row
                wrow[r] = W + int64_t(rl) * a.row_bytes;
                srow[r] = Sc + rl * nb;
                zrow[r] = a.zp ? a.zp + (n0 + rl) * a.zp_row_bytes : nullptr;
            }
            auto load = [&](int c, uint32_t (&w)[R][BITS], float (&sc)[R], float (&dz)[R]) {
                const int b = (c * 32) >> bs_shift;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    load_chunk<BITS>(wrow[r], c, w[r]);
                    sc[r] = to_f32(srow[r][b]);
                    dz[r] = a.zp ? float(kZImplicit - zero_point_code<BITS>(zrow[r], b)) : 0.f;
                }
            };
            for (int c = lane; c < C; c += 32) {
                uint32_t w[R][BITS];
                float sc[R], dz[R];
                load(c, w, sc, dz);
                chunk_accumulate<BITS, R, MT>(w, sc, dz, A4 + a4_base(0, c, C), mstride, Corr + c, C, acc);
            }
            // value q = r * MT + m; each total ends in one lane
            constexpr int N = R * MT;
            float part[N];
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int m = 0; m < MT; ++m) part[r * MT + m] = acc[r][m].x + acc[r][m].y;
            const float total = warp_sum_transpose<N>(part);
            if ((lane & (32 / N - 1)) == 0) {
                const int q = transpose_row<N>(lane), r = q / MT, m = q - r * MT;
                if (r0 + r < rc && m0 + m < a.M) store_from_f32(a.Y, a.y_dtype, (m0 + m) * a.y_ld + n0 + r0 + r, total);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
        if (++st == NST) { st = 0; phase ^= 1; }
    }
}

int ssize_of(int dt) { return dt == kF32 ? 4 : 2; }

int pick_mt(int64_t M) { return M <= 1 ? 1 : (M <= 2 ? 2 : 4); }

// The smallest row count for which every block's packed bytes and scales
// start on a 16-byte boundary (a power of two).
int64_t row_align(int64_t row_bytes, int nb, int ssize) {
    auto g16 = [](int64_t x) { int64_t g = 16; while (x % g) g >>= 1; return 16 / g; };
    return std::max(g16(row_bytes), g16(int64_t(nb) * ssize));
}

// Launch shape: rows per warp R and ring depth.  Each CTA wants ~48 KB of
// weights in flight and the SM wants up to 3 resident CTAs; the largest R
// that still gives >= 0.8 blocks per SM wins.  Measured on the decode
// projections: fewer, larger blocks beat more CTAs per SM there (every CTA
// stages the whole activation row), e.g. 2048 -> 4096 in 3.8 us with 128
// 32-row blocks against 4.9 us with 256 16-row blocks.
struct Shape {
    int R = 4, stages = 2;
};
constexpr int64_t kSmSmem = 228 * 1024, kCtaReserve = 1024;

Shape pick_shape(int64_t N, int64_t row_bytes, int nb, int ssize, int MT, int C, int sm_count) {
    const int64_t align = row_align(row_bytes, nb, ssize);
    Shape best;
    int64_t best_score = -1;
    for (int R : {4, 2, 1}) {
        const int RC = kConsumerWarps * R;
        if (RC % align != 0) continue;
        const Plan p1 = make_plan(MT, C, RC, row_bytes, nb, ssize, 1);
        const int64_t stage = p1.w_stage + p1.s_stage;
        if (p1.fixed + 2 * stage > kSmemBudget) continue;
        int st = static_cast<int>(std::min<int64_t>(kMaxStages, std::max<int64_t>(2, cdiv<int64_t>(49152, stage))));
        while (st > 2 && p1.fixed + st * stage > kSmemBudget) --st;
        auto ctas = [&](int s) { return kSmSmem / (p1.fixed + s * stage + kCtaReserve); };
        while (st > 2 && ctas(st) < 3 && ctas(st - 1) > ctas(st)) --st;
        const int64_t resident = std::min<int64_t>(3, ctas(st));
        const bool enough_blocks = cdiv<int64_t>(N, RC) * 5 >= int64_t(sm_count) * 4;
        const int64_t score = (enough_blocks ? 100 : 0) + 10 * R + resident;
        if (score > best_score) {
            best_score = score;
            best.R = R;
            best.stages = st;
        }
    }
    return best;
}

template <int BITS, int ST, int MT, int R>
cudaError_t launch_typed(GemvArgs a, int stages, int sm_count, bool pdl, cudaStream_t stream) {
    constexpr int RC = kConsumerWarps * R;
    const int ssize = ST == kF32 ? 4 : 2;
    a.rows_per_block = RC;
    a.n_blocks = static_cast<int>(cdiv<int64_t>(a.N, RC));
    const Plan p1 = make_plan(MT, a.chunks, RC, a.row_bytes, a.nb, ssize, 1);
    if (p1.fixed + int64_t(stages) * (p1.w_stage + p1.s_stage) > kSmemBudget) return cudaErrorNotSupported;
    a.stages = stages;
    const int st = stages;
    const Plan p = make_plan(MT, a.chunks, RC, a.row_bytes, a.nb, ssize, st);
    auto kern = gemv_kernel<BITS, ST, MT, R>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(p.total));
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, static_cast<size_t>(p.total));
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorNotSupported;
    const int64_t mgroups = cdiv<int64_t>(a.M, MT);
    const int64_t gx = std::min<int64_t>(a.n_blocks, std::max<int64_t>(1, int64_t(sm_count) * per_sm / mgroups));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(gx), static_cast<unsigned>(mgroups), 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(p.total);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int BITS, int ST, int MT>
cudaError_t launch_r(const GemvArgs& a, const Shape& sh, int sm_count, bool pdl, cudaStream_t stream) {
    if (sh.R == 4) return launch_typed<BITS, ST, MT, 4>(a, sh.stages, sm_count, pdl, stream);
    if (sh.R == 2) return launch_typed<BITS, ST, MT, 2>(a, sh.stages, sm_count, pdl, stream);
    return launch_typed<BITS, ST, MT, 1>(a, sh.stages, sm_count, pdl, stream);
}

template <int BITS, int ST>
cudaError_t launch_mt(const GemvArgs& a, int sm_count, bool pdl, cudaStream_t stream) {
    const int MT = pick_mt(a.M);
    const Shape sh = pick_shape(a.N, a.row_bytes, a.nb, ST == kF32 ? 4 : 2, MT, a.chunks, sm_count);
    switch (MT) {
        case 1: return launch_r<BITS, ST, 1>(a, sh, sm_count, pdl, stream);
        case 2: return launch_r<BITS, ST, 2>(a, sh, sm_count, pdl, stream);
        default: return launch_r<BITS, ST, 4>(a, sh, sm_count, pdl, stream);
    }
}

}  // namespace

cudaError_t gemv_take_error(unsigned int* out) { return take_unit_error(out); }

size_t gemv_smem_bytes(int64_t M, int64_t K, int bits, int bs, int scale_dtype) {
    const int nb = static_cast<int>(cdiv<int64_t>(K, bs));
    const int C = nb * bs / 32;
    const int64_t row_bytes = int64_t(nb) * bs * bits / 8;
    const int ssize = ssize_of(scale_dtype);
    const int64_t RC = std::max<int64_t>(kConsumerWarps, row_align(row_bytes, nb, ssize));
    const Plan p = make_plan(pick_mt(M), C, static_cast<int>(RC), row_bytes, nb, ssize, 2);
    return p.total <= kSmemBudget ? static_cast<size_t>(p.total) : 0;
}

cudaError_t launch_gemv(const GemvArgs& a, int scale_dtype, int sm_count, bool pdl, cudaStream_t stream) {
    if (a.bits == 4) {
        if (scale_dtype == kF32) return launch_mt<4, kF32>(a, sm_count, pdl, stream);
        if (scale_dtype == kF16) return launch_mt<4, kF16>(a, sm_count, pdl, stream);
        return launch_mt<4, kBF16>(a, sm_count, pdl, stream);
    }
    if (scale_dtype == kF32) return launch_mt<3, kF32>(a, sm_count, pdl, stream);
    if (scale_dtype == kF16) return launch_mt<3, kF16>(a, sm_count, pdl, stream);
    return launch_mt<3, kBF16>(a, sm_count, pdl, stream);
}

}  // namespace mnb
