// qmoe.cu -- one QMoE expert-FFN layer ("INT3 QMoE CUDA correctness baseline
// and Qwen experimental results", Summary and "P1: Compatible QMoE v1
// Extension"): routing, FC1 (fused gate/up) with SwiGLU, FC2 (down
// projection) and the weighted combine, on packed INT3/INT4 experts that are
// dequantised while their rows are consumed -- no dequantised expert matrix is
// ever written to global memory ("prohibit all-expert floating-weight
// materialization").
//
// Plans:
//  * decode (one token, or two; k <= 8), SIMT, on the packed-row machinery of
//    gemv_core.cuh: one token takes the fused single-pass kernel
//    (qmoe_decode.cu) where its shape rules allow, else two kernels.  Every CTA
//    routes its own token (the whole CTA ranks up to 256 logits at once), so
//    no routing kernel sits on the critical path.  FC1 runs over (token, slot)
//    x row blocks of the selected expert and writes h = silu(gate) * up in
//    fp32.  FC2 runs over tokens x row blocks, stages the block's rows of all k
//    selected experts and folds the weighted combine into its epilogue (fixed
//    slot order).  Both are launched as programmatic dependents: before its
//    dependency wait each CTA routes and starts the bulk copies of its expert
//    rows into shared memory.
//  * grouped CUDA-core (3 or more tokens with at most 1.5 routed rows per
//    expert on average, or X rows off a 16-byte boundary; gemv_grouped.cu):
//    route -> permutation -> m-tiles of <= 4 sorted rows of one expert -> FC1
//    (+SwiGLU) and FC2 as GEMV rings over each tile's expert -> combine by
//    token in fixed slot order.
//  * tensor-core (more rows per expert, 16-byte-aligned fp16/bf16 activation
//    rows): route -> expert-sorted permutation -> m-tiles of <= 256 routed rows
//    of one expert -> the routed rows copied into sorted order -> grouped
//    tcgen05 FC1 (SwiGLU in the epilogue) -> grouped FC2 -> combine by token
//    in fixed slot order.
//  * tiled SIMT (what neither of the last two takes): route -> permutation ->
//    tiles of <= 4 pairs of one expert -> FC1 tiles (gathered activations) ->
//    FC2 tiles -> combine by token in fixed slot order.
#include <algorithm>

#include "common.cuh"
#include "gemv_core.cuh"
#include "kernels.h"
#include "qmoe.h"
#include "route_core.cuh"

namespace mnb {

namespace {

using namespace gemv;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int R = 4;            // rows per warp unit (two gate/up pairs in FC1)
constexpr int kTileM = 4;       // pairs per tile in the tiled plan
constexpr int kDecodeMaxT = 8;
constexpr int kDecodeMaxK = 8;
constexpr int kPairsPerBlock = 16;  // FC1 gate/up pairs per CTA (32 rows)
constexpr int kRowsPerBlock2 = 16;  // FC2 rows per CTA (tiled plan)
constexpr int kDecodeRows2 = 8;     // FC2 rows per CTA (decode plan)

__host__ __device__ inline int64_t a256(int64_t x) { return (x + 255) / 256 * 256; }

struct Ws {
    int64_t idx, wts, counts, offsets, perm, inv, chunkc, tiles, ntiles, mtiles, nmtiles, h, o, sync, total;
};

__host__ __device__ inline int64_t max_tiles(int64_t P, int64_t E) {
    const int64_t t = (P + kTileM - 1) / kTileM + E;
    return P < t ? P : t;
}

// m-tiles: <= tile_m sorted pairs of one expert, tile_m in [32, 256] on the
// tensor-core plan (grouped_tile_m) and kGroupedGemvRows on the grouped CUDA-core
// plan; the workspace holds enough for the shortest.
constexpr int kMinTileM = kGroupedGemvRows;
// Routed pairs up to which one CTA sorts the pairs and builds the m-tiles.
constexpr int64_t kOneCtaPlanPairs = 8192;
// Mean routed rows per expert up to which the grouped CUDA-core plan beats the
// tensor-core plan: 3/2 (30B-A3B layer, INT3: 180 vs 215 us at 1 row per
// expert, 225 vs 249 us at 1.5, 273 vs 255 us at 2).
constexpr int64_t kGroupedMeanNum = 3, kGroupedMeanDen = 2;
constexpr int64_t kGroupedMinT = 3;
__host__ __device__ inline int64_t max_mtiles(int64_t P, int64_t E) {
    const int64_t t = (P + kMinTileM - 1) / kMinTileM + E;
    return P < t ? P : t;
}

__host__ __device__ inline Ws ws_layout(int64_t T, int64_t H, int64_t I, int64_t E, int k) {
    const int64_t P = T * k;
    Ws w;
    int64_t off = 0;
    w.idx = off; off += a256(P * 4);
    w.wts = off; off += a256(P * 4);
    w.counts = off; off += a256(E * 4);
    w.offsets = off; off += a256((E + 1) * 4);
    w.perm = off; off += a256(P * 4);
    w.inv = off; off += a256(P * 4);
    w.chunkc = off; off += a256(((P + 255) / 256) * E * 4);  // chunk histograms of the permutation
    w.tiles = off; off += a256(max_tiles(P, E) * 8);
    w.ntiles = off; off += 256;
    w.mtiles = off; off += a256(max_mtiles(P, E) * 16);
    w.nmtiles = off; off += 256;
    w.h = off; off += a256(P * I * 4);
    w.o = off; off += a256(P * H * 4);
    w.sync = off; off += 256;  // the fused decode kernel's grid barrier counter
    w.total = off;
    return w;
}

bool use_decode(const QmoeArgs& q) { return q.T <= kDecodeMaxT && q.k <= kDecodeMaxK; }

// Tensor-core plan: gathered activation rows are read with 16-byte copies.
bool use_tc(const QmoeArgs& q) { return q.x_vec != 0; }

// The grouped CUDA-core projections of a layer (see gemv_grouped.cu); the
// caller completes the tile and workspace fields.
void grouped_args(const QmoeArgs& q, GemvArgs& g1, GemvArgs& g2) {
    const int64_t I = q.I, H = q.H;
    g1 = {};
    g1.A = q.X;
    g1.a_dtype = q.act_dtype;
    g1.K = H;
    g1.B = q.fc1_w;
    g1.scales = q.fc1_s;
    g1.zp = q.fc1_zp;
    g1.N = 2 * I;
    g1.bits = q.fc1_bits;
    g1.bs = q.bs;
    g1.nb = static_cast<int>(q.fc1.nb);
    g1.row_bytes = q.fc1.row_bytes;
    g1.zp_row_bytes = static_cast<int>(q.fc1.zp_row);
    g1.y_dtype = kF32;
    g1.y_ld = I;
    g1.chunks = static_cast<int>(q.fc1.nb * q.bs / 32);
    g1.a_vec = q.x_vec;
    g1.swiglu = 1;
    g1.fc1_inter = q.fc1_layout == MNB_FC1_INTERLEAVED;
    g1.pairs = I;
    g1.g_k = q.k;
    g1.w_estride = 2 * I * q.fc1.row_bytes;
    g1.s_estride = 2 * I * q.fc1.nb * 2;
    g1.z_estride = 2 * I * q.fc1.zp_row;
    g1.bias = q.fc1_bias;
    g1.bias_dtype = q.act_dtype;
    g2 = {};
    g2.a_dtype = kF32;  // h
    g2.K = I;
    g2.B = q.fc2_w;
    g2.scales = q.fc2_s;
    g2.zp = q.fc2_zp;
    g2.N = H;
    g2.bits = q.fc2_bits;
    g2.bs = q.bs;
    g2.nb = static_cast<int>(q.fc2.nb);
    g2.row_bytes = q.fc2.row_bytes;
    g2.zp_row_bytes = static_cast<int>(q.fc2.zp_row);
    g2.y_dtype = kF32;
    g2.y_ld = H;
    g2.chunks = static_cast<int>(q.fc2.nb * q.bs / 32);
    g2.a_vec = I % 4 == 0;  // h rows start on 16-byte boundaries
    g2.w_estride = H * q.fc2.row_bytes;
    g2.s_estride = H * q.fc2.nb * 2;
    g2.z_estride = H * q.fc2.zp_row;
    g2.bias = q.fc2_bias;
    g2.bias_dtype = q.act_dtype;
}

// Grouped CUDA-core plan: few routed rows per expert (or activation rows the
// tensor-core plan cannot load), every expert's block start on a 16-byte
// boundary for the bulk copies, and a shared-memory plan that fits.
bool use_grouped(const QmoeArgs& q) {
    const int64_t P = q.T * q.k;
    if (kGroupedMeanDen * P > kGroupedMeanNum * q.E && q.x_vec) return false;
    if (max_mtiles(P, q.E) > 65535) return false;
    const int64_t s1 = q.fc1.nb * 2, s2 = q.fc2.nb * 2;  // scale bytes per row
    if ((2 * q.I * q.fc1.row_bytes) % 16 || (2 * q.I * s1) % 16 || (q.H * q.fc2.row_bytes) % 16 || (q.H * s2) % 16)
        return false;
    // concatenated gate/up halves are copied as separate row ranges
    if (q.fc1_layout != MNB_FC1_INTERLEAVED && (q.fc1.row_bytes % 16 || s1 % 16)) return false;
    GemvArgs g1, g2;
    grouped_args(q, g1, g2);
    return gemv_grouped_fits(g1, q.act_dtype) && gemv_grouped_fits(g2, q.act_dtype);
}

// --------------------------------------------------------- shared memory

struct Fc1Plan {
    int64_t a4, asum, w, s, lg, total;
};
__host__ __device__ inline Fc1Plan fc1_plan(int MT, int C, int64_t row_bytes, int nb, int ssize) {
    Fc1Plan p;
    p.a4 = a4_bytes(MT, C);
    p.asum = round_up(int64_t(MT) * C * 16, 128);  // float4 corrections
    p.w = round_up(int64_t(2 * kPairsPerBlock) * row_bytes, 128);
    p.s = round_up(int64_t(2 * kPairsPerBlock) * nb * ssize, 128);
    p.lg = round_up(int64_t(kBlockRouteMaxE) * 4, 128);  // router logits (decode)
    p.total = 256 + p.a4 + p.asum + p.w + p.s + p.lg;
    return p;
}

// FC2 plan for `rows` output rows per CTA and ACT activation rows; the decode
// kernel adds one fp32 partial per (slot, row) and the router logits.
struct Fc2Plan {
    int64_t a4, asum, w, s, part, lg, total;
};
__host__ __device__ inline Fc2Plan fc2_plan(int rows, int ACT, int C, int64_t row_bytes, int nb, int ssize,
                                            bool decode) {
    Fc2Plan p;
    p.a4 = a4_bytes(ACT, C);
    p.asum = round_up(int64_t(ACT) * C * 16, 128);  // float4 corrections
    p.w = round_up(int64_t(rows) * row_bytes, 128);  // per expert slot
    p.s = round_up(int64_t(rows) * nb * ssize, 128);
    p.part = decode ? round_up(int64_t(ACT) * rows * 4, 128) : 0;
    p.lg = decode ? round_up(int64_t(kBlockRouteMaxE) * 4, 128) : 0;
    p.total = 256 + p.a4 + p.asum + int64_t(ACT) * (p.w + p.s) + p.part + p.lg;
    return p;
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// One warp routes a token with more than kBlockRouteMaxE experts (rare; out of line).
static __device__ __noinline__ void route_wide(const void* row, int ldt, int E, int k, int normalize, int* s_idx,
                                              float* s_w, const void* agg, int adt) {
    warp_route_pl<kMaxExpertsPerLane>(row, ldt, E, k, normalize, s_idx, s_w, 1, agg, adt);
}

// Router row and aggregation-weight row of token t.
__device__ __forceinline__ const void* logits_row(const QmoeArgs& q, int64_t t) {
    return static_cast<const char*>(q.logits) + t * q.E * (q.logits_dtype == kF32 ? 4 : 2);
}
__device__ __forceinline__ const void* agg_row(const QmoeArgs& q, int64_t t) {
    return q.agg ? static_cast<const char*>(q.agg) + t * q.E * (q.agg_dtype == kF32 ? 4 : 2) : nullptr;
}

// Decode kernels route their own token: the whole CTA ranks up to
// kBlockRouteMaxE logits at once, larger routers fall back to one warp.
// Ends with a block barrier; s_logit holds kBlockRouteMaxE floats.
__device__ __forceinline__ void route_token(const QmoeArgs& q, int64_t t, int* s_idx, float* s_w, float* s_logit) {
    const void* row = logits_row(q, t);
    if (q.E <= kBlockRouteMaxE && q.E <= kThreads) {
        block_route(row, q.logits_dtype, static_cast<int>(q.E), q.k, q.normalize, s_idx, s_w, s_logit, agg_row(q, t),
                    q.agg_dtype);
    } else {
        if (threadIdx.x < 32)
            route_wide(row, q.logits_dtype, static_cast<int>(q.E), q.k, q.normalize, s_idx, s_w, agg_row(q, t),
                       q.agg_dtype);
        __syncthreads();
    }
}

// Bias entry i of a bias tensor in the activation dtype (0 without a bias).
__device__ __forceinline__ float bias_at(const void* bias, int dt, int64_t i) {
    return bias ? load_as_f32(bias, dt, i) : 0.f;
}

// ------------------------------------------------------------------ FC1

// FC1 + SwiGLU for one (activation group, expert) x block of kPairsPerBlock
// gate/up pairs.  DECODE: blockIdx.x is the slot p = t*k + j and the CTA
// routes token t itself; h row = p.  Tiled: blockIdx.x is a tile of <= MT
// sorted pairs of one expert; h rows = sorted positions.
template <int BITS, int ST, int MT, bool DECODE>
__global__ void __launch_bounds__(kThreads) fc1_kernel(const __grid_constant__ QmoeArgs q) {
    using S = typename DType<ST>::T;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int C = static_cast<int>(q.fc1.nb * q.bs / 32);
    const int nb = static_cast<int>(q.fc1.nb);
    const int64_t rb = q.fc1.row_bytes;
    const Fc1Plan plan = fc1_plan(MT, C, rb, nb, sizeof(S));
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    int* s_int = reinterpret_cast<int*>(smem + 16);          // [0]=expert [1]=s0 [2]=cnt, [4..4+MT) rows
    float* s_w = reinterpret_cast<float*>(smem + 128);      // routing weights (decode)
    int* s_idx = reinterpret_cast<int*>(smem + 192);        // routing experts (decode)
    float4* A4 = reinterpret_cast<float4*>(smem + 256);
    float4* Corr = reinterpret_cast<float4*>(smem + 256 + plan.a4);
    uint8_t* Wst = smem + 256 + plan.a4 + plan.asum;
    const S* Sst = reinterpret_cast<const S*>(Wst + plan.w);

    char* ws = static_cast<char*>(q.workspace);
    const Ws L = ws_layout(q.T, q.H, q.I, q.E, q.k);
    float* h = reinterpret_cast<float*>(ws + L.h);
    const int64_t P = q.T * q.k;

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
    }
    const int64_t I = q.I;
    const int64_t pair0 = int64_t(blockIdx.y) * kPairsPerBlock;
    const int pc = static_cast<int>(std::min<int64_t>(kPairsPerBlock, I - pair0));
    const bool inter = q.fc1_layout == MNB_FC1_INTERLEAVED;
    // The block of gate/up rows of expert e (and their scales) into shared memory.
    auto copy_rows = [&](int e) {
        const uint8_t* W1 = q.fc1_w + int64_t(e) * 2 * I * rb;
        const S* S1 = static_cast<const S*>(q.fc1_s) + int64_t(e) * 2 * I * nb;
        const uint32_t wrow = static_cast<uint32_t>(rb), srow = static_cast<uint32_t>(nb * sizeof(S));
        const uint32_t total = 2u * pc * (wrow + srow);
        mbar_arrive_expect_tx(bar, total);
        uint8_t* Sdst = Wst + plan.w;
        if (inter) {
            bulk_g2s(Wst, W1 + 2 * pair0 * rb, 2 * pc * wrow, bar);
            bulk_g2s(Sdst, S1 + 2 * pair0 * nb, 2 * pc * srow, bar);
        } else {
            bulk_g2s(Wst, W1 + pair0 * rb, pc * wrow, bar);
            bulk_g2s(Wst + kPairsPerBlock * rb, W1 + (I + pair0) * rb, pc * wrow, bar);
            bulk_g2s(Sdst, S1 + pair0 * nb, pc * srow, bar);
            bulk_g2s(Sdst + kPairsPerBlock * nb * sizeof(S), S1 + (I + pair0) * nb, pc * srow, bar);
        }
    };
    if (DECODE) {
        // The first kernel of the layer reads no input before its dependency
        // wait (the kernel ahead may still be writing the router logits or the
        // weights); it releases the FC2 kernel right after, so FC2 may read
        // the layer's inputs in its own prologue.
        grid_dependency_wait();
        grid_launch_dependents();
        const int64_t p = blockIdx.x;
        const int64_t t = p / q.k;
        route_token(q, t, s_idx, s_w, reinterpret_cast<float*>(Wst + plan.w + plan.s));
        if (tid == 0) {
            s_int[0] = s_idx[p % q.k];
            s_int[1] = static_cast<int>(p);
            s_int[2] = 1;
            s_int[4] = static_cast<int>(t);
            copy_rows(s_int[0]);
        }
    } else {
        grid_dependency_wait();
        grid_launch_dependents();
        const int tile = blockIdx.x;
        const int ntiles = *reinterpret_cast<const int*>(ws + L.ntiles);
        if (tile >= ntiles) return;
        if (tid == 0) {
            const int2 ti = reinterpret_cast<const int2*>(ws + L.tiles)[tile];
            const int* offsets = reinterpret_cast<const int*>(ws + L.offsets);
            const int* perm = reinterpret_cast<const int*>(ws + L.perm);
            const int cnt = min(MT, offsets[ti.x + 1] - ti.y);
            s_int[0] = ti.x;
            s_int[1] = ti.y;
            s_int[2] = cnt;
            for (int m = 0; m < MT; ++m) s_int[4 + m] = m < cnt ? perm[ti.y + m] / q.k : -1;
            copy_rows(ti.x);
        }
    }
    __syncthreads();
    const int e = s_int[0], s0 = s_int[1], cnt = s_int[2];
    stage_chunks<BITS, MT, ST>(
        A4, Corr, C, q.H, q.act_dtype, q.x_vec != 0,
        [&](int m) -> const void* {
            const int t = m < cnt ? s_int[4 + m] : -1;
            return t >= 0 ? static_cast<const char*>(q.X) + int64_t(t) * q.H * 2 : nullptr;
        },
        tid, kThreads);
    __syncthreads();
    const bool ok = mbar_wait(bar, 0);
    if (__syncthreads_or(!ok)) {
        mbar_wait(bar, 0);
        return;
    }
    const int bs_shift = __ffs(q.bs) - 1;
    constexpr int kZImplicit = 1 << (BITS - 1);
    const uint8_t* Z1 = q.fc1_zp ? q.fc1_zp + int64_t(e) * 2 * I * q.fc1.zp_row : nullptr;

    // Warp unit: pairs 2g and 2g+1 -> logical rows (gate 2g, up 2g, gate 2g+1, up 2g+1).
    for (int g = warp; 2 * g < pc; g += kWarps) {
        float2 out2[R][MT];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) out2[r][m] = make_float2(0.f, 0.f);
        int lrow[R];      // row inside the staged block
        int64_t grow[R];  // row inside the expert's FC1 weight
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int pq = min(2 * g + (r >> 1), pc - 1);
            const int up = r & 1;
            lrow[r] = inter ? 2 * pq + up : up * kPairsPerBlock + pq;
            grow[r] = inter ? 2 * (pair0 + pq) + up : up * I + pair0 + pq;
        }
        for (int c = lane; c < C; c += 32) {
            const int b = (c * 32) >> bs_shift;
            uint32_t w[R][BITS];
            float sc[R], zz[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                load_chunk<BITS>(Wst + int64_t(lrow[r]) * rb, c, w[r]);
                sc[r] = to_f32(Sst[lrow[r] * nb + b]);
                zz[r] = Z1 ? float(kZImplicit - zero_point_code<BITS>(Z1 + grow[r] * q.fc1.zp_row, b)) : 0.f;
            }
            chunk_accumulate<BITS, R, MT>(w, sc, zz, A4 + a4_base(0, c, C), a4_groups(C) * 256, Corr + c, C, out2);
        }
        float out[R][MT];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) out[r][m] = warp_sum(out2[r][m].x + out2[r][m].y);
        if (lane == 0) {
#pragma unroll
            for (int pp = 0; pp < 2; ++pp) {
                const int pq = 2 * g + pp;
                if (pq >= pc) break;
                const int64_t pa = pair0 + pq;  // bias rows of the gate and up halves of pair pa
                const float bg = bias_at(q.fc1_bias, q.act_dtype, int64_t(e) * 2 * I + (inter ? 2 * pa : pa));
                const float bu = bias_at(q.fc1_bias, q.act_dtype, int64_t(e) * 2 * I + (inter ? 2 * pa + 1 : I + pa));
#pragma unroll
                for (int m = 0; m < MT; ++m)
                    if (m < cnt)
                        h[int64_t(s0 + m) * I + pair0 + pq] = silu_mul(out[2 * pp][m] + bg, out[2 * pp + 1][m] + bu);
            }
        }
    }
    (void)P;
}

// ------------------------------------------------------- FC2 (decode)

// FC2 + combine for token t = blockIdx.x over rows [n0, n0 + kDecodeRows2) of
// H: the block's rows of all k selected experts are staged, every warp takes
// (slot, row group) tasks, and the k per-slot results of a row are combined
// with the routing weights in slot order.
template <int BITS, int ST>
__global__ void __launch_bounds__(kThreads) fc2_decode_kernel(const __grid_constant__ QmoeArgs q) {
    using S = typename DType<ST>::T;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int k = q.k;
    const int C = static_cast<int>(q.fc2.nb * q.bs / 32);
    const int nb = static_cast<int>(q.fc2.nb);
    const int64_t rb = q.fc2.row_bytes;
    const Fc2Plan plan = fc2_plan(kDecodeRows2, kDecodeMaxK, C, rb, nb, sizeof(S), true);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    float* s_w = reinterpret_cast<float*>(smem + 128);
    int* s_idx = reinterpret_cast<int*>(smem + 192);
    float4* A4 = reinterpret_cast<float4*>(smem + 256);
    float4* Corr = reinterpret_cast<float4*>(smem + 256 + plan.a4);
    uint8_t* Wst = smem + 256 + plan.a4 + plan.asum;
    uint8_t* Sst = Wst + int64_t(kDecodeMaxK) * plan.w;
    float* part = reinterpret_cast<float*>(Sst + int64_t(kDecodeMaxK) * plan.s);  // [slot][row]
    float* s_logit = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(part) + plan.part);

    const int64_t t = blockIdx.x;
    const int64_t H = q.H, I = q.I;
    const int64_t n0 = int64_t(blockIdx.y) * kDecodeRows2;
    const int rc = static_cast<int>(std::min<int64_t>(kDecodeRows2, H - n0));
    const Ws L = ws_layout(q.T, q.H, q.I, q.E, q.k);
    const float* h = reinterpret_cast<const float*>(static_cast<const char*>(q.workspace) + L.h);

    // Prologue, overlapping the FC1 kernel: FC1 releases this launch only
    // after its own dependency wait, when every kernel ahead of the layer has
    // completed, so the router logits and the weights are final here; this
    // CTA routes its token and starts copying the selected experts' rows
    // before waiting for h.
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
    }
    route_token(q, t, s_idx, s_w, s_logit);
    const uint32_t wbytes = static_cast<uint32_t>(rc * rb), sbytes = static_cast<uint32_t>(rc * nb * sizeof(S));
    if (tid == 0) {
        mbar_arrive_expect_tx(bar, k * (wbytes + sbytes));
        for (int j = 0; j < k; ++j) {
            const int e = s_idx[j];
            bulk_g2s(Wst + j * plan.w, q.fc2_w + (int64_t(e) * H + n0) * rb, wbytes, bar);
            bulk_g2s(Sst + j * plan.s, static_cast<const S*>(q.fc2_s) + (int64_t(e) * H + n0) * nb, sbytes, bar);
        }
    }
    grid_dependency_wait();
    grid_launch_dependents();
    stage_chunks<BITS, kDecodeMaxK, kF32>(
        A4, Corr, C, I, kF32, true,
        [&](int j) -> const void* { return j < k ? static_cast<const void*>(h + (t * k + j) * I) : nullptr; }, tid,
        kThreads);
    __syncthreads();
    const bool ok = mbar_wait(bar, 0);
    if (__syncthreads_or(!ok)) {
        mbar_wait(bar, 0);
        return;
    }
    const int bs_shift = __ffs(q.bs) - 1;
    constexpr int kZImplicit = 1 << (BITS - 1);

    const int groups = (rc + R - 1) / R;
    for (int task = warp; task < k * groups; task += kWarps) {
        const int j = task / groups, g = task - j * groups;
        const int e = s_idx[j];
        const uint8_t* W = Wst + j * plan.w;
        const S* Sc = reinterpret_cast<const S*>(Sst + j * plan.s);
        const uint8_t* Z2 = q.fc2_zp ? q.fc2_zp + int64_t(e) * H * q.fc2.zp_row : nullptr;
        float2 out[R][1];
#pragma unroll
        for (int r = 0; r < R; ++r) out[r][0] = make_float2(0.f, 0.f);
        for (int c = lane; c < C; c += 32) {
            const int b = (c * 32) >> bs_shift;
            uint32_t w[R][BITS];
            float sc[R], zz[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int rl = min(g * R + r, rc - 1);
                load_chunk<BITS>(W + int64_t(rl) * rb, c, w[r]);
                sc[r] = to_f32(Sc[rl * nb + b]);
                zz[r] = Z2 ? float(kZImplicit - zero_point_code<BITS>(Z2 + (n0 + rl) * q.fc2.zp_row, b)) : 0.f;
            }
            chunk_accumulate<BITS, R, 1>(w, sc, zz, A4 + a4_base(j, c, C), a4_groups(C) * 256, Corr + j * C + c, C, out);
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float v = warp_sum(out[r][0].x + out[r][0].y);
            if (lane == 0 && g * R + r < rc)
                part[j * kDecodeRows2 + g * R + r] = v + bias_at(q.fc2_bias, q.act_dtype, e * H + n0 + g * R + r);
        }
    }
    __syncthreads();
    if (tid < rc) {
        float acc = 0.f;
        for (int j = 0; j < k; ++j) acc = fmaf(s_w[j], part[j * kDecodeRows2 + tid], acc);
        store_from_f32(q.Y, q.act_dtype, t * H + n0 + tid, acc);
    }
}

// ------------------------------------------------------- FC2 (tiled)

template <int BITS, int ST, int MT>
__global__ void __launch_bounds__(kThreads) fc2_tile_kernel(const __grid_constant__ QmoeArgs q) {
    using S = typename DType<ST>::T;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int C = static_cast<int>(q.fc2.nb * q.bs / 32);
    const int nb = static_cast<int>(q.fc2.nb);
    const int64_t rb = q.fc2.row_bytes;
    const Fc2Plan plan = fc2_plan(kRowsPerBlock2, MT, C, rb, nb, sizeof(S), false);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    int* s_int = reinterpret_cast<int*>(smem + 16);
    float4* A4 = reinterpret_cast<float4*>(smem + 256);
    float4* Corr = reinterpret_cast<float4*>(smem + 256 + plan.a4);
    uint8_t* Wst = smem + 256 + plan.a4 + plan.asum;
    const S* Sc = reinterpret_cast<const S*>(Wst + plan.w);

    char* ws = static_cast<char*>(q.workspace);
    const Ws L = ws_layout(q.T, q.H, q.I, q.E, q.k);
    const float* h = reinterpret_cast<const float*>(ws + L.h);
    float* o = reinterpret_cast<float*>(ws + L.o);
    const int64_t H = q.H, I = q.I;

    grid_dependency_wait();
    const int tile = blockIdx.x;
    if (tile >= *reinterpret_cast<const int*>(ws + L.ntiles)) return;
    if (tid == 0) {
        const int2 ti = reinterpret_cast<const int2*>(ws + L.tiles)[tile];
        s_int[0] = ti.x;
        s_int[1] = ti.y;
        s_int[2] = min(MT, reinterpret_cast<const int*>(ws + L.offsets)[ti.x + 1] - ti.y);
        mbar_init(bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    const int e = s_int[0], s0 = s_int[1], cnt = s_int[2];
    const int64_t n0 = int64_t(blockIdx.y) * kRowsPerBlock2;
    const int rc = static_cast<int>(std::min<int64_t>(kRowsPerBlock2, H - n0));
    if (tid == 0) {
        const uint32_t wbytes = static_cast<uint32_t>(rc * rb), sbytes = static_cast<uint32_t>(rc * nb * sizeof(S));
        mbar_arrive_expect_tx(bar, wbytes + sbytes);
        bulk_g2s(Wst, q.fc2_w + (int64_t(e) * H + n0) * rb, wbytes, bar);
        bulk_g2s(Wst + plan.w, static_cast<const S*>(q.fc2_s) + (int64_t(e) * H + n0) * nb, sbytes, bar);
    }
    stage_chunks<BITS, MT, kF32>(
        A4, Corr, C, I, kF32, true,
        [&](int m) -> const void* { return m < cnt ? static_cast<const void*>(h + (s0 + m) * I) : nullptr; }, tid,
        kThreads);
    __syncthreads();
    grid_launch_dependents();
    const bool ok = mbar_wait(bar, 0);
    if (__syncthreads_or(!ok)) {
        mbar_wait(bar, 0);
        return;
    }
    const int bs_shift = __ffs(q.bs) - 1;
    constexpr int kZImplicit = 1 << (BITS - 1);
    const uint8_t* Z2 = q.fc2_zp ? q.fc2_zp + int64_t(e) * H * q.fc2.zp_row : nullptr;
    for (int g = warp; g * R < rc; g += kWarps) {
        float2 out2[R][MT];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) out2[r][m] = make_float2(0.f, 0.f);
        for (int c = lane; c < C; c += 32) {
            const int b = (c * 32) >> bs_shift;
            uint32_t w[R][BITS];
            float sc[R], zz[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int rl = min(g * R + r, rc - 1);
                load_chunk<BITS>(Wst + int64_t(rl) * rb, c, w[r]);
                sc[r] = to_f32(Sc[rl * nb + b]);
                zz[r] = Z2 ? float(kZImplicit - zero_point_code<BITS>(Z2 + (n0 + rl) * q.fc2.zp_row, b)) : 0.f;
            }
            chunk_accumulate<BITS, R, MT>(w, sc, zz, A4 + a4_base(0, c, C), a4_groups(C) * 256, Corr + c, C, out2);
        }
        float out[R][MT];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) out[r][m] = warp_sum(out2[r][m].x + out2[r][m].y);
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int rl = g * R + r;
                if (rl >= rc) break;
                const float b2 = bias_at(q.fc2_bias, q.act_dtype, int64_t(e) * H + n0 + rl);
#pragma unroll
                for (int m = 0; m < MT; ++m)
                    if (m < cnt) o[int64_t(s0 + m) * H + n0 + rl] = out[r][m] + b2;
            }
        }
    }
}

// ------------------------------------------------------ tiles, combine

// Tiles of <= kTileM consecutive sorted pairs of one expert.  One thread per
// expert (E <= 1024): tile counts, an exclusive scan, then each expert writes
// its tiles (expert, first sorted position).
__global__ void __launch_bounds__(1024) tiles_kernel(char* ws, int64_t T, int64_t H, int64_t I, int64_t E, int k) {
    const Ws L = ws_layout(T, H, I, E, k);
    const int* counts = reinterpret_cast<const int*>(ws + L.counts);
    const int* offsets = reinterpret_cast<const int*>(ws + L.offsets);
    int2* tiles = reinterpret_cast<int2*>(ws + L.tiles);
    __shared__ int scan[1024];
    grid_dependency_wait();
    const int e = threadIdx.x;
    const int n = e < E ? (counts[e] + kTileM - 1) / kTileM : 0;
    scan[e] = n;
    __syncthreads();
    for (int o = 1; o < 1024; o <<= 1) {
        const int v = e >= o ? scan[e - o] : 0;
        __syncthreads();
        scan[e] += v;
        __syncthreads();
    }
    const int first = scan[e] - n;
    for (int i = 0; i < n; ++i) tiles[first + i] = make_int2(e, offsets[e] + i * kTileM);
    if (e == 1023) *reinterpret_cast<int*>(ws + L.ntiles) = scan[1023];
    grid_launch_dependents();
}

// Y[t, n] = sum_j w[t, j] * o[position of (t, j), n], ascending j, fp32 -> act dtype.
__global__ void combine_kernel(const __grid_constant__ QmoeArgs q) {
    const char* ws = static_cast<const char*>(q.workspace);
    const Ws L = ws_layout(q.T, q.H, q.I, q.E, q.k);
    const float* o = reinterpret_cast<const float*>(ws + L.o);
    const float* wts = reinterpret_cast<const float*>(ws + L.wts);
    const int* inv = reinterpret_cast<const int*>(ws + L.inv);
    grid_dependency_wait();
    grid_launch_dependents();
    const int64_t total = q.T * q.H;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t t = i / q.H, n = i - t * q.H;
        float acc = 0.f;
        for (int j = 0; j < q.k; ++j) acc = fmaf(wts[t * q.k + j], o[int64_t(inv[t * q.k + j]) * q.H + n], acc);
        store_from_f32(q.Y, q.act_dtype, i, acc);
    }
}

// m-tiles for the tensor-core plan: {expert, first sorted position, pairs, 0}.
__global__ void __launch_bounds__(1024) mtiles_kernel(char* ws, int64_t T, int64_t H, int64_t I, int64_t E, int k,
                                                      int tile_m) {
    const Ws L = ws_layout(T, H, I, E, k);
    const int* counts = reinterpret_cast<const int*>(ws + L.counts);
    const int* offsets = reinterpret_cast<const int*>(ws + L.offsets);
    int4* tiles = reinterpret_cast<int4*>(ws + L.mtiles);
    __shared__ int scan[1024];
    grid_dependency_wait();
    const int e = threadIdx.x;
    const int cnt = e < E ? counts[e] : 0;
    const int n = (cnt + tile_m - 1) / tile_m;
    scan[e] = n;
    __syncthreads();
    for (int o = 1; o < 1024; o <<= 1) {
        const int v = e >= o ? scan[e - o] : 0;
        __syncthreads();
        scan[e] += v;
        __syncthreads();
    }
    const int first = scan[e] - n;
    for (int i = 0; i < n; ++i)
        tiles[first + i] = make_int4(e, offsets[e] + i * tile_m, min(tile_m, cnt - i * tile_m), 0);
    if (e == 1023) *reinterpret_cast<int*>(ws + L.nmtiles) = scan[1023];
    grid_launch_dependents();
}

// Xs[s, :] = X[perm[s] / k, :]: the routed tokens' rows in expert-sorted
// order (tensor-core plan), 16 bytes per thread step (H % 8 == 0, X rows
// 16-byte aligned), written into the FC2-output region.
template <typename AT>
__global__ void gather_rows_kernel(const __grid_constant__ QmoeArgs q) {
    char* ws = static_cast<char*>(q.workspace);
    const Ws L = ws_layout(q.T, q.H, q.I, q.E, q.k);
    const int* perm = reinterpret_cast<const int*>(ws + L.perm);
    AT* xs = reinterpret_cast<AT*>(ws + L.o);
    grid_dependency_wait();
    grid_launch_dependents();
    const int64_t G = q.H / 8, total = q.T * q.k * G;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t srow = i / G, c = (i - srow * G) * 8;
        const int64_t t = perm[srow] / q.k;
        *reinterpret_cast<uint4*>(xs + srow * q.H + c) =
            *reinterpret_cast<const uint4*>(static_cast<const AT*>(q.X) + t * q.H + c);
    }
}

// Y[t, n] = sum_j w[t, j] * o[position of (t, j), n], ascending j, fp32 -> act
// dtype, from FC2 outputs kept in the activation dtype (tensor-core plan).
// One thread makes 8 consecutive outputs of a token from 16-byte loads of the
// k routed rows (H % 8 == 0; the workspace rows are 16-byte aligned).
template <typename AT>
__device__ __forceinline__ uint32_t pack_pair(float a, float b);
template <>
__device__ __forceinline__ uint32_t pack_pair<__half>(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack_pair<__nv_bfloat16>(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

template <typename AT>
__global__ void combine_sorted_kernel(const __grid_constant__ QmoeArgs q, int y_vec) {
    const char* ws = static_cast<const char*>(q.workspace);
    const Ws L = ws_layout(q.T, q.H, q.I, q.E, q.k);
    const AT* o = reinterpret_cast<const AT*>(ws + L.o);
    const float* wts = reinterpret_cast<const float*>(ws + L.wts);
    const int* inv = reinterpret_cast<const int*>(ws + L.inv);
    grid_dependency_wait();
    grid_launch_dependents();
    const int64_t G = q.H / 8, total = q.T * G;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t t = i / G, n0 = (i - t * G) * 8;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int j = 0; j < q.k; ++j) {
            const float wj = wts[t * q.k + j];
            const uint4 v = *reinterpret_cast<const uint4*>(o + int64_t(inv[t * q.k + j]) * q.H + n0);
            const AT* h = reinterpret_cast<const AT*>(&v);
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[c] = fmaf(wj, to_f32(h[c]), acc[c]);
        }
        if (y_vec) {
            *reinterpret_cast<uint4*>(static_cast<AT*>(q.Y) + t * q.H + n0) =
                make_uint4(pack_pair<AT>(acc[0], acc[1]), pack_pair<AT>(acc[2], acc[3]), pack_pair<AT>(acc[4], acc[5]),
                           pack_pair<AT>(acc[6], acc[7]));
        } else {
#pragma unroll
            for (int c = 0; c < 8; ++c) store_from_f32(q.Y, q.act_dtype, t * q.H + n0 + c, acc[c]);
        }
    }
}

// ------------------------------------------------------------ launching

template <typename Kern>
cudaError_t launch(Kern kern, dim3 grid, int64_t smem, cudaStream_t stream, const QmoeArgs& q, bool pdl) {
    if (smem > 227 * 1024) return cudaErrorNotSupported;
    cudaError_t e = set_kernel_smem(kern, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, q);
}

template <int BITS, int ST, int MT, bool DECODE>
cudaError_t launch_fc1(const QmoeArgs& q, unsigned gx, cudaStream_t stream, bool pdl) {
    const int C = static_cast<int>(q.fc1.nb * q.bs / 32);
    const Fc1Plan p = fc1_plan(MT, C, q.fc1.row_bytes, static_cast<int>(q.fc1.nb), ST == kF32 ? 4 : 2);
    const unsigned gy = static_cast<unsigned>(cdiv<int64_t>(q.I, kPairsPerBlock));
    return launch(fc1_kernel<BITS, ST, MT, DECODE>, dim3(gx, gy, 1), p.total, stream, q, pdl);
}

template <int B1, int B2, int ST>
cudaError_t run_typed(const QmoeArgs& q, int sm_count, bool pdl, cudaStream_t stream) {
    char* ws = static_cast<char*>(q.workspace);
    const Ws L = ws_layout(q.T, q.H, q.I, q.E, q.k);
    const int64_t P = q.T * q.k;
    const int C2 = static_cast<int>(q.fc2.nb * q.bs / 32);
    const unsigned gy2 = static_cast<unsigned>(cdiv<int64_t>(q.H, kRowsPerBlock2));
    cudaError_t e;
    // From kGroupedMinT tokens on the grouped CUDA-core plan beats the two-kernel
    // decode plan (one copy of each touched expert per m-tile rather than per
    // routed pair: 30B-A3B layer, INT3, T = 4: 55 vs 69 us, T = 8: 83 vs 131 us;
    // T = 2: 42 vs 37 us).
    if (use_decode(q) && !(q.T >= kGroupedMinT && use_grouped(q))) {
        // one token: the fused single-pass kernel (qmoe_decode.cu) where its shape rules allow
        if (q.T == 1) {
            e = launch_qmoe_decode_fused(q, sm_count, pdl, stream);
            if (e != cudaErrorNotSupported) return e;
        }
        e = launch_fc1<B1, ST, 1, true>(q, static_cast<unsigned>(P), stream, pdl);
        if (e != cudaSuccess) return e;
        const Fc2Plan p2 = fc2_plan(kDecodeRows2, kDecodeMaxK, C2, q.fc2.row_bytes, static_cast<int>(q.fc2.nb), 2, true);
        const unsigned gyd = static_cast<unsigned>(cdiv<int64_t>(q.H, kDecodeRows2));
        return launch(fc2_decode_kernel<B2, ST>, dim3(static_cast<unsigned>(q.T), gyd, 1), p2.total, stream, q, pdl);
    }
    int32_t* idx = reinterpret_cast<int32_t*>(ws + L.idx);
    float* wts = reinterpret_cast<float*>(ws + L.wts);
    if ((e = launch_route(q.logits, q.logits_dtype, q.T, q.E, q.k, q.normalize, idx, wts, q.agg, q.agg_dtype,
                          stream, pdl)) != cudaSuccess)
        return e;
    // m-tile plans (grouped CUDA-core, tensor-core): tile height kGroupedGemvRows,
    // or from the mean routed rows per expert (FC1 and FC2 alike); up to
    // kOneCtaPlanPairs routed pairs one CTA sorts them and writes the m-tiles in
    // one launch (faster than four launches there)
    const bool grouped = use_grouped(q);
    const bool tc = !grouped && use_tc(q);
    const int tile_m = grouped ? kGroupedGemvRows : tc ? grouped_tile_m(P, q.E) : 0;
    const bool one_cta = (grouped || tc) && P <= kOneCtaPlanPairs && q.E <= 1024;
    if (one_cta) {
        if ((e = launch_permute(idx, q.T, q.k, q.E, reinterpret_cast<int32_t*>(ws + L.counts),
                                reinterpret_cast<int32_t*>(ws + L.offsets), reinterpret_cast<int32_t*>(ws + L.perm),
                                reinterpret_cast<int32_t*>(ws + L.inv), stream, reinterpret_cast<int4*>(ws + L.mtiles),
                                reinterpret_cast<int*>(ws + L.nmtiles), tile_m, pdl)) != cudaSuccess)
            return e;
    } else if ((e = launch_permute_chunked(idx, q.T, q.k, q.E, reinterpret_cast<int32_t*>(ws + L.chunkc),
                                           reinterpret_cast<int32_t*>(ws + L.counts),
                                           reinterpret_cast<int32_t*>(ws + L.offsets),
                                           reinterpret_cast<int32_t*>(ws + L.perm),
                                           reinterpret_cast<int32_t*>(ws + L.inv), stream, pdl)) != cudaSuccess) {
        return e;
    }
    if ((grouped || tc) && !one_cta) {
        if ((e = set_max_carveout(mtiles_kernel)) != cudaSuccess) return e;
        if ((e = launch_ex(mtiles_kernel, dim3(1), dim3(1024), 0, stream, pdl, ws, q.T, q.H, q.I, q.E, q.k, tile_m)) !=
            cudaSuccess)
            return e;
    }
    if (grouped) {
        // FC1 + SwiGLU -> h (fp32, sorted rows), FC2 -> o (fp32, sorted rows), combine
        GemvArgs g1, g2;
        grouped_args(q, g1, g2);
        g1.g_tiles = g2.g_tiles = reinterpret_cast<const int4*>(ws + L.mtiles);
        g1.g_ntiles = g2.g_ntiles = reinterpret_cast<const int*>(ws + L.nmtiles);
        g1.g_perm = reinterpret_cast<const int*>(ws + L.perm);
        g1.Y = ws + L.h;
        g2.A = ws + L.h;
        g2.Y = ws + L.o;
        // expected m-tile count (it sets the CTAs per tile): the P / 4 full tiles
        // plus a partial last tile for about every second touched expert
        const int64_t grid_y = max_mtiles(P, q.E);
        const int64_t est = std::min(grid_y, P / kGroupedGemvRows + std::min(P, q.E) / 2);
        if ((e = launch_gemv_grouped(g1, q.act_dtype, grid_y, est, sm_count, pdl, stream)) != cudaSuccess) return e;
        if ((e = launch_gemv_grouped(g2, q.act_dtype, grid_y, est, sm_count, pdl, stream)) != cudaSuccess) return e;
        const int64_t blocks = std::min<int64_t>(cdiv<int64_t>(q.T * q.H, 256), int64_t(sm_count) * 16);
        if ((e = set_max_carveout(combine_kernel)) != cudaSuccess) return e;
        return launch_ex(combine_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, pdl, q);
    }
    if (tc) {
        TcArgs a = {};
        a.splits = 1;
        a.mtiles = reinterpret_cast<const int4*>(ws + L.mtiles);
        a.n_mtiles = reinterpret_cast<const int*>(ws + L.nmtiles);
        a.bs = q.bs;
        a.y_dtype = q.act_dtype;
        a.experts = q.E;
        // FC1: K = H, 2I rows (pair-interleaved in the tile), SwiGLU into h (act dtype, sorted order)
        a.M = P;
        a.K = q.H;
        a.rows = 2 * q.I;
        a.B = q.fc1_w;
        a.scales = q.fc1_s;
        a.zp = q.fc1_zp;
        a.row_bytes = q.fc1.row_bytes;
        a.nb = static_cast<int>(q.fc1.nb);
        a.zp_row_bytes = static_cast<int>(q.fc1.zp_row);
        a.w_expert_stride = 2 * q.I * q.fc1.row_bytes;
        a.s_expert_stride = 2 * q.I * q.fc1.nb * 2;
        a.z_expert_stride = 2 * q.I * q.fc1.zp_row;
        a.Y = ws + L.h;
        a.ld_y = q.I;
        a.tiles_n = static_cast<int>(cdiv<int64_t>(2 * q.I, 128));
        a.k_steps = static_cast<int>(cdiv<int64_t>(q.H, 64));
        a.perm = reinterpret_cast<const int*>(ws + L.perm);
        a.k = q.k;
        a.I = q.I;
        a.inter = q.fc1_layout == MNB_FC1_INTERLEAVED;
        a.X = q.X;
        a.bias = q.fc1_bias;
        // The routed tokens' rows in expert-sorted order go into the FC2-output
        // region (free until FC2 runs), so FC1 loads them as plain TMA tiles.
        {
            using AT = typename DType<ST>::T;
            const int64_t blocks = std::min<int64_t>(cdiv<int64_t>(P * (q.H / 8), 256), int64_t(sm_count) * 16);
            if ((e = set_max_carveout(gather_rows_kernel<AT>)) != cudaSuccess) return e;
            if ((e = launch_ex(gather_rows_kernel<AT>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, pdl,
                               q)) != cudaSuccess)
                return e;
        }
        if ((e = launch_grouped_tc(true, a, B1, ST, ST, ws + L.o, P, q.H, tile_m, sm_count, pdl, stream)) != cudaSuccess)
            return e;
        // FC2: K = I, H rows; activations are h rows in sorted order (TMA), output o (act dtype, sorted order)
        a.K = q.I;
        a.rows = q.H;
        a.B = q.fc2_w;
        a.scales = q.fc2_s;
        a.zp = q.fc2_zp;
        a.row_bytes = q.fc2.row_bytes;
        a.nb = static_cast<int>(q.fc2.nb);
        a.zp_row_bytes = static_cast<int>(q.fc2.zp_row);
        a.w_expert_stride = q.H * q.fc2.row_bytes;
        a.s_expert_stride = q.H * q.fc2.nb * 2;
        a.z_expert_stride = q.H * q.fc2.zp_row;
        a.Y = ws + L.o;
        a.ld_y = q.H;
        a.bias = q.fc2_bias;
        a.tiles_n = static_cast<int>(cdiv<int64_t>(q.H, 128));
        a.k_steps = static_cast<int>(cdiv<int64_t>(q.I, 64));
        if ((e = launch_grouped_tc(false, a, B2, ST, ST, ws + L.h, P, q.I, tile_m, sm_count, pdl, stream)) != cudaSuccess)
            return e;
        const int64_t blocks = std::min<int64_t>(cdiv<int64_t>(q.T * q.H / 8, 256), int64_t(sm_count) * 16);
        using AT = typename DType<ST>::T;
        const int y_vec = (reinterpret_cast<uintptr_t>(q.Y) & 15) == 0;
        if ((e = set_max_carveout(combine_sorted_kernel<AT>)) != cudaSuccess) return e;
        return launch_ex(combine_sorted_kernel<AT>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, pdl, q,
                         y_vec);
    }
    if ((e = set_max_carveout(tiles_kernel)) != cudaSuccess) return e;
    if ((e = launch_ex(tiles_kernel, dim3(1), dim3(1024), 0, stream, pdl, ws, q.T, q.H, q.I, q.E, q.k)) != cudaSuccess)
        return e;
    const unsigned gx = static_cast<unsigned>(max_tiles(P, q.E));
    if ((e = launch_fc1<B1, ST, kTileM, false>(q, gx, stream, pdl)) != cudaSuccess) return e;
    const Fc2Plan p2 = fc2_plan(kRowsPerBlock2, kTileM, C2, q.fc2.row_bytes, static_cast<int>(q.fc2.nb), 2, false);
    if ((e = launch(fc2_tile_kernel<B2, ST, kTileM>, dim3(gx, gy2, 1), p2.total, stream, q, pdl)) != cudaSuccess) return e;
    const int64_t blocks = std::min<int64_t>(cdiv<int64_t>(q.T * q.H, 256), 152 * 16);
    if ((e = set_max_carveout(combine_kernel)) != cudaSuccess) return e;
    return launch_ex(combine_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, pdl, q);
}

template <int ST>
cudaError_t run_bits(const QmoeArgs& q, int sm_count, bool pdl, cudaStream_t stream) {
    if (q.fc1_bits == 3 && q.fc2_bits == 3) return run_typed<3, 3, ST>(q, sm_count, pdl, stream);
    if (q.fc1_bits == 3 && q.fc2_bits == 4) return run_typed<3, 4, ST>(q, sm_count, pdl, stream);
    if (q.fc1_bits == 4 && q.fc2_bits == 3) return run_typed<4, 3, ST>(q, sm_count, pdl, stream);
    return run_typed<4, 4, ST>(q, sm_count, pdl, stream);
}

}  // namespace

bool qmoe_workspace_bytes(int64_t T, int64_t H, int64_t I, int64_t E, int k, int64_t* bytes) {
    if (T > (int64_t(1) << 24) || H > (int64_t(1) << 24) || I > (int64_t(1) << 24) || k > 1024) return false;
    const int64_t P = T * k;
    if (P >= (int64_t(1) << 31) || P * std::max(H, I) > (int64_t(1) << 40)) return false;
    *bytes = ws_layout(T, H, I, E, k).total;
    return true;
}

cudaError_t qmoe_take_error(unsigned int* out) { return take_unit_error(out); }

void qmoe_ws_decode_regions(int64_t T, int64_t H, int64_t I, int64_t E, int k, int64_t* h_off, int64_t* sync_off) {
    const Ws L = ws_layout(T, H, I, E, k);
    *h_off = L.h;
    *sync_off = L.sync;
}

cudaError_t launch_qmoe(const QmoeArgs& q, int sm_count, bool pdl, cudaStream_t stream) {
    return q.act_dtype == MNB_F16 ? run_bits<kF16>(q, sm_count, pdl, stream) : run_bits<kBF16>(q, sm_count, pdl, stream);
}

}  // namespace mnb
