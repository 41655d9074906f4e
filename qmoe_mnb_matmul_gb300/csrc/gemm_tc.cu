// gemm_tc.cu -- host entry points of the tensor-core GEMM (see gemm_tc_impl.cuh).
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace mnb {

#define MNB_SLICE_DECL(NAME)                                                                                      \
    cudaError_t NAME(int scale_dtype, int a_dtype, int BN, int G, const TcArgs& a, const void* A_rows,          \
                     int64_t a_rows, int64_t a_cols, int grid, bool pdl, cudaStream_t stream);                 \
    cudaError_t NAME##_take_error(unsigned int* out);
MNB_SLICE_DECL(gemm_tc_gemm_b3)
MNB_SLICE_DECL(gemm_tc_gemm_b4)
MNB_SLICE_DECL(gemm_tc_fc1_b3)
MNB_SLICE_DECL(gemm_tc_fc1_b4)
#undef MNB_SLICE_DECL

namespace {

constexpr int kBW = 128;  // weight rows per tile
constexpr int kBK = 64;   // K per stage

// Tile shape: BN activation rows per MMA and G sub-tiles per dequantised
// weight tile.  A tile's time is modelled as max(MMA columns G*BN, the
// dequantisation of its weight K steps, worth ~460 MMA columns per step at the
// measured rates) over the narrow-tile MMA efficiency; the grid walks the
// tiles in waves of one per SM.
struct TcShape {
    int BN, G;
};
TcShape pick_shape(int64_t M, int64_t N, int sm_count) {
    TcShape best{256, 1};
    double best_cost = 1e300;
    const TcShape cands[] = {{256, 1}, {128, 1}, {64, 1}, {32, 1}, {16, 1}};
    for (const TcShape& c : cands) {
        if (c.G == 1 && c.BN > 16 && c.BN / 2 >= M) continue;  // a narrower tile covers M already
        const int64_t tiles = cdiv<int64_t>(N, kBW) * cdiv<int64_t>(M, int64_t(c.BN) * c.G);
        const double waves = double(cdiv<int64_t>(tiles, sm_count));
        const double eff = c.BN >= 256 ? 1.0 : c.BN >= 128 ? 0.9 : c.BN >= 64 ? 0.7 : 0.5;
        const double cost = waves * std::max(double(c.BN * c.G), 460.0) / eff;
        if (cost < best_cost) { best_cost = cost; best = c; }
    }
    return best;
}

// K split: when the output tiles cannot give every SM a tile, the K steps of
// each tile are divided among up to 16 CTAs (an equal share each, at least 4
// steps), their fp32 partial sums go to the workspace, and a second kernel adds
// them in split order.
struct TcPlanK {
    TcShape sh;
    int splits;
};
TcPlanK plan_tc(int64_t M, int64_t K, int64_t N, int sm_count) {
    TcPlanK p{pick_shape(M, N, sm_count), 1};
    const int64_t tiles = cdiv<int64_t>(N, kBW) * cdiv<int64_t>(M, int64_t(p.sh.BN) * p.sh.G);
    const int64_t ksteps = cdiv<int64_t>(K, kBK);
    if (tiles * 2 > sm_count) return p;
    for (int s = 16; s >= 2; --s) {
        if (ksteps % s != 0 || ksteps / s < 4 || tiles * s > int64_t(sm_count) * 5 / 4) continue;
        p.splits = s;
        break;
    }
    return p;
}

// Y[i] = sum over splits s of P[s][i] (in split order), rounded once to Y's
// dtype; with `add` (the remainder pass of an fp32 output) Y[i] += that sum.
__global__ void splitk_reduce_kernel(const float* __restrict__ P, int splits, int64_t MN, void* Y, int y_dtype,
                                     int add) {
    grid_dependency_wait();
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < MN; i += int64_t(gridDim.x) * blockDim.x) {
        float acc = P[i];
        for (int s = 1; s < splits; ++s) acc += P[s * MN + i];
        if (add)
            static_cast<float*>(Y)[i] += acc;
        else
            store_from_f32(Y, y_dtype, i, acc);
    }
}

}  // namespace

size_t gemm_tc_workspace_bytes(int64_t M, int64_t K, int64_t N, int sm_count) {
    const TcPlanK p = plan_tc(M, K, N, sm_count);
    return p.splits > 1 ? size_t(p.splits) * size_t(M) * size_t(N) * sizeof(float) : 0;
}

cudaError_t gemm_tc_take_error(unsigned int* out) {
    unsigned int first = 0;
    for (auto take : {gemm_tc_gemm_b3_take_error, gemm_tc_gemm_b4_take_error, gemm_tc_fc1_b3_take_error,
                      gemm_tc_fc1_b4_take_error}) {
        unsigned int v = 0;
        const cudaError_t e = take(&v);
        if (e != cudaSuccess) return e;
        if (first == 0) first = v;
    }
    *out = first;
    return cudaSuccess;
}

cudaError_t launch_gemm_tc(const GemmTcArgs& g, int scale_dtype, int sm_count, bool pdl, cudaStream_t stream) {
    TcPlanK plan = plan_tc(g.M, g.K, g.N, sm_count);
    const int64_t ksteps = cdiv<int64_t>(g.K, kBK);
    const size_t per_split = size_t(g.M) * size_t(g.N) * sizeof(float);
    // fewer splits when the caller's workspace holds fewer partial sums (none: one CTA per tile)
    while (plan.splits > 1 &&
           (g.workspace == nullptr || g.workspace_bytes < per_split * plan.splits || ksteps % plan.splits != 0))
        --plan.splits;
    const TcShape sh = plan.sh;
    TcArgs a = {};
    a.M = g.M;
    a.K = g.K;
    a.rows = g.N;
    a.B = g.B;
    a.scales = g.scales;
    a.zp = g.zp;
    a.row_bytes = g.row_bytes;
    a.nb = g.nb;
    a.bs = g.bs;
    a.zp_row_bytes = g.zp_row_bytes;
    a.Y = g.Y;
    a.y_dtype = g.y_dtype;
    a.ld_y = g.N;
    a.tiles_n = static_cast<int>(cdiv<int64_t>(g.N, kBW));
    a.tiles_m = static_cast<int>(cdiv<int64_t>(g.M, int64_t(sh.BN) * sh.G));
    a.splits = plan.splits;
    a.k_steps = static_cast<int>(cdiv<int64_t>(g.K, kBK)) / plan.splits;
    a.partials = plan.splits > 1 ? static_cast<float*>(g.workspace) : nullptr;
    const int grid = static_cast<int>(std::min<int64_t>(int64_t(a.tiles_n) * a.tiles_m * a.splits, sm_count));
    auto fn = g.bits == 4 ? gemm_tc_gemm_b4 : gemm_tc_gemm_b3;
    // An fp32 output from 16-bit activations takes two passes: the product with
    // the weights rounded to the activation type, then the product with what
    // that rounding left (the remainder, also 16-bit) added to the output, so
    // the weight reaches ~16 significant bits (two 8- or 11-bit terms).
    const int passes = (g.y_dtype == kF32 && g.a_dtype != kF32) ? 2 : 1;
    for (int pass = 0; pass < passes; ++pass) {
        a.remainder = pass;
        cudaError_t e = fn(scale_dtype, g.a_dtype, sh.BN, sh.G, a, g.A, g.M, g.K, grid, pdl, stream);
        if (e != cudaSuccess) return e;
        if (plan.splits == 1) continue;
        const int64_t MN = g.M * g.N;
        const int64_t blocks = std::min<int64_t>(cdiv<int64_t>(MN, 256), int64_t(sm_count) * 8);
        if ((e = set_max_carveout(splitk_reduce_kernel)) != cudaSuccess) return e;
        if ((e = launch_ex(splitk_reduce_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, pdl,
                           static_cast<const float*>(a.partials), plan.splits, MN, g.Y, g.y_dtype, pass)) != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

// Dense gate/up with SwiGLU on the tensor cores: the FC1 mode of the grouped
// kernel over one "expert" (the whole matrix), plain activation-row tiles.
cudaError_t launch_gate_up_tc(const GemmTcArgs& g, int64_t I, bool inter, int scale_dtype, int sm_count, bool pdl,
                              cudaStream_t stream) {
    TcArgs a = {};
    a.M = g.M;
    a.K = g.K;
    a.rows = 2 * I;
    a.B = g.B;
    a.scales = g.scales;
    a.zp = g.zp;
    a.row_bytes = g.row_bytes;
    a.nb = g.nb;
    a.bs = g.bs;
    a.zp_row_bytes = g.zp_row_bytes;
    a.Y = g.Y;
    a.y_dtype = g.y_dtype;
    a.ld_y = I;
    a.tiles_n = static_cast<int>(cdiv<int64_t>(2 * I, kBW));
    const int bn = grouped_tile_m(g.M, 1);
    a.tiles_m = static_cast<int>(cdiv<int64_t>(g.M, int64_t(bn)));
    a.splits = 1;
    a.k_steps = static_cast<int>(cdiv<int64_t>(g.K, kBK));
    a.I = I;
    a.inter = inter ? 1 : 0;
    a.experts = 1;
    const int grid = static_cast<int>(std::min<int64_t>(int64_t(a.tiles_n) * a.tiles_m, sm_count));
    auto fn = g.bits == 4 ? gemm_tc_fc1_b4 : gemm_tc_fc1_b3;
    return fn(scale_dtype, g.a_dtype, bn, 1, a, g.A, g.M, g.K, grid, pdl, stream);
}

// Activation rows per grouped tile: the power of two in [32, 256] at or above
// four times the mean rows per matrix.  Every tile dequantises its expert's
// weights again, which costs more than the tensor-core work of a tile, so a
// tile should hold all of an expert's rows (routing is uneven: four times the
// mean); only where even that leaves most of a 256-row tile empty does a
// shorter tile save MMA work.
int grouped_tile_m(int64_t rows, int64_t matrices) {
    const int64_t mean = (rows + matrices - 1) / std::max<int64_t>(matrices, 1);
    int bn = 32;
    while (bn < 256 && bn < 4 * mean) bn <<= 1;
    return bn;
}

cudaError_t launch_grouped_tc(bool fc1, const TcArgs& a, int bits, int scale_dtype, int a_dtype, const void* A_rows,
                              int64_t a_rows, int64_t a_cols, int tile_m, int sm_count, bool pdl, cudaStream_t stream) {
    auto fn = fc1 ? (bits == 4 ? gemm_tc_fc1_b4 : gemm_tc_fc1_b3) : (bits == 4 ? gemm_tc_gemm_b4 : gemm_tc_gemm_b3);
    return fn(scale_dtype, a_dtype, tile_m, 1, a, A_rows, a_rows, a_cols, sm_count, pdl, stream);
}

}  // namespace mnb
