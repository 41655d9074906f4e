// gemm_tc.cu -- host entry points of the tensor-core GEMM (see gemm_tc_impl.cuh).
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace mnb {

#define MNB_SLICE_DECL(NAME)                                                                                      \
    cudaError_t NAME(int scale_dtype, int a_dtype, int BN, const TcArgs& a, const void* A_rows, int64_t a_rows, \
                     int64_t a_cols, int grid, bool pdl, cudaStream_t stream);                                \
    cudaError_t NAME##_take_error(unsigned int* out);
MNB_SLICE_DECL(gemm_tc_gemm_b3)
MNB_SLICE_DECL(gemm_tc_gemm_b4)
MNB_SLICE_DECL(gemm_tc_fc1_b3)
MNB_SLICE_DECL(gemm_tc_fc1_b4)
#undef MNB_SLICE_DECL

namespace {

constexpr int kBW = 128;  // weight rows per tile
constexpr int kBK = 64;   // K per stage

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

}  // namespace

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
    const int BN = pick_bn(g.M, g.N, sm_count);
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
    a.tiles_m = static_cast<int>(cdiv<int64_t>(g.M, BN));
    a.k_steps = static_cast<int>(cdiv<int64_t>(g.K, kBK));
    const int grid = static_cast<int>(std::min<int64_t>(int64_t(a.tiles_n) * a.tiles_m, sm_count));
    auto fn = g.bits == 4 ? gemm_tc_gemm_b4 : gemm_tc_gemm_b3;
    return fn(scale_dtype, g.a_dtype, BN, a, g.A, g.M, g.K, grid, pdl, stream);
}

int grouped_tile_rows() { return 256; }

cudaError_t launch_grouped_tc(bool fc1, const TcArgs& a, int bits, int scale_dtype, int a_dtype, const void* A_rows,
                              int64_t a_rows, int64_t a_cols, int sm_count, bool pdl, cudaStream_t stream) {
    const int BN = grouped_tile_rows();
    auto fn = fc1 ? (bits == 4 ? gemm_tc_fc1_b4 : gemm_tc_fc1_b3) : (bits == 4 ? gemm_tc_gemm_b4 : gemm_tc_gemm_b3);
    return fn(scale_dtype, a_dtype, BN, a, A_rows, a_rows, a_cols, sm_count, pdl, stream);
}

}  // namespace mnb
