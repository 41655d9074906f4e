// gemv_grouped.cu -- the QMoE expert projections on CUDA cores for layers with
// few routed rows per expert ("INT3 QMoE CUDA correctness baseline and Qwen
// experimental results", "P1: Compatible QMoE v1 Extension": the selected
// experts' packed weights are dequantised while they are consumed).
//
// With a handful of routed rows per expert the tensor-core plan spends its time
// dequantising every expert's weight tile once per K step for a few activation
// columns; here each CTA streams one expert's packed rows through the GEMV ring
// and takes exact dp4a chunk products against the fixed-point images of up to
// four routed rows (one m-tile), so the cost per weight code is a few integer
// instructions per row.  Kernel: gemv_grouped_kernel (gemv_impl.cuh).
#include "gemv_impl.cuh"

namespace mnb {

namespace {

constexpr int kGroupedR = 2;  // weight rows per pass with four activation rows (registers)
constexpr int kGroupedRows = 4;  // rows per warp of a block (short m-tiles take them in one pass)
constexpr int64_t kGroupedCtaSmem = 112 * 1024;  // two CTAs per SM

struct GroupedShape {
    int RC = 0, stages = 0;
    int64_t smem = 0;
};

GroupedShape grouped_shape(const GemvArgs& a, int ssize) {
    GroupedShape g;
    const int64_t align = row_align(a.row_bytes, a.nb, ssize);
    const int RC = static_cast<int>(std::max<int64_t>(kConsumerWarps * kGroupedRows, a.swiglu ? 2 * align : align));
    const Plan p1 = make_plan(kGroupedGemvRows, a.chunks, RC, a.row_bytes, a.nb, ssize, 1);
    const int64_t stage = p1.w_stage + p1.s_stage;
    const int64_t st = std::min<int64_t>(kMaxStages, (kGroupedCtaSmem - p1.fixed) / stage);
    if (st < 2) return g;
    g.RC = RC;
    g.stages = static_cast<int>(st);
    g.smem = make_plan(kGroupedGemvRows, a.chunks, RC, a.row_bytes, a.nb, ssize, g.stages).total;
    return g;
}

template <int BITS, int ST>
cudaError_t launch_grouped_typed(GemvArgs a, int64_t grid_y, int64_t est_tiles, int sm_count, bool pdl,
                                 cudaStream_t stream) {
    const GroupedShape g = grouped_shape(a, ST == kF32 ? 4 : 2);
    if (g.stages == 0 || grid_y < 1 || grid_y > 65535) return cudaErrorNotSupported;
    a.rows_per_block = g.RC;
    a.n_blocks = static_cast<int>(cdiv<int64_t>(a.N, g.RC));
    a.stages = g.stages;
    a.prefetch_all = 0;
    // CTAs per m-tile: about two CTAs per SM over the expected tiles
    const int64_t want = (2 * int64_t(sm_count) + std::max<int64_t>(est_tiles, 1) / 2) / std::max<int64_t>(est_tiles, 1);
    const int64_t gx = std::max<int64_t>(1, std::min<int64_t>(want, a.n_blocks));
    auto kern = gemv_grouped_kernel<BITS, ST, kGroupedGemvRows, kGroupedR>;
    cudaError_t e = set_kernel_smem(kern, g.smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(gx), static_cast<unsigned>(grid_y), 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(g.smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

bool gemv_grouped_fits(const GemvArgs& a, int scale_dtype) {
    return (a.bits == 3 || a.bits == 4) && scale_dtype != kF32 && grouped_shape(a, 2).stages > 0;
}

cudaError_t launch_gemv_grouped(const GemvArgs& a, int scale_dtype, int64_t grid_y, int64_t est_tiles, int sm_count,
                                bool pdl, cudaStream_t stream) {
    if (!gemv_grouped_fits(a, scale_dtype)) return cudaErrorNotSupported;
    if (a.bits == 4)
        return scale_dtype == kF16 ? launch_grouped_typed<4, kF16>(a, grid_y, est_tiles, sm_count, pdl, stream)
                                   : launch_grouped_typed<4, kBF16>(a, grid_y, est_tiles, sm_count, pdl, stream);
    return scale_dtype == kF16 ? launch_grouped_typed<3, kF16>(a, grid_y, est_tiles, sm_count, pdl, stream)
                               : launch_grouped_typed<3, kBF16>(a, grid_y, est_tiles, sm_count, pdl, stream);
}

}  // namespace mnb
