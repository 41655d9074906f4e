// qmoe_decode.cu -- one QMoE layer for one token in a single pass over the
// selected experts' weights ("INT3 QMoE CUDA correctness baseline and Qwen
// experimental results", Summary: routing, fused gate/up FC1 with SwiGLU,
// the down projection FC2 and the weighted combine; no expert matrix is ever
// dequantised into global memory).
//
// Two launches:
//  * qmoe_decode_prep_kernel (one CTA) waits for the work ahead of the layer,
//    releases the layer kernel and zeroes the grid barrier counter in the
//    workspace.
//  * qmoe_decode_fused_kernel, at most one CTA per SM, all resident at once.  Its prologue runs
//    while the prep kernel finishes: the prep kernel released it only after
//    its own dependency wait, so the router logits and the expert weights are
//    final.  Every CTA routes the token, then issues in one go the bulk copies
//    of its slice of the k experts' FC1 gate/up pairs and of its slice of
//    their FC2 rows (all weight traffic of the layer is in flight at once).
//    After its dependency wait it stages the token's activations, computes
//    h = silu(gate) * up for its pairs and publishes h, meets every other CTA
//    at a grid barrier (a counter with a bounded wait that records
//    MNB_ERR_TIMEOUT), stages all k rows of h, computes FC2 for its output
//    rows from the rows already in shared memory, and combines the k slots in
//    slot order.
// Dot products use the exact dp4a chunk products of gemv_int.cuh.
#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "gemv_core.cuh"
#include "gemv_int.cuh"
#include "qmoe.h"
#include "route_core.cuh"

namespace mnb {

namespace {

using namespace gemv_int;

constexpr int kWarps = 16;  // alone on its SM: 16 warps to hide the instruction latencies
constexpr int kThreads = kWarps * 32;
constexpr int kMaxK = 8;
constexpr int kMaxPairs = 48;      // FC1 gate/up pairs per CTA
constexpr int kMaxRows2 = 16;      // FC2 output rows per CTA
constexpr int64_t kSmemCap = 227 * 1024;

__host__ __device__ inline int64_t r128(int64_t x) { return (x + 127) / 128 * 128; }

struct DecPlan {
    int64_t ximg, xcorr, himg, hcorr, w1, s1, w2, s2, part, total;
};

__host__ __device__ inline DecPlan dec_plan(int C1, int C2, int k, int64_t rb1, int nb1, int64_t rb2, int nb2,
                                            int ssize) {
    DecPlan p;
    int64_t off = 2048;  // barriers, routing, router logits
    p.ximg = off; off += qimg_bytes(1, C1);
    p.xcorr = off; off += corr_bytes(1, C1);
    p.himg = off; off += qimg_bytes(k, C2);
    p.hcorr = off; off += corr_bytes(k, C2);
    p.w1 = off; off += r128(2 * kMaxPairs * rb1);
    p.s1 = off; off += r128(2 * kMaxPairs * nb1 * ssize);
    p.w2 = off; off += r128(int64_t(k) * kMaxRows2 * rb2);
    p.s2 = off; off += r128(int64_t(k) * kMaxRows2 * nb2 * ssize);
    p.part = off; off += r128(int64_t(kMaxK) * kMaxRows2 * 4);
    p.total = off;
    return p;
}

// Items [first, last) of CTA x among g CTAs, in units of u items: contiguous,
// unit counts differing by at most one.
__host__ __device__ inline void split(int64_t n, int64_t u, int x, int g, int64_t& first, int64_t& last) {
    const int64_t units = n / u, q = units / g, r = units - q * g;
    first = (x * q + (x < r ? x : r)) * u;
    last = first + (q + (x < r ? 1 : 0)) * u;
}

// The smallest count of rows (FC2) or gate/up pairs (FC1, two rows each)
// whose packed bytes and 16-bit scales are whole 16-byte units, so that every
// CTA's bulk copies start and end on 16-byte boundaries.
__host__ __device__ inline int64_t copy_unit(int64_t row_bytes, int64_t scale_bytes, int rows_per_item) {
    int64_t u = 1;
    while ((u * rows_per_item * row_bytes) % 16 || (u * rows_per_item * scale_bytes) % 16) u *= 2;
    return u;
}

__global__ void qmoe_decode_prep_kernel(unsigned int* counter) {
    grid_dependency_wait();
    grid_launch_dependents();
    if (threadIdx.x == 0) *counter = 0u;
}

__device__ __forceinline__ unsigned int load_acquire(const unsigned int* p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// Reduces the R sums of each lane over the warp; lane 0 ends with them in v[0..R).
template <int R>
__device__ __forceinline__ void warp_sums(float (&v)[R]) {
#pragma unroll
    for (int r = 0; r < R; ++r) v[r] = warp_sum(v[r]);
}

template <int B1, int B2, int ST>
__global__ void __launch_bounds__(kThreads, 1) qmoe_decode_fused_kernel(const __grid_constant__ QmoeArgs q,
                                                                       int64_t h_off, int64_t sync_off) {
    using S = typename DType<ST>::T;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int k = q.k;
    const int64_t H = q.H, I = q.I;
    const int C1 = static_cast<int>(q.fc1.nb * q.bs / 32), C2 = static_cast<int>(q.fc2.nb * q.bs / 32);
    const int nb1 = static_cast<int>(q.fc1.nb), nb2 = static_cast<int>(q.fc2.nb);
    const int64_t rb1 = q.fc1.row_bytes, rb2 = q.fc2.row_bytes;
    const DecPlan plan = dec_plan(C1, C2, k, rb1, nb1, rb2, nb2, sizeof(S));
    uint64_t* bar1 = reinterpret_cast<uint64_t*>(smem);
    uint64_t* bar2 = bar1 + 1;
    volatile int* s_fail = reinterpret_cast<volatile int*>(smem + 16);
    int* s_idx = reinterpret_cast<int*>(smem + 64);
    float* s_w = reinterpret_cast<float*>(smem + 128);
    float* s_logit = reinterpret_cast<float*>(smem + 1024);  // kBlockRouteMaxE floats
    uint4* Xq = reinterpret_cast<uint4*>(smem + plan.ximg);
    int2* Xc = reinterpret_cast<int2*>(smem + plan.xcorr);
    uint4* Hq = reinterpret_cast<uint4*>(smem + plan.himg);
    int2* Hc = reinterpret_cast<int2*>(smem + plan.hcorr);
    uint8_t* W1 = smem + plan.w1;
    uint8_t* S1 = smem + plan.s1;
    uint8_t* W2 = smem + plan.w2;
    uint8_t* S2 = smem + plan.s2;
    float* part = reinterpret_cast<float*>(smem + plan.part);  // [slot][row]
    char* ws = static_cast<char*>(q.workspace);
    float* h = reinterpret_cast<float*>(ws + h_off);
    unsigned int* counter = reinterpret_cast<unsigned int*>(ws + sync_off);
    const bool inter = q.fc1_layout == MNB_FC1_INTERLEAVED;

    // this CTA's FC1 pairs (flat over the k slots) and FC2 output rows
    int64_t pr0, pr1, n0, n1;
    const int64_t ss_ = sizeof(S);
    split(int64_t(k) * I, copy_unit(rb1, nb1 * ss_, inter ? 2 : 1), blockIdx.x, gridDim.x, pr0, pr1);
    split(H, copy_unit(rb2, nb2 * ss_, 1), blockIdx.x, gridDim.x, n0, n1);
    const int np = static_cast<int>(pr1 - pr0), nr = static_cast<int>(n1 - n0);

    // ------------------------------------------------------ prologue
    if (tid == 0) {
        mbar_init(bar1, 1);
        mbar_init(bar2, 1);
        *s_fail = 0;
        fence_barrier_init();
    }
    if (q.E <= kBlockRouteMaxE && q.E <= kThreads) {
        block_route_fast(q.logits, q.logits_dtype, static_cast<int>(q.E), k, q.normalize, s_idx, s_w, s_logit, q.agg,
                         q.agg_dtype);
    } else {
        if (tid < 32) warp_route(q.logits, q.logits_dtype, static_cast<int>(q.E), k, q.normalize, s_idx, s_w, 1, q.agg,
                                 q.agg_dtype);
        __syncthreads();
    }
    // local FC1 pair lp: gate row at lrow(lp, 0), up row at lrow(lp, 1) of the staged rows
    auto lrow = [&](int lp, int up) { return inter ? 2 * lp + up : up * kMaxPairs + lp; };
    // The copies, issued by the lanes of warp 0 at once (lane 0 arms both
    // barriers first): FC1 pairs [pr0, pr1) fall into at most two slots (two
    // segments, lanes 0-3 and 4-7: packed rows and scales, of the gate and
    // up halves when those are separate); FC2 rows [n0, n1) of slot j on
    // lanes 8 + 2j (packed rows) and 9 + 2j (scales).
    if (warp == 0) {
        const int64_t ss = sizeof(S);
        if (lane == 0) {
            mbar_arrive_expect_tx(bar1, static_cast<uint32_t>(2 * int64_t(np) * (rb1 + nb1 * ss)));
            mbar_arrive_expect_tx(bar2, static_cast<uint32_t>(int64_t(k) * nr * (rb2 + nb2 * ss)));
        }
        __syncwarp();
        if (lane < 8) {
            const int seg = lane >> 2, sub = lane & 3;
            const int j0 = static_cast<int>(pr0 / I);
            const int64_t split_at = min(pr1, int64_t(j0 + 1) * I);
            const int64_t p = seg == 0 ? pr0 : split_at, pe = seg == 0 ? split_at : pr1;
            const bool scales = sub & 1;
            const int up = sub >> 1;
            if (p < pe && (!inter || up == 0)) {
                const int j = j0 + seg;
                const int64_t a0 = p - int64_t(j) * I, cnt = pe - p;
                const int lp = static_cast<int>(p - pr0);
                const int64_t e = s_idx[j];
                // rows: interleaved 2 a0 .. (gate and up together), else up * I + a0 ..
                const int64_t r0 = inter ? 2 * a0 : up * I + a0, nrows = inter ? 2 * cnt : cnt;
                if (scales) {
                    const uint8_t* src = static_cast<const uint8_t*>(q.fc1_s) + (e * 2 * I + r0) * nb1 * ss;
                    bulk_g2s(S1 + lrow(lp, up) * nb1 * ss, src, static_cast<uint32_t>(nrows * nb1 * ss), bar1);
                } else {
                    bulk_g2s(W1 + lrow(lp, up) * rb1, q.fc1_w + (e * 2 * I + r0) * rb1,
                             static_cast<uint32_t>(nrows * rb1), bar1);
                }
            }
        } else if (lane < 8 + 2 * k) {
            const int j = (lane - 8) >> 1;
            const int64_t e = s_idx[j];
            if (lane & 1)
                bulk_g2s(S2 + int64_t(j) * kMaxRows2 * nb2 * ss,
                         static_cast<const uint8_t*>(q.fc2_s) + (e * H + n0) * nb2 * ss,
                         static_cast<uint32_t>(nr * nb2 * ss), bar2);
            else
                bulk_g2s(W2 + int64_t(j) * kMaxRows2 * rb2, q.fc2_w + (e * H + n0) * rb2, static_cast<uint32_t>(nr * rb2),
                         bar2);
        }
    }
    grid_dependency_wait();

    // --------------------------------------------------------- FC1 + SwiGLU
    stage_image(
        Xq, Xc, 1, C1, H, q.act_dtype, q.x_vec != 0, [&](int) -> const void* { return q.X; }, tid, kThreads);
    __syncthreads();
    const int bs_shift = __ffs(q.bs) - 1;
    bool ok = warp_wait(bar1, 0);
    if (ok) {
        constexpr int Z1 = 1 << (B1 - 1);
        // warp unit: pairs lp, lp + 1 -> rows gate lp, up lp, gate lp+1, up lp+1
        for (int lp0 = 2 * warp; lp0 < np; lp0 += 2 * kWarps) {
            const uint8_t* wr[4];
            const S* sr[4];
            const uint8_t* zr[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int lp = min(lp0 + (r >> 1), np - 1), up = r & 1;
                wr[r] = W1 + lrow(lp, up) * rb1;
                sr[r] = reinterpret_cast<const S*>(S1 + lrow(lp, up) * nb1 * sizeof(S));
                const int64_t p = pr0 + lp;
                const int j = static_cast<int>(p / I);
                const int64_t a = p - int64_t(j) * I;
                const int64_t grow = inter ? 2 * a + up : up * I + a;  // row inside the expert's FC1 weight
                zr[r] = q.fc1_zp ? q.fc1_zp + (int64_t(s_idx[j]) * 2 * I + grow) * q.fc1.zp_row : nullptr;
            }
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            auto chunks = [&](auto has_zp) {
                for (int c = lane; c < C1; c += 32) {
                    const int b = (c * 32) >> bs_shift;
                    uint4 qv[4];
                    const uint4* qp = Xq + qbase(0, c, C1);
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) qv[qq] = qp[qq * 32];
                    const int2 cr = Xc[c];
                    const float p2 = __int_as_float(cr.y);
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        uint32_t w[B1];
                        gemv::load_chunk<B1>(wr[r], c, w);
                        int z = Z1;
                        if constexpr (decltype(has_zp)::value) z = gemv::zero_point_code<B1>(zr[r], b);
                        const int T = chunk_dot<B1>(w, qv) - z * cr.x;
                        acc[r] = fmaf(to_f32(sr[r][b]) * p2, static_cast<float>(T), acc[r]);
                    }
                }
            };
            if (q.fc1_zp)
                chunks(std::true_type{});
            else
                chunks(std::false_type{});
            warp_sums<4>(acc);
            if (lane == 0) {
#pragma unroll
                for (int pp = 0; pp < 2; ++pp) {
                    const int lp = lp0 + pp;
                    if (lp >= np) break;
                    const int64_t p = pr0 + lp;
                    const int j = static_cast<int>(p / I);
                    const int64_t a = p - int64_t(j) * I;
                    float bg = 0.f, bu = 0.f;  // biases of the gate and up rows of pair a
                    if (q.fc1_bias) {
                        const int64_t base = int64_t(s_idx[j]) * 2 * I;
                        bg = load_as_f32(q.fc1_bias, q.act_dtype, base + (inter ? 2 * a : a));
                        bu = load_as_f32(q.fc1_bias, q.act_dtype, base + (inter ? 2 * a + 1 : I + a));
                    }
                    h[int64_t(j) * I + a] = silu_mul(acc[2 * pp] + bg, acc[2 * pp + 1] + bu);
                }
            }
        }
    }
    if (!ok) *s_fail = 1;
    __syncthreads();

    // ------------------------------------------------------- grid barrier
    // Every CTA of the grid is resident at once (one per SM at most, and the
    // work ahead of the layer has completed before this kernel starts), so
    // the counter reaches gridDim.x; should other work hold SMs, the bounded
    // wait gives up, records MNB_ERR_TIMEOUT and the CTA retires.
    if (tid == 0) {
        __threadfence();  // this CTA's h before its arrival
        atomicAdd(counter, 1u);
        const unsigned int need = gridDim.x;
        if (load_acquire(counter) < need) {
            const uint64_t t0 = global_ns();
            while (load_acquire(counter) < need) {
                if (global_ns() - t0 > kWaitNs) {
                    record_error(MNB_ERR_TIMEOUT);
                    *s_fail = 1;
                    break;
                }
                __nanosleep(64);
            }
        }
        __threadfence();
    }
    __syncthreads();
    grid_launch_dependents();
    if (*s_fail) {
        if (tid == 0) {  // let the copies land before the CTA exits (bounded)
            mbar_wait(bar1, 0);
            mbar_wait(bar2, 0);
        }
        __syncthreads();
        return;
    }

    // ----------------------------------------------------- FC2 + combine
    stage_image(
        Hq, Hc, k, C2, I, kF32, true, [&](int j) -> const void* { return h + int64_t(j) * I; }, tid, kThreads);
    __syncthreads();
    ok = warp_wait(bar2, 0);
    // tasks: (slot j, rows r0 .. r0+3 of the CTA's output rows), spread over the warps
    const int groups2 = (nr + 3) / 4;
    for (int task = warp; ok && task < k * groups2; task += kWarps) {
        constexpr int Z2 = 1 << (B2 - 1);
        const int j = task / groups2, r0 = (task - j * groups2) * 4;
        const int64_t e = s_idx[j];
        const uint8_t* Wj = W2 + int64_t(j) * kMaxRows2 * rb2;
        const S* Sj = reinterpret_cast<const S*>(S2 + int64_t(j) * kMaxRows2 * nb2 * sizeof(S));
        {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            const uint8_t* wr[4];
            const S* sr[4];
            const uint8_t* zr[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int rl = min(r0 + r, nr - 1);
                wr[r] = Wj + int64_t(rl) * rb2;
                sr[r] = Sj + rl * nb2;
                zr[r] = q.fc2_zp ? q.fc2_zp + (e * H + n0 + rl) * q.fc2.zp_row : nullptr;
            }
            auto chunks = [&](auto has_zp) {
                for (int c = lane; c < C2; c += 32) {
                    const int b = (c * 32) >> bs_shift;
                    uint4 qv[4];
                    const uint4* qp = Hq + qbase(j, c, C2);
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) qv[qq] = qp[qq * 32];
                    const int2 cr = Hc[j * C2 + c];
                    const float p2 = __int_as_float(cr.y);
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        uint32_t w[B2];
                        gemv::load_chunk<B2>(wr[r], c, w);
                        int z = Z2;
                        if constexpr (decltype(has_zp)::value) z = gemv::zero_point_code<B2>(zr[r], b);
                        const int T = chunk_dot<B2>(w, qv) - z * cr.x;
                        acc[r] = fmaf(to_f32(sr[r][b]) * p2, static_cast<float>(T), acc[r]);
                    }
                }
            };
            if (q.fc2_zp)
                chunks(std::true_type{});
            else
                chunks(std::false_type{});
            warp_sums<4>(acc);
            if (lane == 0) {
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    if (r0 + r < nr)
                        part[j * kMaxRows2 + r0 + r] =
                            acc[r] + (q.fc2_bias ? load_as_f32(q.fc2_bias, q.act_dtype, e * H + n0 + r0 + r) : 0.f);
            }
        }
    }
    if (!ok) *s_fail = 1;
    __syncthreads();
    if (*s_fail) return;
    if (tid < nr) {
        float y = 0.f;
        for (int j = 0; j < k; ++j) y = fmaf(s_w[j], part[j * kMaxRows2 + tid], y);
        store_from_f32(q.Y, q.act_dtype, n0 + tid, y);
    }
}

template <int B1, int B2, int ST>
cudaError_t launch_typed(const QmoeArgs& q, int grid, int64_t smem, int64_t h_off, int64_t sync_off, bool pdl,
                         cudaStream_t stream) {
    char* ws = static_cast<char*>(q.workspace);
    // the counter is zeroed by a one-CTA kernel that waits for the work ahead
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1, 1, 1);
        cfg.blockDim = dim3(32, 1, 1);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = pdl ? 1 : 0;
        cudaError_t e = set_max_carveout(qmoe_decode_prep_kernel);
        if (e != cudaSuccess) return e;
        e = cudaLaunchKernelEx(&cfg, qmoe_decode_prep_kernel, reinterpret_cast<unsigned int*>(ws + sync_off));
        if (e != cudaSuccess) return e;
    }
    auto kern = qmoe_decode_fused_kernel<B1, B2, ST>;
    cudaError_t e = set_kernel_smem(kern, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);  // <= one CTA per SM
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, q, h_off, sync_off);
}

template <int ST>
cudaError_t launch_bits(const QmoeArgs& q, int grid, int64_t smem, int64_t h_off, int64_t sync_off, bool pdl,
                        cudaStream_t stream) {
    if (q.fc1_bits == 3 && q.fc2_bits == 3) return launch_typed<3, 3, ST>(q, grid, smem, h_off, sync_off, pdl, stream);
    if (q.fc1_bits == 3 && q.fc2_bits == 4) return launch_typed<3, 4, ST>(q, grid, smem, h_off, sync_off, pdl, stream);
    if (q.fc1_bits == 4 && q.fc2_bits == 3) return launch_typed<4, 3, ST>(q, grid, smem, h_off, sync_off, pdl, stream);
    return launch_typed<4, 4, ST>(q, grid, smem, h_off, sync_off, pdl, stream);
}

}  // namespace

cudaError_t qmoe_decode_take_error(unsigned int* out) { return take_unit_error(out); }

cudaError_t launch_qmoe_decode_fused(const QmoeArgs& q, int sm_count, bool pdl, cudaStream_t stream) {
    if (q.T != 1 || q.k > kMaxK) return cudaErrorNotSupported;
    const int ssize = 2;
    const int nb1 = static_cast<int>(q.fc1.nb), nb2 = static_cast<int>(q.fc2.nb);
    const int64_t rb1 = q.fc1.row_bytes, rb2 = q.fc2.row_bytes;
    // every bulk copy must be a whole number of 16-byte units at 16-byte
    // offsets: CTAs take pairs and rows in copy units, which must tile an
    // expert (I pairs) and the output (H rows)
    const bool inter = q.fc1_layout == MNB_FC1_INTERLEAVED;
    const int64_t u1 = copy_unit(rb1, int64_t(nb1) * ssize, inter ? 2 : 1), u2 = copy_unit(rb2, int64_t(nb2) * ssize, 1);
    if (u1 > 8 || u2 > 8 || q.I % u1 || q.H % u2) return cudaErrorNotSupported;
    // bases of the expert matrices (16-byte aligned pointers, whole-unit expert strides)
    if ((2 * q.I * rb1) % 16 || (2 * q.I * nb1 * ssize) % 16 || (q.H * rb2) % 16 || (q.H * nb2 * ssize) % 16)
        return cudaErrorNotSupported;
    const int64_t pairs = int64_t(q.k) * q.I;
    int grid = static_cast<int>(std::min<int64_t>(sm_count, std::min<int64_t>(pairs / u1, q.H / u2)));
    if (grid < 1) return cudaErrorNotSupported;
    if (cdiv<int64_t>(pairs / u1, grid) * u1 > kMaxPairs || cdiv<int64_t>(q.H / u2, grid) * u2 > kMaxRows2)
        return cudaErrorNotSupported;
    if (cdiv<int64_t>(pairs / u1, grid) * u1 > q.I) return cudaErrorNotSupported;  // a CTA's pairs span <= 2 slots
    const int C1 = static_cast<int>(q.fc1.nb * q.bs / 32), C2 = static_cast<int>(q.fc2.nb * q.bs / 32);
    const DecPlan p = dec_plan(C1, C2, q.k, rb1, nb1, rb2, nb2, ssize);
    if (p.total > kSmemCap) return cudaErrorNotSupported;
    int64_t h_off = 0, sync_off = 0;
    qmoe_ws_decode_regions(q.T, q.H, q.I, q.E, q.k, &h_off, &sync_off);
    return q.act_dtype == MNB_F16 ? launch_bits<kF16>(q, grid, p.total, h_off, sync_off, pdl, stream)
                                  : launch_bits<kBF16>(q, grid, p.total, h_off, sync_off, pdl, stream);
}

}  // namespace mnb
