// gemv_impl.cuh -- packed INT4 / INT3 weight-only GEMV (M = 1 decode) and
// small-M matmul on CUDA cores, sm_103a: the kernel and its launch templates,
// instantiated by gemv.cu (the raw row-local layout) and gemv_pp.cu (the
// prepacked layout).
//
// Follows "Qwen3 Missing-Kernel Implementation Plan", rows K02/K03: scales and
// zero points are applied while bounded panels of the packed weights are
// consumed; no dequantised weight matrix is ever written to global memory.
//
// Design (HBM-bound: the packed weights and scales are the traffic):
//  * A CTA owns one contiguous range of row blocks (RC = 8 warps x rpw rows).
//    Rows are contiguous in the [N, nb, blob] layout, so the range's packed
//    bytes and scales are two contiguous byte ranges: before its grid
//    dependency wait the CTA asks L2 to prefetch them (the whole range when
//    the matrix is small enough to sit in L2 beside its neighbours, else the
//    first ring-full); right after the wait it lets the next kernel on the
//    stream launch, whose CTAs then prefetch their own rows while this one
//    computes.  Nothing the CTA reads is read before the wait (a prefetch
//    only warms L2, which stays coherent with any later write).
//  * Warp 8 is the producer: one lane keeps a ring of NST stages filled with
//    bulk (TMA) copies of whole row blocks, waiting on per-stage "empty"
//    mbarriers; the 8 consumer warps wait on the per-stage "full" mbarriers.
//  * The activations are staged once per CTA as a fixed-point image
//    (gemv_int.cuh); each consumer warp owns a slice of rpw rows of a block
//    and walks their 32-code chunks R rows at a time, one chunk per lane,
//    with exact dp4a integer dot
//    products per chunk; the R x MT sums are reduced together with shuffles
//    that hand half of the values to the partner lane at each step (fixed
//    order, so results are deterministic).
#pragma once

#include <algorithm>
#include <mutex>
#include <type_traits>
#include <unordered_map>

#include "common.cuh"
#include "gemv_core.cuh"
#include "gemv_int.cuh"
#include "kernels.h"

namespace mnb {

namespace {

using namespace gemv_int;

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxStages = 8;
constexpr int64_t kSmemBudget = 227 * 1024;

__host__ __device__ constexpr int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

struct Plan {
    int64_t qimg, corr, w_stage, s_stage, fixed;
    int stages;
    int64_t total;
};

__host__ __device__ inline Plan make_plan(int MT, int C, int RC, int64_t row_bytes, int nb, int ssize, int stages) {
    Plan p;
    p.qimg = qimg_bytes(MT, C);
    p.corr = corr_bytes(MT, C);
    p.w_stage = round_up(int64_t(RC) * row_bytes, 128);
    p.s_stage = round_up(int64_t(RC) * nb * ssize, 128);
    p.fixed = 256 + p.qimg + p.corr;
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

// Blocks [first, last) of CTA x among gx CTAs: contiguous, sizes differing by at most one.
__device__ __forceinline__ void cta_blocks(int nblk, int x, int gx, int& first, int& last) {
    const int q = nblk / gx, r = nblk - q * gx;
    first = x * q + min(x, r);
    last = first + q + (x < r ? 1 : 0);
}

// PP: the weight comes in the prepacked layout (rows of codes, scales and zero
// points, whole 16-byte units; INT3 chunks regrouped), checked against its
// device header after the dependency wait.
// GR: one projection of a grouped QMoE layer: blockIdx.y is an m-tile of <= MT
// expert-sorted rows of one expert (read after the dependency wait), whose
// weight starts e * stride bytes into B, scales and zero points; activation
// rows come through the routing permutation (FC1) or in sorted order (FC2),
// output rows are sorted positions, and an optional per-expert bias is added.
template <int BITS, int ST, int MT, int R, bool PP, bool GR>
__device__ __forceinline__ void gemv_body(const GemvArgs& a) {
    using S = typename DType<ST>::T;
    // Blocks of RC = 8 * rpw rows: warp w takes rows [w rpw, (w+1) rpw) of
    // every block, R rows at a time (rpw = R for the large matrices; small
    // matrices have one block per CTA and rpw of 1..4).
    const int RC = a.rows_per_block;
    const int rpw = RC / kConsumerWarps;
    extern __shared__ __align__(128) uint8_t smem[];

    const int C = a.chunks, nb = a.nb;
    const Plan plan = make_plan(MT, C, RC, a.row_bytes, nb, PP ? 0 : int(sizeof(S)), a.stages);
    const int NST = plan.stages;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kMaxStages;
    uint4* Q = reinterpret_cast<uint4*>(smem + 256);
    int2* Corr = reinterpret_cast<int2*>(smem + 256 + plan.qimg);
    uint8_t* Wst = smem + plan.fixed;
    uint8_t* Sst = Wst + NST * plan.w_stage;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // activation / output rows [mbase, mbase + mcnt) (GR: set from the m-tile)
    int64_t mbase = int64_t(blockIdx.y) * MT;
    int mcnt = static_cast<int>(min(int64_t(MT), a.M - mbase));
    // the weight, its scales and zero points (GR: the m-tile's expert)
    const uint8_t* Bw = a.B;
    const uint8_t* Sw = static_cast<const uint8_t*>(a.scales);
    const uint8_t* Zw = a.zp;
    int ge = 0;
    int b_first, b_last;
    cta_blocks(a.n_blocks, blockIdx.x, gridDim.x, b_first, b_last);
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
        // L2 prefetch of this CTA's rows (a hint that reads nothing we use;
        // a grouped CTA learns its expert only after the wait)
        if (!GR && b_first < b_last) {
            const int pf_last = a.prefetch_all ? b_last : min(b_last, b_first + NST);
            const int64_t r0 = int64_t(b_first) * RC, r1 = min(int64_t(pf_last) * RC, a.N);
            const int64_t ss = sizeof(S);
            auto prefetch = [](const uint8_t* p, int64_t bytes) {
                const uintptr_t start = reinterpret_cast<uintptr_t>(p) & ~uintptr_t(15);
                int64_t n = int64_t(reinterpret_cast<uintptr_t>(p) + bytes - start) & ~int64_t(15);
                for (int64_t off = 0; off < n; off += int64_t(1) << 30) {
                    const int64_t len = min(n - off, int64_t(1) << 30);
                    bulk_prefetch_l2(reinterpret_cast<const void*>(start + off), static_cast<uint32_t>(len));
                }
            };
            prefetch(a.B + r0 * a.row_bytes, (r1 - r0) * a.row_bytes);
            if (!PP) prefetch(static_cast<const uint8_t*>(a.scales) + r0 * nb * ss, (r1 - r0) * nb * ss);
            if (PP) bulk_prefetch_l2(a.pp_header, MNB_PREPACK_HEADER_BYTES);  // read right after the wait
        }
    }
    // The next kernel on the stream may start its prologue (its own L2
    // prefetch) once this one has passed its dependency wait: one kernel of a
    // chain runs ahead, no more (letting several run ahead measured slower).
    grid_dependency_wait();
    grid_launch_dependents();
    if constexpr (PP) {
        // the device header must describe this weight: a buffer re-prepacked
        // for another weight, or overwritten, is refused before any code is read
        volatile int* ok = reinterpret_cast<volatile int*>(smem + 2 * kMaxStages * 8);
        if (tid == 0) {
            const mnb_prepacked_desc* h = static_cast<const mnb_prepacked_desc*>(a.pp_header);
            const bool good = h->magic == MNB_PREPACK_MAGIC && h->version == MNB_PREPACK_VERSION &&
                              h->identity == a.pp_identity && h->N == a.N && h->K == a.K && h->bits == a.bits &&
                              h->block_size == a.bs && h->row_stride == a.row_bytes;
            *ok = good ? 1 : 0;
            if (!good && blockIdx.x == 0 && blockIdx.y == 0) record_error(MNB_ERR_INVALID_ARG);
        }
        __syncthreads();
        if (!*ok) return;  // nothing in flight yet: no copy has been issued
    } else if constexpr (GR) {
        // [0] expert (-1: no tile), [1] first sorted row, [2] rows, [4 + m] activation row of row m
        volatile int* gt = reinterpret_cast<volatile int*>(smem + 2 * kMaxStages * 8);
        if (tid == 0) {
            int4 t = make_int4(-1, 0, 0, 0);
            if (static_cast<int>(blockIdx.y) < *a.g_ntiles) t = a.g_tiles[blockIdx.y];
            gt[0] = t.x;
            gt[1] = t.y;
            gt[2] = t.z;
            for (int m = 0; m < MT; ++m) {
                const int srow = t.y + (m < t.z ? m : 0);
                gt[4 + m] = (t.x >= 0 && a.g_perm) ? a.g_perm[srow] / a.g_k : srow;
            }
        }
        __syncthreads();
        if (gt[0] < 0) return;  // past the device's tile count: nothing issued
        ge = gt[0];
        mbase = gt[1];
        mcnt = gt[2];
        Bw += int64_t(ge) * a.w_estride;
        Sw += int64_t(ge) * a.s_estride;
        if (Zw) Zw += int64_t(ge) * a.z_estride;
    } else {
        __syncthreads();
    }

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------- producer
        if (lane != 0) return;
        int st = 0;
        uint32_t round = 0;  // times the ring has wrapped
        for (int blk = b_first; blk < b_last; ++blk) {
            if (round && !mbar_wait(&empty[st], (round - 1) & 1)) {
                for (int j = 0; j < NST; ++j) mbar_wait(&full[j], 0);  // give in-flight copies a bounded chance
                return;
            }
            const int64_t n0 = int64_t(blk) * RC;
            const int rc = block_rows(blk);
            uint8_t* W = Wst + st * plan.w_stage;
            uint8_t* Sd = Sst + st * plan.s_stage;
            if (PP) {
                // prepacked rows are whole 16-byte units holding their scales and zero points
                const uint32_t wb = static_cast<uint32_t>(rc * a.row_bytes);
                mbar_arrive_expect_tx(&full[st], wb);
                bulk_g2s(W, a.B + n0 * a.row_bytes, wb, &full[st]);
            } else if (a.swiglu && !a.fc1_inter) {
                // concatenated gate/up halves: the block's pairs [n0/2, n0/2 + rc/2) of
                // the gate rows, then the same pairs of the up rows (every copy whole
                // 16-byte units: the launcher checks the row alignment)
                const int64_t p0 = n0 / 2, np = rc / 2, ss = int64_t(nb) * sizeof(S);
                const uint32_t wb = static_cast<uint32_t>(np * a.row_bytes), sb = static_cast<uint32_t>(np * ss);
                mbar_arrive_expect_tx(&full[st], 2 * (wb + sb));
                for (int up = 0; up < 2; ++up) {
                    const int64_t r = up * a.pairs + p0;
                    bulk_g2s(W + up * (RC / 2) * a.row_bytes, Bw + r * a.row_bytes, wb, &full[st]);
                    bulk_g2s(Sd + up * (RC / 2) * ss, Sw + r * ss, sb, &full[st]);
                }
            } else {
                const int64_t wtot = rc * a.row_bytes, stot = int64_t(rc) * nb * sizeof(S);
                const uint32_t wb = static_cast<uint32_t>(wtot) & ~15u, sb = static_cast<uint32_t>(stot) & ~15u;
                const uint8_t* wsrc = Bw + n0 * a.row_bytes;
                const uint8_t* ssrc = Sw + n0 * nb * int64_t(sizeof(S));
                // bytes past the last 16-byte multiple of a partial block: plain copies, published by the arrive below
                if (wb < wtot) copy_bytes(W, wsrc, wb, wtot);
                if (sb < stot) copy_bytes(Sd, ssrc, sb, stot);
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(&full[st], wb + sb);
                if (wb) bulk_g2s(W, wsrc, wb, &full[st]);
                if (sb) bulk_g2s(Sd, ssrc, sb, &full[st]);
            }
            if (++st == NST) { st = 0; ++round; }
        }
        return;
    }

    // ------------------------------------------------------------ consumers
    const int esz = a.a_dtype == kF32 ? 4 : 2;
    stage_image(
        Q, Corr, MT, C, a.K, a.a_dtype, a.a_vec != 0,
        [&](int m) -> const void* {
            if constexpr (GR) {
                if (m >= mcnt) return nullptr;
                const int64_t row = reinterpret_cast<volatile const int*>(smem + 2 * kMaxStages * 8)[4 + m];
                return static_cast<const char*>(a.A) + row * a.K * esz;
            } else {
                return mbase + m < a.M ? static_cast<const char*>(a.A) + (mbase + m) * a.K * esz : nullptr;
            }
        },
        tid, kConsumerWarps * 32, a.int8a ? 4 * a.bs / 32 : 0);
    consumer_sync();

    const int bs_shift = __ffs(a.bs) - 1;
    // BITS == 0: any width 1..8 given at run time (codes read straight from shared memory)
    const int bits_rt = BITS ? BITS : a.bits;
    const int kZImplicit = 1 << (bits_rt - 1);
    // The block loop over MTE activation rows of the image (MTE <= MT), RE
    // weight rows per pass: a grouped CTA runs it at its m-tile's row count, so
    // a short tile costs no more than its rows.
    auto consume = [&](auto mte) {
        constexpr int MTE = decltype(mte)::value;
        // grouped: four weight rows per pass for short m-tiles (the launch's
        // blocks hold four rows per warp), two for full ones (registers)
        constexpr int RE = (GR && MTE <= 2) ? 4 : R;
        int st = 0;
        uint32_t phase = 0;
        for (int blk = b_first; blk < b_last; ++blk) {
            if (!warp_wait(&full[st], phase)) return;
            const int64_t n0 = int64_t(blk) * RC;
            const int rc = block_rows(blk);
            const uint8_t* W = Wst + st * plan.w_stage;
            const S* Sc = reinterpret_cast<const S*>(Sst + st * plan.s_stage);
            // this warp's slice of the block, RE rows at a time
            const int w_end = min(rc, (warp + 1) * rpw);
            for (int r0 = warp * rpw; r0 < w_end; r0 += RE) {
                float acc[RE][MTE];
#pragma unroll
                for (int r = 0; r < RE; ++r)
#pragma unroll
                    for (int m = 0; m < MTE; ++m) acc[r][m] = 0.f;
                const uint8_t* wrow[RE];
                const S* srow[RE];
                const uint8_t* zrow[RE];
#pragma unroll
                for (int r = 0; r < RE; ++r) {
                    const int rl = min(r0 + r, w_end - 1);  // rows past the slice end recompute its last row
                    // concatenated gate/up: logical row 2i / 2i+1 sits in the gate / up half of the stage
                    const int sl = (a.swiglu && !a.fc1_inter) ? ((rl & 1) ? RC / 2 + (rl >> 1) : (rl >> 1)) : rl;
                    wrow[r] = W + int64_t(sl) * a.row_bytes;
                    if constexpr (PP) {  // the row's scales and zero points follow its codes in the stage
                        srow[r] = reinterpret_cast<const S*>(wrow[r] + a.pp_scale_off);
                        zrow[r] = a.pp_zp_off >= 0 ? wrow[r] + a.pp_zp_off : nullptr;
                    } else {
                        srow[r] = Sc + sl * nb;
                        const int64_t phys =
                            (a.swiglu && !a.fc1_inter) ? ((rl & 1) ? a.pairs : 0) + (n0 + rl) / 2 : n0 + rl;
                        zrow[r] = Zw ? Zw + phys * a.zp_row_bytes : nullptr;
                    }
                }
                // the chunk loop; HAS_ZP: explicit zero points (a uniform branch, taken once per block)
                auto chunks = [&](auto has_zp) {
                    for (int c = lane; c < C; c += 32) {
                        const int b = (c * 32) >> bs_shift;
                        uint4 q[MTE][4];
                        float p2[MTE];
                        int V[MTE];
#pragma unroll
                        for (int m = 0; m < MTE; ++m) {
                            const uint4* qp = Q + qbase(m, c, C);
#pragma unroll
                            for (int qq = 0; qq < 4; ++qq) q[m][qq] = qp[qq * 32];
                            const int2 cr = Corr[m * C + c];
                            V[m] = cr.x;
                            p2[m] = __int_as_float(cr.y);
                        }
#pragma unroll
                        for (int r = 0; r < RE; ++r) {
                            const float sc = to_f32(srow[r][b]);
                            int z = kZImplicit;
                            if constexpr (BITS == 0) {
                                if constexpr (decltype(has_zp)::value) z = zero_point_any(zrow[r], b, bits_rt);
                                uint32_t lo[4], hi[4];
                                codes_any(wrow[r] + c * 4 * bits_rt, bits_rt, lo, hi);
#pragma unroll
                                for (int m = 0; m < MTE; ++m) {
                                    const int T = chunk_dot_bytes(lo, hi, q[m]) - z * V[m];
                                    acc[r][m] = fmaf(sc * p2[m], static_cast<float>(T), acc[r][m]);
                                }
                            } else {
                                uint32_t w[BITS];
                                gemv::load_chunk<BITS>(wrow[r], c, w);
                                if constexpr (decltype(has_zp)::value) z = gemv::zero_point_code<BITS>(zrow[r], b);
#pragma unroll
                                for (int m = 0; m < MTE; ++m) {
                                    const int T = chunk_dot<BITS, PP>(w, q[m]) - z * V[m];
                                    acc[r][m] = fmaf(sc * p2[m], static_cast<float>(T), acc[r][m]);
                                }
                            }
                        }
                    }
                };
                if (PP ? a.pp_zp_off >= 0 : a.zp != nullptr)
                    chunks(std::true_type{});
                else
                    chunks(std::false_type{});
                // value q = r * MTE + m; each total ends in one lane
                if (a.swiglu) {
                    // rows 2i, 2i+1 of the group are the gate and up rows of one pair:
                    // every lane gets every total, lane 0 stores silu(gate) * up
                    if constexpr (RE % 2 == 0) {
#pragma unroll
                        for (int r = 0; r < RE; ++r)
#pragma unroll
                            for (int m = 0; m < MTE; ++m) acc[r][m] = warp_sum(acc[r][m]);
                        if (lane == 0) {
#pragma unroll
                            for (int pp = 0; pp < RE / 2; ++pp) {
#pragma unroll
                                for (int m = 0; m < MTE; ++m) {
                                    if (r0 + 2 * pp + 1 < w_end && (GR ? m < mcnt : mbase + m < a.M)) {
                                        float gt = acc[2 * pp][m], up = acc[2 * pp + 1][m];
                                        if constexpr (GR) {
                                            if (a.bias) {  // rows in the weight's layout, per expert
                                                const int64_t i = (n0 + r0) / 2 + pp, b0 = int64_t(ge) * 2 * a.pairs;
                                                gt += load_as_f32(a.bias, a.bias_dtype, b0 + (a.fc1_inter ? 2 * i : i));
                                                up += load_as_f32(a.bias, a.bias_dtype,
                                                                  b0 + (a.fc1_inter ? 2 * i + 1 : a.pairs + i));
                                            }
                                        }
                                        store_from_f32(a.Y, a.y_dtype, (mbase + m) * a.y_ld + (n0 + r0) / 2 + pp,
                                                       gt / (1.0f + expf(-gt)) * up);
                                    }
                                }
                            }
                        }
                    }
                } else {
                    constexpr int N = RE * MTE;
                    float part[N];
#pragma unroll
                    for (int r = 0; r < RE; ++r)
#pragma unroll
                        for (int m = 0; m < MTE; ++m) part[r * MTE + m] = acc[r][m];
                    const float total = warp_sum_transpose<N>(part);
                    if ((lane & (32 / N - 1)) == 0) {
                        const int qv = transpose_row<N>(lane), r = qv / MTE, m = qv - r * MTE;
                        if (r0 + r < w_end && (GR ? m < mcnt : mbase + m < a.M)) {
                            float y = total;
                            if constexpr (GR) {
                                if (a.bias) y += load_as_f32(a.bias, a.bias_dtype, int64_t(ge) * a.N + n0 + r0 + r);
                            }
                            store_from_f32(a.Y, a.y_dtype, (mbase + m) * a.y_ld + n0 + r0 + r, y);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
            if (++st == NST) { st = 0; phase ^= 1; }
        }
    };
    if constexpr (GR) {
        if (mcnt == 1)
            consume(std::integral_constant<int, 1>{});
        else if (mcnt == 2 && MT > 2)
            consume(std::integral_constant<int, (MT > 2 ? 2 : MT)>{});
        else
            consume(std::integral_constant<int, MT>{});
    } else {
        consume(std::integral_constant<int, MT>{});
    }
}

template <int BITS, int ST, int MT, int R, bool PP = false>
__global__ void __launch_bounds__(kThreads) gemv_kernel(const __grid_constant__ GemvArgs a) {
    gemv_body<BITS, ST, MT, R, PP, false>(a);
}

// The grouped form, held to two CTAs per SM (registers).
template <int BITS, int ST, int MT, int R>
__global__ void __launch_bounds__(kThreads, 2) gemv_grouped_kernel(const __grid_constant__ GemvArgs a) {
    gemv_body<BITS, ST, MT, R, false, true>(a);
}

int ssize_of(int dt) { return dt == kF32 ? 4 : 2; }

int pick_mt(int64_t M) { return M <= 1 ? 1 : (M <= 2 ? 2 : 4); }

// The smallest row count for which every block's packed bytes and scales
// start on a 16-byte boundary (a power of two).
int64_t row_align(int64_t row_bytes, int nb, int ssize) {
    auto g16 = [](int64_t x) { int64_t g = 16; while (x % g) g >>= 1; return 16 / g; };
    return std::max(g16(row_bytes), g16(int64_t(nb) * ssize));
}

// Matrices up to this many bytes are prefetched into L2 whole before the
// dependency wait: a few of them fit in the 129 MB L2 beside the kernels
// still running, so a chain of decode projections streams without gaps.
constexpr int64_t kPrefetchAllBytes = int64_t(32) << 20;

// Launch shape.
//  * Small matrices (prefetched into L2 whole; the layer projections of a
//    decode step): one block per CTA, one CTA per SM, every warp a slice of
//    rows, the block's rows and scales moved by two bulk copies.  Such a
//    launch is mostly latency (the dependency release, one L2 round trip for
//    the activations and the rows, the stores); this keeps the compute part to
//    one short pass per warp and the copies few and large.
//  * Large matrices (the vocabulary head): a ring with `cps` CTAs per SM (three
//    where the kernel's registers allow, else two) and up to ~80 KB of ring
//    each, so that 120-190 KB per SM are in flight (bulk copies need well over
//    64 KB in flight per SM to reach HBM bandwidth); each warp takes R rows of
//    every block.
struct Shape {
    int R = 4, stages = 2, grid = 1, rows_per_block = 32;
    bool prefetch_all = false;
};

Shape pick_shape(int64_t N, int64_t row_bytes, int nb, int ssize, int MT, int C, int sm_count, int64_t mgroups,
                 int force_r = 0, bool pairs = false, int cps = 2) {
    const int64_t align = row_align(row_bytes, nb, ssize);
    const int64_t row_total = row_bytes + int64_t(nb) * ssize;
    const bool small = N * row_total <= kPrefetchAllBytes;
    Shape best;
    if (small) {
        // one block per CTA and one CTA per SM (at ~70 registers a thread an
        // SM holds three such CTAs: this kernel's, and the next two kernels'
        // of a chain, which prefetch their rows meanwhile), each warp a slice
        // of rpw rows of the block (two bulk copies per CTA)
        const int64_t ctas = std::max<int64_t>(1, sm_count / mgroups);
        int64_t rpw = cdiv<int64_t>(N, ctas * kConsumerWarps);
        rpw = rpw <= 2 ? rpw : rpw <= 4 ? 4 : cdiv<int64_t>(rpw, 2) * 2;  // 1, 2, 4, then even
        if (pairs && rpw % 2) ++rpw;  // SwiGLU: every warp slice holds whole gate/up pairs
        while ((rpw * kConsumerWarps) % (pairs ? 2 * align : align) != 0) ++rpw;
        int R = force_r ? force_r : rpw % 4 == 0 ? 4 : rpw % 2 == 0 ? 2 : 1;
        if (MT == 4 && R == 4) R = 2;  // four activation rows: at most two weight rows per pass (registers)
        const int64_t RC = rpw * kConsumerWarps;
        const Plan p = make_plan(MT, C, static_cast<int>(RC), row_bytes, nb, ssize, 1);
        if (rpw <= 8 && p.total <= 100 * 1024) {
            best.R = R;
            best.rows_per_block = static_cast<int>(RC);
            best.stages = 1;
            best.grid = static_cast<int>(cdiv<int64_t>(N, RC));
            best.prefetch_all = true;
            return best;
        }
    }
    const int64_t per_group = std::max<int64_t>(1, int64_t(sm_count) * cps / mgroups);  // CTAs per activation group
    const int64_t per_cta = (kSmemBudget / cps) & ~int64_t(1023);  // shared memory of one of cps CTAs
    double best_cost = -1;
    for (int R : {4, 2, 1}) {
        if (MT == 4 && R == 4) continue;
        if (force_r && R != force_r) continue;
        if (pairs && R == 1) continue;
        const int RC = kConsumerWarps * R;
        if (RC % (pairs ? 2 * align : align) != 0) continue;
        const Plan p1 = make_plan(MT, C, RC, row_bytes, nb, ssize, 1);
        const int64_t stage = p1.w_stage + p1.s_stage;
        const int64_t cap = cps == 2 ? std::max<int64_t>(112 * 1024, p1.fixed + 2 * stage) : per_cta;
        if (p1.fixed + 2 * stage > (cps == 2 ? kSmemBudget : per_cta)) continue;
        int st = static_cast<int>(std::min<int64_t>(kMaxStages, std::max<int64_t>(2, (80 * 1024) / stage)));
        while (st > 2 && p1.fixed + st * stage > cap) --st;
        const int64_t nblk = cdiv<int64_t>(N, RC);
        const int64_t ctas = std::max<int64_t>(1, std::min<int64_t>(nblk, per_group));
        const int64_t share = cdiv<int64_t>(nblk, ctas) * RC;  // rows of the busiest CTA
        // fewer rows per warp re-read the activation image more often per code
        const double cost = double(share) * (R == 4 ? 1.0 : R == 2 ? 1.03 : 1.08);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best.R = R;
            best.rows_per_block = RC;
            best.stages = st;
            // as few CTAs as give every CTA the busiest CTA's share
            best.grid = static_cast<int>(cdiv<int64_t>(nblk, cdiv<int64_t>(nblk, ctas)));
        }
    }
    best.prefetch_all = small;
    if (best_cost < 0) best.stages = 0;  // no row count fits this many CTAs per SM
    return best;
}

template <int BITS, int ST, int MT, int R, bool PP = false>
cudaError_t launch_typed(GemvArgs a, const Shape& sh, bool pdl, cudaStream_t stream) {
    const int ssize = PP ? 0 : ST == kF32 ? 4 : 2;
    a.rows_per_block = sh.rows_per_block;
    a.n_blocks = static_cast<int>(cdiv<int64_t>(a.N, sh.rows_per_block));
    a.stages = sh.stages;
    a.prefetch_all = sh.prefetch_all ? 1 : 0;
    const Plan p = make_plan(MT, a.chunks, sh.rows_per_block, a.row_bytes, a.nb, ssize, sh.stages);
    if (sh.stages < 1 || p.total > kSmemBudget) return cudaErrorNotSupported;
    auto kern = gemv_kernel<BITS, ST, MT, R, PP>;
    cudaError_t e = set_kernel_smem(kern, p.total);
    if (e != cudaSuccess) return e;
    const int64_t mgroups = cdiv<int64_t>(a.M, MT);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(std::min<int64_t>(sh.grid, a.n_blocks)), static_cast<unsigned>(mgroups), 1);
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

// CTAs of this instantiation an SM holds with `smem` bytes of dynamic shared
// memory (registers, shared memory and threads), cached per (kernel, smem).
template <int BITS, int ST, int MT, int R, bool PP>
int resident_ctas(int64_t smem) {
    static std::mutex mu;
    static std::unordered_map<int64_t, int> cache;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(smem);
    if (it != cache.end()) return it->second;
    auto kern = gemv_kernel<BITS, ST, MT, R, PP>;
    int n = 0;
    if (set_kernel_smem(kern, smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, static_cast<size_t>(smem)) != cudaSuccess)
        n = 0;
    cache.emplace(smem, n);
    return n;
}

template <int BITS, int ST, int MT, bool PP>
int resident_ctas_r(int R, int64_t smem) {
    if constexpr (BITS == 0) {
        return resident_ctas<0, ST, MT, 2, PP>(smem);
    } else {
        if constexpr (MT < 4) {
            if (R == 4) return resident_ctas<BITS, ST, MT, 4, PP>(smem);
        }
        if (R == 2) return resident_ctas<BITS, ST, MT, 2, PP>(smem);
        return resident_ctas<BITS, ST, MT, 1, PP>(smem);
    }
}

// The launch shape of the large-matrix ring: three CTAs per SM where that
// instantiation's registers and shared memory let three be resident (the
// rows are split evenly over co-resident CTAs, so a CTA that had to wait for
// a free slot would double the time), else two.
template <int BITS, int ST, int MT, bool PP>
Shape pick_shape_resident(const GemvArgs& a, int ssize, int sm_count, int64_t mgroups, int force_r) {
    const Shape sh2 = pick_shape(a.N, a.row_bytes, a.nb, ssize, MT, a.chunks, sm_count, mgroups, force_r,
                                 a.swiglu != 0, 2);
    if (sh2.prefetch_all) return sh2;  // the small-matrix shape: one CTA per SM
    // a third CTA with the same rows per pass (fewer rows per pass re-read the
    // activation image more often: measured slower than two CTAs)
    const Shape sh3 = pick_shape(a.N, a.row_bytes, a.nb, ssize, MT, a.chunks, sm_count, mgroups, sh2.R,
                                 a.swiglu != 0, 3);
    if (sh3.stages == 0 || sh3.R != sh2.R) return sh2;
    const Plan p = make_plan(MT, a.chunks, sh3.rows_per_block, a.row_bytes, a.nb, ssize, sh3.stages);
    return resident_ctas_r<BITS, ST, MT, PP>(sh3.R, p.total) >= 3 ? sh3 : sh2;
}

template <int BITS, int ST, int MT, bool PP = false>
cudaError_t launch_r(const GemvArgs& a, const Shape& sh, bool pdl, cudaStream_t stream) {
    if constexpr (BITS == 0) {  // any width: one register tile (the shape picks R = 2)
        return launch_typed<0, ST, MT, 2>(a, sh, pdl, stream);
    } else {
        if constexpr (MT < 4) {
            if (sh.R == 4) return launch_typed<BITS, ST, MT, 4, PP>(a, sh, pdl, stream);
        }
        if (sh.R == 2) return launch_typed<BITS, ST, MT, 2, PP>(a, sh, pdl, stream);
        return launch_typed<BITS, ST, MT, 1, PP>(a, sh, pdl, stream);
    }
}

template <int BITS, int ST, bool PP = false>
cudaError_t launch_mt(const GemvArgs& a, int sm_count, bool pdl, cudaStream_t stream) {
    // any width: at most two activation rows per pass (the code extraction takes the registers)
    const int MT = BITS == 0 ? std::min(pick_mt(a.M), 2) : pick_mt(a.M);
    const int64_t mgroups = cdiv<int64_t>(a.M, MT);
    const int ssize = PP ? 0 : ST == kF32 ? 4 : 2;
    if constexpr (BITS == 0) {
        if (MT == 1) return launch_r<0, ST, 1>(a, pick_shape_resident<0, ST, 1, false>(a, ssize, sm_count, mgroups, 2),
                                               pdl, stream);
        return launch_r<0, ST, 2>(a, pick_shape_resident<0, ST, 2, false>(a, ssize, sm_count, mgroups, 2), pdl,
                                  stream);
    } else {
        switch (MT) {
            case 1:
                return launch_r<BITS, ST, 1, PP>(a, pick_shape_resident<BITS, ST, 1, PP>(a, ssize, sm_count, mgroups, 0),
                                                 pdl, stream);
            case 2:
                return launch_r<BITS, ST, 2, PP>(a, pick_shape_resident<BITS, ST, 2, PP>(a, ssize, sm_count, mgroups, 0),
                                                 pdl, stream);
            default:
                return launch_r<BITS, ST, 4, PP>(a, pick_shape_resident<BITS, ST, 4, PP>(a, ssize, sm_count, mgroups, 0),
                                                 pdl, stream);
        }
    }
}

}  // namespace

}  // namespace mnb
