// route_core.cuh -- one warp (or one CTA) routes one token: fp32 softmax over E router
// logits, the k largest logits (ties to the lower expert index), weights
// renormalised over the selected k or left as softmax probabilities
// ("feat(qwen4): component kernels extracted from the brick PRs": fp32 softmax,
// canonical top-k, optional renormalisation; "INT3 QMoE CUDA correctness
// baseline and Qwen experimental results": routing of the QMoE layer).
#pragma once

#include "common.cuh"

namespace mnb {

constexpr int kMaxExpertsPerLane = 32;  // E <= 1024
constexpr int kNoExpert = 0x7fffffff;

// One warp, PL logits per lane (E <= 32 PL): expert e lives in slot e / 32 of
// lane e % 32, so the argmax scans only the PL slots a lane can hold.
// Logit e of a router row stored in dtype dt (fp32, fp16 or bf16; widened exactly).
__device__ __forceinline__ float logit_at(const void* row, int dt, int e) { return load_as_f32(row, dt, e); }

// With aggregation weights, slot j's combine weight is agg[idx[j]] (dtype adt)
// instead of the routing probability; called by the lane that owns slot j.
__device__ __forceinline__ float agg_or(const void* agg, int adt, int e, float p) {
    return agg ? load_as_f32(agg, adt, e) : p;
}

template <int PL, typename IdxT, typename WT>
__device__ __forceinline__ void warp_route_pl(const void* __restrict__ row, int ldt, int E, int k, int normalize,
                                              IdxT* idx, WT* w, int stride, const void* agg = nullptr, int adt = 0) {
    const int lane = threadIdx.x & 31;
    const int per_lane = (E + 31) >> 5;
    float v[PL];
    uint32_t taken = 0;
    float lmax = -INFINITY;
#pragma unroll
    for (int i = 0; i < PL; ++i) {
        const int e = i * 32 + lane;
        const bool ok = i < per_lane && e < E;
        v[i] = ok ? logit_at(row, ldt, e) : -INFINITY;
        if (ok) lmax = fmaxf(lmax, v[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));

    float sel_sum = 0.f;
    int my_e = 0;
    float my_p = 0.f;
    for (int j = 0; j < k; ++j) {
        float bv = 0.f;
        int be = kNoExpert;
#pragma unroll
        for (int i = 0; i < PL; ++i) {
            const int e = i * 32 + lane;
            if (i < per_lane && e < E && !((taken >> i) & 1u)) {
                if (be == kNoExpert || v[i] > bv) { bv = v[i]; be = e; }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oe = __shfl_xor_sync(0xffffffffu, be, o);
            const bool better = (oe != kNoExpert) && (be == kNoExpert || ov > bv || (ov == bv && oe < be));
            if (better) { bv = ov; be = oe; }
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        const float p = expf(bv - lmax);
        sel_sum += p;
        if (j < 32) {  // lane j keeps slot j until the end
            if (lane == j) {
                my_e = be;
                my_p = p;
            }
        } else if (lane == 0) {  // k > 32: park the raw weight in the output
            idx[j * stride] = static_cast<IdxT>(be);
            w[j * stride] = static_cast<WT>(agg ? agg_or(agg, adt, be, p) : p);
        }
    }
    float denom = sel_sum;
    if (!normalize) {
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < PL; ++i) {
            const int e = i * 32 + lane;
            if (i < per_lane && e < E) s += expf(v[i] - lmax);
        }
        denom = warp_sum(s);
    }
    if (lane < k) {
        idx[lane * stride] = static_cast<IdxT>(my_e);
        w[lane * stride] = static_cast<WT>(agg ? agg_or(agg, adt, my_e, 0.f) : my_p / denom);
    }
    __syncwarp();
    if (k > 32 && lane == 0 && !agg)
        for (int j = 32; j < k; ++j) w[j * stride] = static_cast<WT>(static_cast<float>(w[j * stride]) / denom);
    __syncwarp();
}

// Every lane of the warp must call this.  Slot j's expert and weight are
// written to idx[j * stride] / w[j * stride] (any address space) by lane j
// (slots past 32 by lane 0).
// The scan width is fixed at compile time from E, so a 128-expert router pays
// for four logits per lane, not for the 1024-expert maximum.
template <typename IdxT, typename WT>
__device__ __forceinline__ void warp_route(const void* __restrict__ row, int ldt, int E, int k, int normalize,
                                           IdxT* idx, WT* w, int stride, const void* agg = nullptr, int adt = 0) {
    if (E <= 32) return warp_route_pl<1>(row, ldt, E, k, normalize, idx, w, stride, agg, adt);
    if (E <= 64) return warp_route_pl<2>(row, ldt, E, k, normalize, idx, w, stride, agg, adt);
    if (E <= 128) return warp_route_pl<4>(row, ldt, E, k, normalize, idx, w, stride, agg, adt);
    if (E <= 256) return warp_route_pl<8>(row, ldt, E, k, normalize, idx, w, stride, agg, adt);
    if (E <= 512) return warp_route_pl<16>(row, ldt, E, k, normalize, idx, w, stride, agg, adt);
    return warp_route_pl<kMaxExpertsPerLane>(row, ldt, E, k, normalize, idx, w, stride, agg, adt);
}

// Routing of one token by a whole CTA (blockDim.x >= E): every thread ranks
// one logit against all E (the number of logits that beat it, ties going to
// the lower expert index, NaN taken as -inf), the ranks below k name the
// selected experts in order, and one lane forms the weights exactly as
// warp_route does (same sums in the same order).  All threads must call this;
// it ends with a block barrier.  s_logit is shared scratch of E floats.
constexpr int kBlockRouteMaxE = 256;

template <typename WT>
__device__ __forceinline__ void block_route(const void* __restrict__ row, int ldt, int E, int k, int normalize,
                                            int* idx, WT* w, float* s_logit, const void* agg = nullptr, int adt = 0) {
    const int tid = threadIdx.x, lane = tid & 31;
    if (tid < E) {
        const float x = logit_at(row, ldt, tid);
        s_logit[tid] = x != x ? -INFINITY : x;
    }
    __syncthreads();
    if (tid < E) {
        const float v = s_logit[tid];
        int r0 = 0, r1 = 0;
        int j = 0;
#pragma unroll 4
        for (; j + 1 < tid; j += 2) {  // lower indices beat v on ties
            const float u0 = s_logit[j], u1 = s_logit[j + 1];
            r0 += u0 >= v;
            r1 += u1 >= v;
        }
        if (j < tid) r0 += s_logit[j] >= v;
#pragma unroll 4
        for (j = tid + 1; j + 1 < E; j += 2) {  // higher indices only when strictly greater
            const float u0 = s_logit[j], u1 = s_logit[j + 1];
            r0 += u0 > v;
            r1 += u1 > v;
        }
        if (j < E) r0 += s_logit[j] > v;
        const int r = r0 + r1;
        if (r < k) idx[r] = tid;
    }
    __syncthreads();
    if (tid < 32) {
        const float lmax = s_logit[idx[0]];
        float denom = 0.f;
        if (!normalize) {
            float sum = 0.f;
#pragma unroll 1
            for (int e = lane; e < E; e += 32) sum += expf(s_logit[e] - lmax);
            denom = warp_sum(sum);
        }
        if (lane == 0) {
            float sel = 0.f;
#pragma unroll 1
            for (int j = 0; j < k; ++j) {
                const float p = expf(s_logit[idx[j]] - lmax);
                sel += p;
                w[j] = static_cast<WT>(p);
            }
            if (normalize) denom = sel;
#pragma unroll 1
            for (int j = 0; j < k; ++j)
                w[j] = static_cast<WT>(agg ? agg_or(agg, adt, idx[j], 0.f) : static_cast<float>(w[j]) / denom);
        }
    }
    __syncthreads();
}

// block_route with the ranking split over `tpl` adjacent lanes per logit
// (tpl = the largest power of two <= min(8, blockDim.x / E)) and the k
// selected probabilities formed by k lanes at once; the k selected
// probabilities are summed by a fixed shuffle tree.  Same selection (ties to
// the lower index, NaN as -inf) and the same weights up to the order of that
// sum.  Needs blockDim.x >= E, a multiple of 32; all threads must call it; it
// ends with a block barrier.  s_logit is shared scratch of E floats.
template <typename WT>
__device__ __forceinline__ void block_route_fast(const void* __restrict__ row, int ldt, int E, int k, int normalize,
                                                 int* idx, WT* w, float* s_logit, const void* agg = nullptr,
                                                 int adt = 0) {
    const int tid = threadIdx.x, lane = tid & 31;
    int tpl = 1;
    while (tpl < 8 && E * tpl * 2 <= int(blockDim.x)) tpl *= 2;
    if (tid < E) {
        const float x = logit_at(row, ldt, tid);
        s_logit[tid] = x != x ? -INFINITY : x;
    }
    __syncthreads();
    const int e = tid / tpl, part = tid - e * tpl;
    if (e < E) {
        const float v = s_logit[e];
        int r = 0;
        for (int j = part; j < E; j += tpl) {  // lower indices beat v on ties, higher ones only when greater
            const float u = s_logit[j];
            r += j < e ? (u >= v) : (u > v);
        }
        for (int o = 1; o < tpl; o <<= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
        if (part == 0 && r < k) idx[r] = e;
    } else if (tpl > 1) {
        int r = 0;  // lanes past E still take part in the shuffles of their warp
        for (int o = 1; o < tpl; o <<= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    }
    __syncthreads();
    if (tid < 32) {
        const float lmax = s_logit[idx[0]];
        const float p = lane < k ? expf(s_logit[idx[lane]] - lmax) : 0.f;
        float denom;
        if (normalize) {
            denom = warp_sum(p);
        } else {
            float sum = 0.f;
#pragma unroll 1
            for (int x = lane; x < E; x += 32) sum += expf(s_logit[x] - lmax);
            denom = warp_sum(sum);
        }
        if (lane < k) w[lane] = static_cast<WT>(agg ? agg_or(agg, adt, idx[lane], 0.f) : p / denom);
    }
    __syncthreads();
}

}  // namespace mnb
