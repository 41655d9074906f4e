// route_core.cuh -- one warp routes one token: fp32 softmax over E router
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

// Every lane of the warp must call this.  Slot j's expert and weight are
// written to idx[j * stride] / w[j * stride] (any address space) by lane 0.
template <typename IdxT, typename WT>
__device__ __forceinline__ void warp_route(const float* __restrict__ row, int E, int k, int normalize, IdxT* idx,
                                           WT* w, int stride) {
    const int lane = threadIdx.x & 31;
    const int per_lane = (E + 31) >> 5;
    float v[kMaxExpertsPerLane];
    uint32_t taken = 0;
    float lmax = -INFINITY;
#pragma unroll
    for (int i = 0; i < kMaxExpertsPerLane; ++i) {
        const int e = i * 32 + lane;
        const bool ok = i < per_lane && e < E;
        v[i] = ok ? row[e] : -INFINITY;
        if (ok) lmax = fmaxf(lmax, v[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));

    float sel_sum = 0.f;
    for (int j = 0; j < k; ++j) {
        float bv = 0.f;
        int be = kNoExpert;
#pragma unroll
        for (int i = 0; i < kMaxExpertsPerLane; ++i) {
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
        if (lane == 0) {
            idx[j * stride] = static_cast<IdxT>(be);
            w[j * stride] = static_cast<WT>(p);
        }
    }
    float denom = sel_sum;
    if (!normalize) {
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < kMaxExpertsPerLane; ++i) {
            const int e = i * 32 + lane;
            if (i < per_lane && e < E) s += expf(v[i] - lmax);
        }
        denom = warp_sum(s);
    }
    __syncwarp();
    if (lane == 0)
        for (int j = 0; j < k; ++j) w[j * stride] = static_cast<WT>(static_cast<float>(w[j * stride]) / denom);
    __syncwarp();
}

}  // namespace mnb
