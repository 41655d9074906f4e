// common.cuh -- device helpers shared by the sm_103a kernels: dtype access,
// mbarrier / bulk-copy / programmatic-dependent-launch wrappers (inline PTX),
// the packed f32x2 FMA, and the device error word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mnb.h"

namespace mnb {

constexpr int kF32 = MNB_F32, kF16 = MNB_F16, kBF16 = MNB_BF16;

// Device error word: 0 = no error, otherwise an mnb_status value, set by the
// first kernel of this translation unit that hits an error.  Every translation
// unit has its own word (no relocatable device code is needed);
// mnb_get_last_device_error collects and clears them through the per-unit host
// accessors declared in kernels.h.
static __device__ unsigned int g_device_error = 0;

__device__ __forceinline__ void record_error(unsigned int code) { atomicCAS(&g_device_error, 0u, code); }

// Host: read and clear this translation unit's error word (synchronous copies).
static inline cudaError_t take_unit_error(unsigned int* out) {
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof v);
    if (e == cudaSuccess && v != 0) e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero);
    *out = v;
    return e;
}

// ---------------------------------------------------------------- dtypes

template <int DT> struct DType;
template <> struct DType<kF32> { using T = float; };
template <> struct DType<kF16> { using T = __half; };
template <> struct DType<kBF16> { using T = __nv_bfloat16; };

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// Load element i of a runtime-typed array as float (exact widening).
__device__ __forceinline__ float load_as_f32(const void* p, int dtype, int64_t i) {
    if (dtype == kF32) return static_cast<const float*>(p)[i];
    if (dtype == kF16) return __half2float(static_cast<const __half*>(p)[i]);
    return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
}

// Store float x as element i of a runtime-typed array, round-to-nearest-even.
__device__ __forceinline__ void store_from_f32(void* p, int dtype, int64_t i, float x) {
    if (dtype == kF32)
        static_cast<float*>(p)[i] = x;
    else if (dtype == kF16)
        static_cast<__half*>(p)[i] = __float2half_rn(x);
    else
        static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(x);
}

// ------------------------------------------------------------ f32x2 math

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// ------------------------------------------------------------- mbarrier

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy (bulk copies, tcgen05).
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Gives up
// after ~kWaitLimit polls (each try_wait suspends for a hardware-chosen time
// slice), records MNB_ERR_TIMEOUT and returns false.
constexpr uint32_t kWaitLimit = 1u << 24;

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    for (uint32_t i = 0; i < kWaitLimit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    record_error(MNB_ERR_TIMEOUT);
    return false;
}

// ------------------------------------------------------------ bulk copies

// Global -> shared bulk copy (TMA, non-tensor); dst/src 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Hint: bring [src, src+bytes) into L2 (16-byte aligned, bytes % 16 == 0).  A
// prefetch only warms L2, which is coherent, so it may run before the grid
// dependency wait.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ------------------------------------------- programmatic dependent launch

// Wait until the preceding kernel in the stream has completed and its memory
// is visible (no-op when launched without programmatic serialisation).
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allow the next kernel in the stream to start its prologue.
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

// ------------------------------------------------------------- misc

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <typename T>
__host__ __device__ constexpr T cdiv(T a, T b) {
    return (a + b - 1) / b;
}

}  // namespace mnb
