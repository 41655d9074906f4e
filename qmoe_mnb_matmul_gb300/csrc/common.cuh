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

// try_wait suspends the thread (instead of returning at once) until the phase
// completes or about kSuspendNs nanoseconds pass, so waiting warps do not
// take issue slots from working ones.
constexpr uint32_t kSuspendNs = 20000;

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "n"(kSuspendNs)
        : "memory");
    return ok != 0;
}

// (a & b) | c in one logic instruction.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait for the phase with the given parity to complete.  Gives up
// after about kWaitNs nanoseconds of wall time, records MNB_ERR_TIMEOUT and
// returns false.
constexpr uint64_t kWaitNs = 2000000000ull;

// The same wait with a limit of limit_ns nanoseconds.
__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) break;
    }
    record_error(MNB_ERR_TIMEOUT);
    return false;
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) { return mbar_wait_for(bar, parity, kWaitNs); }

// Warp-uniform bounded wait: lane 0 waits, every lane gets the same verdict.
__device__ __forceinline__ bool warp_wait_for(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait_for(bar, parity, limit_ns) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) { return warp_wait_for(bar, parity, kWaitNs); }

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
//
// Every kernel of this library calls this only after its own
// grid_dependency_wait (or not at all), and the first kernel of every call
// reads nothing before its wait (it may only warm L2, which is coherent).  A
// later kernel of the same call (QMoE decode FC2) may read the call's inputs
// in its prologue: the kernel that released it had already waited, so
// everything ahead of the call has completed.
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

// ------------------------------------------------------------- misc

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Sums each of N per-lane values over the warp (N a power of two, <= 32) and
// returns, in every lane, the total of value transpose_row<N>(lane).  At each
// of the first log2(N) steps a lane hands half of the values it still holds
// to its partner and keeps the other half, so the warp needs N - 1 + log2(32/N)
// shuffles instead of 5 N.  The order of the additions is fixed.
template <int N>
__device__ __forceinline__ float warp_sum_transpose(float (&v)[N]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int n = N, off = 16; n > 1; n >>= 1, off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float give = upper ? v[i] : v[i + n / 2];
            const float keep = upper ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, give, off);
        }
    }
    float s = v[0];
#pragma unroll
    for (int off = 16 / N; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    return s;
}

// The value whose total warp_sum_transpose<N> leaves in this lane; lanes whose
// low log2(32/N) bits are zero hold one distinct value each.
template <int N>
__device__ __forceinline__ int transpose_row(int lane) {
    int row = 0;
#pragma unroll
    for (int n = N, off = 16; n > 1; n >>= 1, off >>= 1)
        if (lane & off) row += n / 2;
    return row;
}

template <typename T>
__host__ __device__ constexpr T cdiv(T a, T b) {
    return (a + b - 1) / b;
}

// Every kernel of the library runs with the largest shared-memory carveout.
// When consecutive kernels on a stream prefer different carveouts, an SM must
// drain before it takes the next kernel's CTAs, which also cancels the early
// start of programmatic dependents: the 141-launch decode step ran 10 % slower
// with the carveouts the driver picked per kernel.
template <typename Kernel>
inline cudaError_t set_max_carveout(Kernel kern) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                static_cast<int>(cudaSharedmemCarveoutMaxShared));
}

// The kernel's dynamic shared memory and the common carveout.
template <typename Kernel>
inline cudaError_t set_kernel_smem(Kernel kern, int64_t dyn_bytes) {
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(dyn_bytes));
    return e != cudaSuccess ? e : set_max_carveout(kern);
}

}  // namespace mnb

namespace mnb {

// ------------------------------------------------------------- tcgen05 / TMA

// Tensor (tiled) TMA load of a 2-D box at coordinates {x (inner), y} into
// shared memory, completing on `bar` with the box's byte count.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// Four whole rows y0..y3 (any order, any rows) of a 2D tensor, columns x ..
// x + box width, stacked in shared memory like a 4-row tile.  The tensor map's
// box must be one row high; x * element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_gather4(void* dst, const void* tmap, int x, int y0, int y1, int y2, int y3,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
        "l"(tmap), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// Asynchronous global -> shared copies of 16 / 8 / 4 bytes (Ampere-style), with group completion.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// TMEM allocation (one full warp executes these).
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16 (bf16 or fp16 inputs, fp32 accumulate).
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane (base lane + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,"
        "%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major operand tile stored in 128-byte
// swizzled atoms of 8 rows x 128 bytes (the TMA SWIZZLE_128B layout): start
// address >> 4 in bits 0..13, leading-dimension byte offset (unused for this
// layout, 1) in 16..29, stride byte offset between 8-row atoms (1024 >> 4) in
// 32..45, descriptor version 1 in 46..47, layout type SWIZZLE_128B (2) in 61..63.
__device__ __forceinline__ uint64_t smem_desc_sw128(const void* tile) {
    const uint64_t addr = smem_u32(tile);
    return ((addr >> 4) & 0x3FFFull) | (1ull << 16) | (uint64_t(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator (bits 4..5 = 1), A and B
// format (bits 7..9, 10..12: 0 = fp16, 1 = bf16), both K-major (bits 15, 16 =
// 0), N >> 3 in bits 17..22, M >> 4 in bits 24..28.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool bf16) {
    return (1u << 4) | (uint32_t(bf16) << 7) | (uint32_t(bf16) << 10) | (uint32_t(N >> 3) << 17) |
           (uint32_t(M >> 4) << 24);
}

}  // namespace mnb
