// route.cu -- MoE routing (softmax + canonical top-k), the expert-sorted
// permutation of routed pairs, and the raw-code unpack export.
//
// Routing semantics follow "feat(qwen4): component kernels extracted from the
// brick PRs" (fp32 softmax, canonical top-k, optional renormalisation of the
// selected probabilities) and the QMoE routing step of "INT3 QMoE CUDA
// correctness baseline and Qwen experimental results".
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "route_core.cuh"

namespace mnb {

namespace {

// ------------------------------------------------------------------ unpack

// One thread per code: code k of a row is stream bits bits*k .. +bits-1 of the
// row's bytes, least significant bit first.
__global__ void unpack_kernel(const uint8_t* __restrict__ packed, int64_t rows, int64_t K, int bits,
                              int64_t row_bytes, uint8_t* __restrict__ codes) {
    const int64_t total = rows * K;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t n = i / K, k = i - n * K;
        const uint8_t* row = packed + n * row_bytes;
        const int64_t bit = k * bits;
        const int64_t byte = bit >> 3;
        const int sh = static_cast<int>(bit & 7);
        uint32_t v = row[byte];
        if (sh + bits > 8) v |= static_cast<uint32_t>(row[byte + 1]) << 8;
        codes[i] = static_cast<uint8_t>((v >> sh) & ((1u << bits) - 1u));
    }
}

// Output byte b of a packed row holds stream bits 8b .. 8b+7, i.e. parts of the
// codes k with bits*k in [8b - bits + 1, 8b + 7]; codes past K (the padding of a
// partial last block) contribute zeros, so the padding is canonical.
__global__ void pack_kernel(const uint8_t* __restrict__ codes, int64_t rows, int64_t K, int bits,
                            int64_t row_bytes, uint8_t* __restrict__ packed) {
    const int64_t total = rows * row_bytes;
    const uint32_t mask = (1u << bits) - 1u;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t n = i / row_bytes, b = i - n * row_bytes;
        const int64_t k_lo = (8 * b) / bits, k_hi = min((8 * b + 7) / bits, K - 1);
        uint32_t out = 0;
        for (int64_t k = k_lo; k <= k_hi; ++k) {
            const uint32_t q = codes[n * K + k] & mask;
            const int64_t off = k * bits - 8 * b;  // the code's first bit relative to the byte
            out |= off >= 0 ? (q << off) : (q >> -off);
        }
        packed[i] = static_cast<uint8_t>(out & 0xFFu);
    }
}

// ----------------------------------------------------------------- routing

// One warp per token (see route_core.cuh).
__global__ void route_kernel(const void* __restrict__ logits, int ldt, int64_t T, int E, int k, int normalize,
                             int32_t* __restrict__ idx, float* __restrict__ wout, const void* agg, int adt) {
    const int64_t t = blockIdx.x * int64_t(blockDim.x >> 5) + (threadIdx.x >> 5);
    grid_dependency_wait();
    grid_launch_dependents();
    if (t >= T) return;
    const int esz = ldt == kF32 ? 4 : 2, asz = adt == kF32 ? 4 : 2;
    warp_route(static_cast<const char*>(logits) + t * E * esz, ldt, E, k, normalize, idx + t * k, wout + t * k, 1,
               agg ? static_cast<const char*>(agg) + t * E * asz : nullptr, adt);
}

// ------------------------------------------------------------- permutation

// One CTA of 1024 threads.  Warp w owns the contiguous pair range
// [w*seg, (w+1)*seg).  Pass 1 counts pairs per (warp, expert); a scan gives
// every (warp, expert) its first output slot; pass 2 walks the same range in
// order, 32 pairs at a time, ranking equal experts with match_any so that the
// order inside an expert is the pair order (stable).
constexpr int kPermThreads = 1024;
constexpr int kPermWarps = kPermThreads / 32;

// With `mtiles` set it also writes the grouped tensor-core plan's m-tiles
// {expert, first sorted position, rows, 0} of <= tile_m rows per expert and
// their count (one launch in place of the count / scan / scatter / m-tile
// kernels, for the pair counts where one CTA is the faster plan).
__global__ void __launch_bounds__(kPermThreads) permute_kernel(const int32_t* __restrict__ idx, int64_t P,
                                                               int E, int32_t* __restrict__ counts,
                                                               int32_t* __restrict__ offsets,
                                                               int32_t* __restrict__ perm,
                                                               int32_t* __restrict__ inv_perm,
                                                               int4* __restrict__ mtiles = nullptr,
                                                               int* __restrict__ n_mtiles = nullptr,
                                                               int tile_m = 0) {
    extern __shared__ int32_t cnt[];  // [kPermWarps][E], then tot[E+1]
    int32_t* tot = cnt + kPermWarps * E;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    grid_dependency_wait();
    grid_launch_dependents();
    for (int i = tid; i < kPermWarps * E; i += kPermThreads) cnt[i] = 0;
    __syncthreads();
    const int64_t seg = (P + kPermWarps - 1) / kPermWarps;
    const int64_t p0 = warp * seg, p1 = (P < p0 + seg) ? P : p0 + seg;
    const uint32_t lt = (1u << lane) - 1u;
    int32_t* mycnt = cnt + warp * E;
    for (int64_t base = p0; base < p1; base += 32) {
        const int64_t p = base + lane;
        const bool valid = p < p1;
        const int e = valid ? idx[p] : -1 - lane;
        const uint32_t same = __match_any_sync(0xffffffffu, e);
        if (valid && (same & lt) == 0) mycnt[e] += __popc(same);
        __syncwarp();
    }
    __syncthreads();
    // per-expert totals and the exclusive scan over experts (E <= 1024, one thread each)
    int32_t my_total = 0;
    if (tid < E)
        for (int w = 0; w < kPermWarps; ++w) my_total += cnt[w * E + tid];
    // block-wide exclusive scan of my_total over tid < E
    __shared__ int32_t warp_sums[kPermWarps];
    int32_t x = (tid < E) ? my_total : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int32_t s = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        warp_sums[lane] = s;  // inclusive
    }
    __syncthreads();
    const int32_t incl = x + (warp > 0 ? warp_sums[warp - 1] : 0);
    if (tid < E) {
        const int32_t excl = incl - my_total;
        tot[tid] = excl;
        counts[tid] = my_total;
        offsets[tid] = excl;
        if (tid == E - 1) offsets[E] = incl;
        // first slot of each warp's pairs of expert tid, in warp order
        int32_t run = excl;
        for (int w = 0; w < kPermWarps; ++w) {
            const int32_t c = cnt[w * E + tid];
            cnt[w * E + tid] = run;
            run += c;
        }
    }
    __syncthreads();
    for (int64_t base = p0; base < p1; base += 32) {
        const int64_t p = base + lane;
        const bool valid = p < p1;
        const int e = valid ? idx[p] : -1 - lane;
        const uint32_t same = __match_any_sync(0xffffffffu, e);
        int32_t slot = 0;
        if (valid) slot = mycnt[e] + __popc(same & lt);
        __syncwarp();
        if (valid && (same & lt) == 0) mycnt[e] += __popc(same);
        __syncwarp();
        if (valid) {
            perm[slot] = static_cast<int32_t>(p);
            if (inv_perm) inv_perm[p] = slot;
        }
    }
    if (mtiles == nullptr) return;
    // m-tiles: expert tid's ceil(count / tile_m) tiles after the tiles of the
    // experts before it (the same block-wide scan as above)
    const int ntile = tid < E ? (my_total + tile_m - 1) / tile_m : 0;
    int32_t y = ntile;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t v = __shfl_up_sync(0xffffffffu, y, o);
        if (lane >= o) y += v;
    }
    __syncthreads();  // warp_sums is reused
    if (lane == 31) warp_sums[warp] = y;
    __syncthreads();
    if (warp == 0) {
        int32_t s = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t v = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += v;
        }
        warp_sums[lane] = s;
    }
    __syncthreads();
    const int32_t tincl = y + (warp > 0 ? warp_sums[warp - 1] : 0);
    if (tid < E) {
        const int32_t first = tincl - ntile, base = incl - my_total;
        for (int i = 0; i < ntile; ++i)
            mtiles[first + i] = make_int4(tid, base + i * tile_m, min(tile_m, my_total - i * tile_m), 0);
    }
    if (tid == kPermThreads - 1) *n_mtiles = warp_sums[kPermWarps - 1];
}

// ------------------------------------------- permutation over many CTAs
// Chunks of kPermChunk consecutive pairs.  perm_count_kernel: per-chunk expert
// histograms.  perm_scan_kernel: per expert, the exclusive scan over chunks
// (in place) and the totals; then the exclusive scan over experts (offsets).
// perm_scatter_kernel: each warp ranks its 32 pairs among equal experts, the
// warps of a chunk add the counts of earlier warps, and every pair lands at
// offsets[e] + (earlier chunks) + (earlier warps) + (earlier lanes): stable.
constexpr int kPermChunk = 256;

__global__ void __launch_bounds__(kPermChunk) perm_count_kernel(const int32_t* __restrict__ idx, int64_t P, int E,
                                                                int32_t* __restrict__ chunkc) {
    extern __shared__ int32_t hist[];
    grid_dependency_wait();
    grid_launch_dependents();
    for (int e = threadIdx.x; e < E; e += kPermChunk) hist[e] = 0;
    __syncthreads();
    const int64_t p = int64_t(blockIdx.x) * kPermChunk + threadIdx.x;
    if (p < P) atomicAdd(&hist[idx[p]], 1);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kPermChunk) chunkc[int64_t(blockIdx.x) * E + e] = hist[e];
}

// The chunks of each expert are split into `parts` consecutive ranges, one
// thread per (range, expert): a first pass sums the range, the ranges' sums
// are scanned in shared memory, and a second pass writes the exclusive
// prefixes.  Loads go out kScanBatch at a time, so a range costs a few memory
// round trips rather than one per chunk.
constexpr int kScanThreads = 1024, kScanBatch = 16;

__global__ void __launch_bounds__(kScanThreads) perm_scan_kernel(int32_t* __restrict__ chunkc, int n_chunks, int E,
                                                                 int32_t* __restrict__ counts,
                                                                 int32_t* __restrict__ offsets) {
    __shared__ int32_t part_sums[kScanThreads];  // [part][E]
    __shared__ int32_t warp_sums[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int parts = E <= kScanThreads ? kScanThreads / E : 1;
    const int e = tid % E, part = tid / E;
    const bool active = part < parts;
    const int per = (n_chunks + parts - 1) / parts;
    const int c0 = part * per, c1 = min(n_chunks, c0 + per);
    grid_dependency_wait();
    grid_launch_dependents();
    int32_t sum = 0;
    if (active) {
        for (int c = c0; c < c1; c += kScanBatch) {
            int32_t v[kScanBatch];
#pragma unroll
            for (int j = 0; j < kScanBatch; ++j) v[j] = c + j < c1 ? chunkc[int64_t(c + j) * E + e] : 0;
#pragma unroll
            for (int j = 0; j < kScanBatch; ++j) sum += v[j];
        }
        part_sums[part * E + e] = sum;
    }
    __syncthreads();
    int32_t run = 0, total = 0;
    if (active) {
        for (int q = 0; q < parts; ++q) {
            const int32_t ps = part_sums[q * E + e];
            run += q < part ? ps : 0;
            total += ps;
        }
        for (int c = c0; c < c1; c += kScanBatch) {
            int32_t v[kScanBatch];
#pragma unroll
            for (int j = 0; j < kScanBatch; ++j) v[j] = c + j < c1 ? chunkc[int64_t(c + j) * E + e] : 0;
#pragma unroll
            for (int j = 0; j < kScanBatch; ++j) {
                if (c + j < c1) chunkc[int64_t(c + j) * E + e] = run;
                run += v[j];
            }
        }
    }
    // exclusive scan of the expert totals (threads 0 .. E-1 hold expert tid's total)
    int32_t x = tid < E ? total : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int32_t v = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += y;
        }
        warp_sums[lane] = v;
    }
    __syncthreads();
    const int32_t incl = x + (warp > 0 ? warp_sums[warp - 1] : 0);
    if (tid < E) {
        counts[tid] = total;
        offsets[tid] = incl - total;
        if (tid == E - 1) offsets[E] = incl;
    }
}

__global__ void __launch_bounds__(kPermChunk) perm_scatter_kernel(const int32_t* __restrict__ idx, int64_t P, int E,
                                                                  const int32_t* __restrict__ chunkc,
                                                                  const int32_t* __restrict__ offsets,
                                                                  int32_t* __restrict__ perm,
                                                                  int32_t* __restrict__ inv_perm) {
    constexpr int kWarps = kPermChunk / 32;
    extern __shared__ int32_t whist[];  // [kWarps][E]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    grid_dependency_wait();
    grid_launch_dependents();
    for (int i = tid; i < kWarps * E; i += kPermChunk) whist[i] = 0;
    __syncthreads();
    const int64_t p = int64_t(blockIdx.x) * kPermChunk + tid;
    const int e = p < P ? idx[p] : -1 - lane;
    const uint32_t same = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(same & ((1u << lane) - 1u));
    if (e >= 0 && rank == 0) whist[warp * E + e] = __popc(same);
    __syncthreads();
    for (int x = tid; x < E; x += kPermChunk) {  // counts of earlier warps, per expert
        int32_t run = 0;
        for (int w = 0; w < kWarps; ++w) {
            const int32_t v = whist[w * E + x];
            whist[w * E + x] = run;
            run += v;
        }
    }
    __syncthreads();
    if (e >= 0) {
        const int32_t slot = offsets[e] + chunkc[int64_t(blockIdx.x) * E + e] + whist[warp * E + e] + rank;
        perm[slot] = static_cast<int32_t>(p);
        if (inv_perm) inv_perm[p] = slot;
    }
}

}  // namespace

int64_t permute_chunks(int64_t P) { return (P + kPermChunk - 1) / kPermChunk; }

cudaError_t launch_permute_chunked(const int32_t* idx, int64_t T, int k, int64_t E, int32_t* chunkc, int32_t* counts,
                                   int32_t* offsets, int32_t* perm, int32_t* inv_perm, cudaStream_t stream, bool pdl) {
    const int64_t P = T * k;
    const int64_t n = permute_chunks(P);
    const size_t hist = size_t(E) * sizeof(int32_t);
    cudaError_t e;
    if ((e = set_max_carveout(perm_count_kernel)) != cudaSuccess || (e = set_max_carveout(perm_scan_kernel)) != cudaSuccess ||
        (e = set_max_carveout(perm_scatter_kernel)) != cudaSuccess)
        return e;
    if ((e = launch_ex(perm_count_kernel, dim3(static_cast<unsigned>(n)), dim3(kPermChunk), hist, stream, pdl, idx, P,
                       static_cast<int>(E), chunkc)) != cudaSuccess)
        return e;
    if ((e = launch_ex(perm_scan_kernel, dim3(1), dim3(kScanThreads), 0, stream, pdl, chunkc, static_cast<int>(n),
                       static_cast<int>(E), counts, offsets)) != cudaSuccess)
        return e;
    const size_t whist = size_t(kPermChunk / 32) * E * sizeof(int32_t);
    return launch_ex(perm_scatter_kernel, dim3(static_cast<unsigned>(n)), dim3(kPermChunk), whist, stream, pdl, idx, P,
                     static_cast<int>(E), static_cast<const int32_t*>(chunkc), static_cast<const int32_t*>(offsets),
                     perm, inv_perm);
}

cudaError_t launch_unpack_codes(const uint8_t* packed, int64_t rows, int64_t K, int bits, int bs,
                                uint8_t* codes, cudaStream_t stream) {
    const int64_t nb = cdiv<int64_t>(K, bs);
    const int64_t row_bytes = nb * bs * bits / 8;
    const int64_t total = rows * K;
    const int threads = 256;
    const int64_t blocks = std::min<int64_t>(cdiv<int64_t>(total, threads), 65535 * 16);
    const cudaError_t e = set_max_carveout(unpack_kernel);
    if (e != cudaSuccess) return e;
    unpack_kernel<<<static_cast<unsigned>(std::max<int64_t>(blocks, 1)), threads, 0, stream>>>(
        packed, rows, K, bits, row_bytes, codes);
    return cudaGetLastError();
}

cudaError_t launch_pack_codes(const uint8_t* codes, int64_t rows, int64_t K, int bits, int bs, uint8_t* packed,
                              cudaStream_t stream) {
    const int64_t nb = cdiv<int64_t>(K, bs);
    const int64_t row_bytes = nb * bs * bits / 8;
    const int threads = 256;
    const int64_t blocks = std::min<int64_t>(cdiv<int64_t>(rows * row_bytes, threads), 65535 * 16);
    const cudaError_t e = set_max_carveout(pack_kernel);
    if (e != cudaSuccess) return e;
    pack_kernel<<<static_cast<unsigned>(std::max<int64_t>(blocks, 1)), threads, 0, stream>>>(codes, rows, K, bits,
                                                                                           row_bytes, packed);
    return cudaGetLastError();
}

cudaError_t launch_route(const void* logits, int ldt, int64_t T, int64_t E, int k, int normalize, int32_t* idx,
                         float* w, const void* agg, int adt, cudaStream_t stream, bool pdl) {
    const int warps = 8;
    const int64_t blocks = cdiv<int64_t>(T, warps);
    const cudaError_t e = set_max_carveout(route_kernel);
    if (e != cudaSuccess) return e;
    return launch_ex(route_kernel, dim3(static_cast<unsigned>(blocks)), dim3(warps * 32), 0, stream, pdl, logits, ldt, T,
                     static_cast<int>(E), k, normalize, idx, w, agg, adt);
}

cudaError_t launch_permute(const int32_t* idx, int64_t T, int k, int64_t E, int32_t* counts, int32_t* offsets,
                           int32_t* perm, int32_t* inv_perm, cudaStream_t stream, int4* mtiles, int* n_mtiles,
                           int tile_m, bool pdl) {
    const size_t smem = (size_t(kPermWarps) * E + E + 1) * sizeof(int32_t);
    cudaError_t e = set_kernel_smem(permute_kernel, static_cast<int64_t>(smem));
    if (e != cudaSuccess) return e;
    return launch_ex(permute_kernel, dim3(1), dim3(kPermThreads), smem, stream, pdl, idx, T * k, static_cast<int>(E),
                     counts, offsets, perm, inv_perm, mtiles, n_mtiles, tile_m);
}

}  // namespace mnb
