// gemm_tc_impl.cuh -- weight-only matmul on the 5th-generation tensor cores
// (tcgen05, sm_103a) with the weights dequantised tile by tile in shared
// memory: the small-M / prefill MatMulNBits GEMM ("Qwen3 Missing-Kernel
// Implementation Plan", row K03: small-M and prefill GEMM on the same
// compressed weights, bounded workspace, partial blocks and output tails) and
// the grouped per-expert FC1 (+SwiGLU) and FC2 GEMMs of the QMoE prefill (the
// "selected-expert / tiled-dequantisation plus GEMM" prefill the QMoE CUDA
// page names as missing).
//
// Tiles are 128 weight rows x G*BN activation rows.  The MMA is "swap-AB":
// the dequantised weight tile is operand A (M = 128) and each of the G
// activation sub-tiles operand B (N = BN <= 256), so the fp32 accumulators in
// tensor memory hold Y^T (lane = weight row, column = activation row) and small
// M costs no padding on the weight side.  The kernel supports G = 2 (every
// dequantised weight K step feeding two MMAs, 512 accumulator columns), but
// the launcher always takes G = 1, whose two 256-column halves of tensor
// memory double-buffer consecutive tiles: with only two activation stages
// beside G = 2's tiles it measured slower.  One persistent CTA per SM walks
// the tiles.
//
// Warp roles (768 threads, 24 warps; warp w issues from SM sub-partition
// w % 4).  The three single-lane roles share sub-partition 1 with one epilogue
// warp and one dequant warp: the dequant warps' long ALU streams on the other
// three sub-partitions would otherwise take the issue slots that the MMA
// issuer needs every K step (measured: with them mixed in, issuing a K step's
// four MMAs and two commits took ~500 cycles).
//   warp 9      activation producer: TMA tiles [BN x 64] (128-byte swizzle); in
//               the grouped FC1 the routed tokens' rows were first copied
//               into expert-sorted order, so the same tile loads serve
//   warp 1      TMEM owner; one lane issues tcgen05.mma (K = 16, 4 per stage)
//   warp 5      packed-weight producer: per K step one TMA tile of the 128
//               rows' packed bytes [128 x 32 B] and one of their scales
//               [128 x 16 B] into an 8-slot ring (where the rows are 16-byte
//               aligned; otherwise each dequant thread copies its own row
//               with cp.async into the same slots)
//   16 warps    dequant (all the others but warp 21, which idles), four groups
//               of 4 warps taking every fourth K step: one thread per weight
//               row, both 32-code chunks of the K step; codes -> s (q - z) ->
//               fp16/bf16 -> swizzled 16-byte stores
//   warps 12-15 epilogue (TMEM lane quarter = warp % 4): tcgen05.ld of the
//               accumulators -> output dtype (FC1: SwiGLU of lane pairs) ->
//               masked stores
// The activation tiles and the dequantised weight tiles of the K steps sit in
// two separate shared rings: the activation ring is deep (its tiles come from
// L2 / HBM with the longest latency), the weight ring holds one slot per
// dequant group plus one.  A tcgen05.commit releases a slot of each when the MMAs that
// read it complete.  Packed rows come as tensor tiles rather than per-thread
// copies because a 32-lane copy of 32 scattered rows costs a shared-memory
// wavefront per lane.  Every wait is bounded.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "gemv_core.cuh"
#include "kernels.h"

namespace mnb {

namespace {

using namespace gemv;

constexpr int kBK = 64;     // K elements per stage: one 128-byte swizzle atom of 16-bit values
constexpr int kBW = 128;    // weight rows per tile (MMA M)
constexpr int kMmaWarp = 1;   // TMEM owner and MMA issuer
constexpr int kPackWarp = 5;  // TMA producer of packed rows and scales
constexpr int kActWarp = 9;   // TMA producer of activation tiles
constexpr int kEpilogueWarp0 = 12;  // warps 12..15
constexpr int kWarpsTC = 24;
// Warps with a role other than dequantisation (warp 21 idles).
constexpr uint32_t kNonDequantWarps = (1u << kMmaWarp) | (1u << kPackWarp) | (1u << kActWarp) |
                                      (0xFu << kEpilogueWarp0) | (1u << 21);
// Rank of warp w among the dequant warps, or -1.
__device__ __forceinline__ int dequant_rank(int w) {
    return ((kNonDequantWarps >> w) & 1u) ? -1 : w - __popc(kNonDequantWarps & ((1u << w) - 1u));
}
// Four groups of 4 dequantisation warps take every fourth K step: one thread
// per weight row makes all 64 codes of the row's K step, and each group has
// four MMA steps' time for its 128 x 64 weight slice.
constexpr int kDequantGroups = 4;
constexpr int kDequantWarps = 16 / kDequantGroups;            // warps per group
constexpr int kChunksPerThread = kDequantGroups == 4 ? 2 : 1;  // 32-code chunks of a row's K step per thread
// Dequantised-weight ring depth: at least one slot per group (a group's parity
// wait needs it), plus one so that a group may start its next K step one MMA
// step before the slot it last wrote has been read.
constexpr int kWeightSlots = kDequantGroups + 1;
// Packed ring: K step g of the CTA's sequence -> slot g % 8, so each group owns
// two slots and has its next K step in flight while it works on the current.
constexpr int kPackSlots = 2 * kDequantGroups;
constexpr int kPackRow = 32;  // bytes of a row's K step in a slot (INT3: a 16-byte-aligned 32-byte window)
constexpr int kSclRow = 16;   // bytes of a row's scale window in a slot
static_assert(kWarpsTC - __builtin_popcount(kNonDequantWarps) == kDequantGroups * kDequantWarps,
              "every dequant group needs its warps");
constexpr int kThreadsTC = kWarpsTC * 32;
constexpr int kMaxStagesTC = 8;

enum { kModeGemm = 0, kModeFc1 = 1 };

struct TcPlan {
    int64_t bars, act, w, pack, scl, total;
};

__host__ __device__ inline TcPlan tc_plan(int BN, int G, int stages, int stages_w, int bits) {
    TcPlan p;
    p.bars = 1024;                                           // barriers and the TMEM address
    p.act = int64_t(G) * BN * 128;                           // activations of one stage (G sub-tiles)
    p.w = int64_t(kBW) * 128;                                // dequantised weights of one stage
    p.pack = int64_t(kPackSlots) * kBW * kPackRow;  // [slot][row][32 bytes]
    p.scl = int64_t(kPackSlots) * kBW * kSclRow;    // [slot][row][16 bytes]
    p.total = p.bars + int64_t(stages) * p.act + int64_t(stages_w) * p.w + p.pack + p.scl;
    return p;
}

// Byte offset of 16-byte chunk c (k elements 8c .. 8c+7) of row r inside a
// 128-byte-swizzled tile: atoms of 8 rows x 128 bytes, chunk index XOR row % 8.
__device__ __forceinline__ uint32_t sw128(int r, int c) {
    return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

template <int ST>
__device__ __forceinline__ float scale_from_word(uint32_t word, int64_t idx) {
    if constexpr (ST == kF32) {
        return __uint_as_float(word);
    } else {
        const uint32_t h = (idx & 1) ? (word >> 16) : (word & 0xFFFFu);
        if constexpr (ST == kF16) return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
        return __uint_as_float(h << 16);
    }
}

template <int AT>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    if constexpr (AT == kBF16) {
        const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<const uint32_t*>(&v);
    } else {
        const __half2 v = __floats2half2_rn(a, b);
        return *reinterpret_cast<const uint32_t*>(&v);
    }
}

// The pair (a, b) rounded to the 16-bit type (REM false), or what that
// rounding left behind, a - round16(a), itself rounded to the 16-bit type
// (REM true; the difference is exact in fp32).
template <int AT, bool REM>
__device__ __forceinline__ uint32_t pack2_part(float2 v) {
    const uint32_t hi = pack2<AT>(v.x, v.y);
    if constexpr (!REM) {
        return hi;
    } else {
        float2 h;
        if constexpr (AT == kBF16) {
            h = make_float2(__uint_as_float(hi << 16), __uint_as_float(hi & 0xFFFF0000u));
        } else {
            h = __half22float2(*reinterpret_cast<const __half2*>(&hi));
        }
        return pack2<AT>(v.x - h.x, v.y - h.y);
    }
}

// Named barrier of the four epilogue warps (barrier 0 is __syncthreads).
__device__ __forceinline__ void epilogue_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Ring position of the i-th K step of this CTA: stage index and how many
// times the ring has wrapped, advanced without divisions.
struct RingPos {
    int stage = 0;
    uint32_t round = 0;
    __device__ __forceinline__ void next(int S) {
        if (++stage == S) { stage = 0; ++round; }
    }
};

// Tile t -> (expert, first activation row, rows, first weight row, split of K
// and its first K step).
struct Tile {
    int e, s0, cnt, n0, split, ks0;
};

__device__ __forceinline__ Tile tile_of(const TcArgs& a, int t, int BN) {
    Tile x;
    if (a.mtiles) {
        const int j = t / a.tiles_n;
        const int4 mt = a.mtiles[j];
        x.e = mt.x;
        x.s0 = mt.y;
        x.cnt = mt.z;
        x.n0 = (t - j * a.tiles_n) * kBW;
        x.split = 0;
        x.ks0 = 0;
    } else {
        x.split = t % a.splits;  // splits of one output tile run on neighbouring CTAs
        t /= a.splits;
        x.ks0 = x.split * a.k_steps;
        const int nt = t / a.tiles_m;
        const int mtile = t - nt * a.tiles_m;
        x.e = 0;
        x.s0 = mtile * BN;
        x.cnt = static_cast<int>(a.M - x.s0 < BN ? a.M - x.s0 : int64_t(BN));
        x.n0 = nt * kBW;
    }
    return x;
}

// Accumulator slot s (columns s*BN ..) of sub-tile g of the tl-th tile of this
// CTA, and how many earlier tiles used that slot.
template <int G>
__device__ __forceinline__ int acc_slot(int tl, int g) { return G == 1 ? (tl & 1) : g; }
template <int G>
__device__ __forceinline__ int acc_uses(int tl) { return G == 1 ? (tl >> 1) : tl; }

template <int BITS, int ST, int AT, int BN, int G, int MODE>
__global__ void __launch_bounds__(kThreadsTC, 1) gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_a,
                                                                const __grid_constant__ CUtensorMap tmap_w,
                                                                const __grid_constant__ CUtensorMap tmap_s,
                                                                const __grid_constant__ TcArgs a) {
    static_assert(G == 1 || G == 2, "one or two activation sub-tiles per tile");
    constexpr int UN = G * BN;  // activation rows per tile
    extern __shared__ __align__(1024) uint8_t smem[];
    const int S = a.stages, SW = a.stages_w;
    const TcPlan plan = tc_plan(BN, G, S, SW, BITS);
    uint64_t* full_a = reinterpret_cast<uint64_t*>(smem);
    // (full_a + kMaxStagesTC: unused; the activation stages are released
    // through empty_w, the barrier of the K step that last read them)
    uint64_t* full_w = full_a + 2 * kMaxStagesTC;
    uint64_t* empty_w = full_a + 3 * kMaxStagesTC;
    uint64_t* acc_full = full_a + 4 * kMaxStagesTC;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* pfull = full_a + 5 * kMaxStagesTC;   // packed slot loaded (TMA)
    uint64_t* pempty = full_a + 6 * kMaxStagesTC;  // packed slot read by its group's 4 warps
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(full_a + 7 * kMaxStagesTC);
    volatile int* epi_fail = reinterpret_cast<volatile int*>(tmem_holder + 1);  // the epilogue's wait gave up
    uint8_t* act = smem + plan.bars;
    uint8_t* wt = act + S * plan.act;
    uint8_t* pack = wt + SW * plan.w;
    uint8_t* scl = pack + plan.pack;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (smem_u32(smem) & 1023) {  // the swizzled tiles need 1024-byte alignment
        if (tid == 0) record_error(MNB_ERR_UNSUPPORTED);
        return;
    }
    const int ksteps = a.k_steps;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&full_a[s], 1);
        for (int s = 0; s < SW; ++s) {
            mbar_init(&full_w[s], kDequantWarps);
            mbar_init(&empty_w[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4);
        }
        for (int s = 0; s < kPackSlots; ++s) {
            mbar_init(&pfull[s], 1);
            mbar_init(&pempty[s], kDequantWarps);
        }
        *epi_fail = 0;
        fence_barrier_init();
        prefetch_tmap(&tmap_a);
        if (a.w_tma) prefetch_tmap(&tmap_w);
        if (a.s_tma) prefetch_tmap(&tmap_s);
    }
    if (warp == kMmaWarp) tmem_alloc(tmem_holder, a.tmem_cols);
    grid_dependency_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const int n_tiles = a.mtiles ? *a.n_mtiles * a.tiles_n : a.tiles_n * a.tiles_m * a.splits;
    bool failed = false;

    const int dq_rank = dequant_rank(warp);
    if (warp == kActWarp) {
        // ------------------------------------------------- activation producer
        // TMA tiles of the activation rows (FC1: the routed tokens' rows, already
        // copied into expert-sorted order), G sub-tiles of BN rows per K step.
        // A stage is free again once the MMAs of the K step that last used it
        // have completed: the one commit per K step goes to the weight ring's
        // barrier of that step (`done` walks the weight ring S steps behind).
        // With S <= SW that barrier cannot have moved a phase past the step.
        if (lane == 0) {
            RingPos rp, done;
            for (int t = blockIdx.x; t < n_tiles && !failed; t += gridDim.x) {
                const Tile x = tile_of(a, t, UN);
                for (int ks = 0; ks < ksteps; ++ks, rp.next(S)) {
                    if (rp.round) {
                        if (!mbar_wait(&empty_w[done.stage], done.round & 1)) { failed = true; break; }
                        done.next(SW);
                    }
                    mbar_arrive_expect_tx(&full_a[rp.stage], UN * 128);
#pragma unroll
                    for (int g = 0; g < G; ++g)  // rows past the matrix read as zeros
                        tma_load_2d(act + rp.stage * plan.act + g * BN * 128, &tmap_a, (x.ks0 + ks) * kBK,
                                    x.s0 + g * BN, &full_a[rp.stage]);
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // --------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(kBW, BN, AT == kBF16);
            RingPos rp, rw;
            int tl = 0;
            for (int t = blockIdx.x; t < n_tiles && !failed; t += gridDim.x, ++tl) {
                const int uses = acc_uses<G>(tl);
                for (int ks = 0; ks < ksteps && !failed; ++ks, rp.next(S), rw.next(SW)) {
                    if (!mbar_wait(&full_a[rp.stage], rp.round & 1) || !mbar_wait(&full_w[rw.stage], rw.round & 1)) {
                        failed = true;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t da = smem_desc_sw128(wt + rw.stage * plan.w);
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const int slot = acc_slot<G>(tl, g);
                        if (ks == 0 && uses > 0) {  // the epilogue has drained this slot's previous tile
                            if (!mbar_wait(&acc_empty[slot], (uses - 1) & 1)) { failed = true; break; }
                            tc_fence_after();
                        }
                        const uint32_t d = tmem + slot * BN;
                        const uint64_t db = smem_desc_sw128(act + rp.stage * plan.act + g * BN * 128);
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk)
                            tc_mma_f16(d, da + 2 * kk, db + 2 * kk, idesc, (ks | kk) != 0);
                    }
                    if (failed) break;
                    tc_commit(&empty_w[rw.stage]);  // frees the step's weight slot and activation stage
                }
                if (failed) break;
#pragma unroll
                for (int g = 0; g < G; ++g) tc_commit(&acc_full[acc_slot<G>(tl, g)]);
            }
        }
    } else if (warp == kPackWarp) {
        // ----------------------------------------------- packed-row producer
        // One TMA tile of packed bytes (and one of scales) per K step of the
        // CTA's sequence into slot g % 8; the FC1 gate/up halves of a tile
        // (rows p and I + p) come as two 64-row tiles.
        if (lane == 0 && a.w_tma) {
            constexpr int kStepBytes = BITS == 4 ? 32 : 24;
            const int SS = ST == kF32 ? 4 : 2;
            const bool halves = MODE == kModeFc1 && !a.inter;
            const uint32_t tx = kBW * kPackRow + (a.s_tma ? kBW * kSclRow : 0);
            const int bs_shift = __ffs(a.bs) - 1;
            RingPos pp;
            for (int t = blockIdx.x; t < n_tiles && !failed; t += gridDim.x) {
                const Tile x = tile_of(a, t, UN);
                const int y0 = static_cast<int>(x.e * a.rows + (halves ? x.n0 / 2 : x.n0));
                const int y1 = static_cast<int>(y0 + a.I);  // halves: the up rows
                for (int ks = 0; ks < ksteps; ++ks, pp.next(kPackSlots)) {
                    if (pp.round && !mbar_wait(&pempty[pp.stage], (pp.round - 1) & 1)) { failed = true; break; }
                    mbar_arrive_expect_tx(&pfull[pp.stage], tx);
                    const int kabs = x.ks0 + ks;
                    const int xw = (kabs * kStepBytes) & ~15;                       // 16-byte aligned window
                    uint8_t* dw = pack + pp.stage * (kBW * kPackRow);
                    if (halves) {
                        tma_load_2d(dw, &tmap_w, xw, y0, &pfull[pp.stage]);
                        tma_load_2d(dw + 64 * kPackRow, &tmap_w, xw, y1, &pfull[pp.stage]);
                    } else {
                        tma_load_2d(dw, &tmap_w, xw, y0, &pfull[pp.stage]);
                    }
                    if (a.s_tma) {
                        const int xs = (((kabs * kBK) >> bs_shift) * SS) & ~15;
                        uint8_t* ds = scl + pp.stage * (kBW * kSclRow);
                        if (halves) {
                            tma_load_2d(ds, &tmap_s, xs, y0, &pfull[pp.stage]);
                            tma_load_2d(ds + 64 * kSclRow, &tmap_s, xs, y1, &pfull[pp.stage]);
                        } else {
                            tma_load_2d(ds, &tmap_s, xs, y0, &pfull[pp.stage]);
                        }
                    }
                }
            }
        }
    } else if (dq_rank >= 0) {
        // ------------------------------------------------------------ dequant
        const int group = dq_rank / kDequantWarps;  // takes K steps = group (mod groups)
        const int dq = (dq_rank - group * kDequantWarps) * 32 + lane;
        const int r = dq & (kBW - 1);                               // row of the packed slot
        const int h0 = kChunksPerThread == 2 ? 0 : dq >> 7;         // this thread's first chunk
        // Tile row (MMA lane) this thread makes: FC1 gate and up rows of pair p
        // sit in slot rows p and 64 + p, and go to tile rows 2p and 2p + 1.
        const int orow = (MODE == kModeFc1 && !a.inter) ? 2 * (r & 63) + (r >> 6) : r;
        constexpr int kCB = BITS == 4 ? 16 : 12;  // packed bytes per 32-code chunk
        constexpr int kStepBytes = 2 * kCB;       // packed bytes of a row per K step
        constexpr int kZ = 1 << (BITS - 1);
        constexpr int SS = ST == kF32 ? 4 : 2;
        const bool w_tma = a.w_tma != 0, s_tma = a.s_tma != 0;
        const int nb = a.nb, bs_shift = __ffs(a.bs) - 1;
        const int64_t kcodes = int64_t(nb) * a.bs;  // codes stored per row
        const int64_t n_scales = a.rows * nb;
        // One tile's source stream for this thread: packed bytes of its weight
        // row, that expert's scales, and the row's first scale index.
        struct RowStream {
            const uint8_t* w;  // packed bytes at the tile's first K step
            const uint8_t* s;
            int64_t si0;
            int ks0;           // the tile's first K step (split of K)
            bool ok;
        };
        auto stream_of = [&](const Tile& x) -> RowStream {
            int64_t wr;
            if (MODE == kModeFc1) {
                const int64_t p = x.n0 / 2 + (orow >> 1), up = orow & 1;  // pair-interleaved tile rows
                wr = p < a.I ? (a.inter ? 2 * p + up : up * a.I + p) : -1;
            } else {
                wr = x.n0 + orow < a.rows ? x.n0 + orow : -1;
            }
            RowStream st;
            st.ok = wr >= 0;
            st.w = a.B + x.e * a.w_expert_stride + (st.ok ? wr : 0) * a.row_bytes + int64_t(x.ks0) * kStepBytes;
            st.s = static_cast<const uint8_t*>(a.scales) + x.e * a.s_expert_stride;
            st.si0 = (st.ok ? wr : 0) * nb;
            st.ks0 = x.ks0;
            return st;
        };
        // This group's K steps, in order: the CTA's tiles t = blockIdx.x + j * gridDim.x,
        // each with ksteps steps, numbered globally; the group takes every fourth one.
        struct Cursor {
            int t, ks;
        };
        auto advance = [&](Cursor& c) {  // kDequantGroups global steps on
            c.ks += kDequantGroups;
            while (c.ks >= ksteps && c.t < n_tiles) {
                c.ks -= ksteps;
                c.t += gridDim.x;
            }
        };
        // Where the rows are not 16-byte aligned, each thread copies what the
        // producer's tiles do not bring, one own K step ahead (cp.async).
        const bool own_copies = !(w_tma && s_tma);
        Cursor pc{static_cast<int>(blockIdx.x), group};  // prefetch cursor
        while (pc.ks >= ksteps && pc.t < n_tiles) {
            pc.ks -= ksteps;
            pc.t += gridDim.x;
        }
        int pslot = 0;
        RowStream ps{nullptr, nullptr, 0, 0, false};
        if (own_copies && pc.t < n_tiles) ps = stream_of(tile_of(a, pc.t, UN));
        // one half-precision scale: the 4-byte word that holds it (the last scale
        // of the array alone, where its word would run past the end)
        auto copy_scale_word = [&](uint32_t* dst, const uint8_t* base, int64_t si) {
            if (ST == kF32) {
                cp_async4(dst, reinterpret_cast<const float*>(base) + si);
            } else if ((si | 1) < n_scales) {
                cp_async4(dst, reinterpret_cast<const uint32_t*>(base) + (si >> 1));
            } else {
                *dst = reinterpret_cast<const uint16_t*>(base)[si];
            }
        };
        auto issue = [&]() {
            const int64_t k0 = int64_t(ps.ks0 + pc.ks) * kBK;  // first code of this K step
            if (pc.t < n_tiles && ps.ok && k0 < kcodes) {
                const int slot = group + kDequantGroups * pslot;
                const bool two = k0 + 32 < kcodes;  // the second chunk holds stored codes
                if (!w_tma) {
                    const uint8_t* src = ps.w + int64_t(pc.ks) * kStepBytes;
                    uint8_t* dst = pack + (slot * kBW + r) * kPackRow;
#pragma unroll
                    for (int i = 0; i < kChunksPerThread; ++i) {
                        const int hh = h0 + i;
                        if (hh == 1 && !two) break;
                        if constexpr (BITS == 4) {
                            cp_async16(dst + hh * kCB, src + hh * kCB);
                        } else {
#pragma unroll
                            for (int q = 0; q < 3; ++q) cp_async4(dst + hh * kCB + 4 * q, src + hh * kCB + 4 * q);
                        }
                    }
                }
                if (!s_tma) {  // word hh: the word holding chunk hh's scale
                    uint32_t* sdst = reinterpret_cast<uint32_t*>(scl + (slot * kBW + r) * kSclRow);
#pragma unroll
                    for (int i = 0; i < kChunksPerThread; ++i) {
                        const int hh = h0 + i;
                        if (hh == 1 && !two) break;
                        copy_scale_word(sdst + hh, ps.s, ps.si0 + ((k0 + 32 * hh) >> bs_shift));
                    }
                }
            }
            cp_async_commit();
            pslot ^= 1;
            if (pc.t < n_tiles) {
                const int t_before = pc.t;
                advance(pc);
                if (pc.t != t_before && pc.t < n_tiles) ps = stream_of(tile_of(a, pc.t, UN));
            }
        };
        if (own_copies) issue();
        // consumer cursor and its place in the weight ring (global step g -> slot g % SW)
        Cursor cc = Cursor{static_cast<int>(blockIdx.x), group};
        while (cc.ks >= ksteps && cc.t < n_tiles) {
            cc.ks -= ksteps;
            cc.t += gridDim.x;
        }
        RingPos rp;
        for (int i = 0; i < group; ++i) rp.next(SW);
        uint32_t own = 0;  // this group's K steps so far: packed slot group + 4 (own & 1), its use own >> 1
        uint32_t swo[4 * kChunksPerThread];  // this thread's 16-byte slots of a weight tile row
#pragma unroll
        for (int c = 0; c < 4 * kChunksPerThread; ++c) swo[c] = sw128(orow, 4 * h0 + c);
        int cur_t = -1;
        RowStream cs{nullptr, nullptr, 0, 0, false};
        const uint8_t* zrow = nullptr;
        while (cc.t < n_tiles && !failed) {
            if (cc.t != cur_t) {
                cur_t = cc.t;
                const Tile x = tile_of(a, cur_t, UN);
                cs = stream_of(x);
                zrow = (a.zp && cs.ok) ? a.zp + x.e * a.z_expert_stride + (cs.si0 / nb) * a.zp_row_bytes : nullptr;
            }
            const int ks = cs.ks0 + cc.ks;  // absolute K step
            const int slot = group + kDequantGroups * static_cast<int>(own & 1);
            if (own_copies) {
                issue();
                cp_async_wait<1>();
            }
            if (w_tma && !warp_wait(&pfull[slot], (own >> 1) & 1)) { failed = true; break; }
            if (rp.round && !warp_wait(&empty_w[rp.stage], (rp.round - 1) & 1)) { failed = true; break; }
            uint8_t* wdst = wt + rp.stage * plan.w;
            const int64_t kstep0 = int64_t(ks) * kBK;
            // packed bytes of this row's K step (the tensor tile's window starts
            // on a 16-byte boundary: INT3 steps at odd positions sit 8 bytes in)
            const uint8_t* prow = pack + (slot * kBW + r) * kPackRow + (w_tma ? (ks * kStepBytes) & 15 : 0);
            // scales: the tensor tile holds the row's 16-byte window around the
            // step's first scale; own copies hold the step's one or two words
            const uint8_t* srow = scl + (slot * kBW + r) * kSclRow;
            uint4 swin = make_uint4(0, 0, 0, 0);
            if (s_tma) swin = *reinterpret_cast<const uint4*>(srow);
            const int xs = static_cast<int>(((kstep0 >> bs_shift) * SS) & ~int64_t(15));
            // the chunks of this row's K step; REM: the remainder operand of the
            // second pass of an fp32 output (a uniform branch, taken once per step)
            auto make_chunks = [&](auto rem) {
#pragma unroll
            for (int i = 0; i < kChunksPerThread; ++i) {
                const int hh = h0 + i;
                const int64_t kc = kstep0 + 32 * hh;  // first code of this chunk
                const bool live = cs.ok && kc < kcodes;
                uint32_t w[BITS];
                float sc = 0.f, z = float(kZ);
                if (live) {
                    const uint8_t* src = prow + hh * kCB;
                    if constexpr (BITS == 4) {
                        const uint4 v = *reinterpret_cast<const uint4*>(src);
                        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
                    } else {
#pragma unroll
                        for (int q = 0; q < BITS; ++q) w[q] = reinterpret_cast<const uint32_t*>(src)[q];
                    }
                    const int64_t si = cs.si0 + (kc >> bs_shift);
                    if (s_tma) {
                        const int b = static_cast<int>((kc >> bs_shift) * SS) - xs;  // byte in the window
                        const int wi = b >> 2;
                        const uint32_t word = wi == 0 ? swin.x : wi == 1 ? swin.y : wi == 2 ? swin.z : swin.w;
                        sc = scale_from_word<ST>(word, b >> 1);
                    } else {
                        sc = scale_from_word<ST>(reinterpret_cast<const uint32_t*>(srow)[hh], si);
                    }
                    if (zrow) z = float(zero_point_code<BITS>(zrow, static_cast<int>(kc >> bs_shift)));
                } else {
#pragma unroll
                    for (int q = 0; q < BITS; ++q) w[q] = 0;
                }
                // w = s (q - z) = f * s 2^(24-p) - s (2^(23-p) + z), one fp32 rounding per value;
                // the pre-scale depends only on the code's position class p
                constexpr int kCls = BITS == 4 ? 2 : 3;
                float mc[kCls], ac[kCls];
#pragma unroll
                for (int c = 0; c < kCls; ++c) {
                    const int p = code_pos<BITS>(c);
                    mc[c] = sc * float(1u << (24 - p));
                    ac[c] = -sc * (float(1u << (23 - p)) + z);
                }
                uint32_t outw[16];
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    float2 f01, f23;
                    chunk_codes4<BITS>(w, g, f01, f23);
                    const int j = 4 * g;
                    const float2 v01 = ffma2(f01, make_float2(mc[j % kCls], mc[(j + 1) % kCls]),
                                             make_float2(ac[j % kCls], ac[(j + 1) % kCls]));
                    const float2 v23 = ffma2(f23, make_float2(mc[(j + 2) % kCls], mc[(j + 3) % kCls]),
                                             make_float2(ac[(j + 2) % kCls], ac[(j + 3) % kCls]));
                    outw[2 * g] = pack2_part<AT, decltype(rem)::value>(v01);
                    outw[2 * g + 1] = pack2_part<AT, decltype(rem)::value>(v23);
                }
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    *reinterpret_cast<uint4*>(wdst + swo[4 * i + c]) =
                        make_uint4(outw[4 * c], outw[4 * c + 1], outw[4 * c + 2], outw[4 * c + 3]);
            }
            };
            if (a.remainder)
                make_chunks(std::true_type{});
            else
                make_chunks(std::false_type{});
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&full_w[rp.stage]);
                if (w_tma) mbar_arrive(&pempty[slot]);
            }
            ++own;
#pragma unroll
            for (int i = 0; i < kDequantGroups; ++i) rp.next(SW);
            advance(cc);
        }
        cp_async_wait<0>();
    } else if (warp >= kEpilogueWarp0 && warp < kEpilogueWarp0 + 4) {
        // ----------------------------------------------------------- epilogue
        // One lane polls the accumulator barrier; the four epilogue warps meet
        // on a named barrier, so the others take no issue slots while waiting.
        const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
        const bool poller = warp == kEpilogueWarp0 && lane == 0;
        int tl = 0;
        for (int t = blockIdx.x; t < n_tiles && !failed; t += gridDim.x, ++tl) {
            const Tile x = tile_of(a, t, UN);
            const int uses = acc_uses<G>(tl);
            const int rr = quarter * 32 + lane;  // tile row of this thread
#pragma unroll 1
            for (int g = 0; g < G; ++g) {
                const int slot = acc_slot<G>(tl, g);
                if (poller && !mbar_wait(&acc_full[slot], uses & 1)) *epi_fail = 1;
                epilogue_sync();
                if (*epi_fail) { failed = true; break; }
                tc_fence_after();
                const int cnt = x.cnt - g * BN;  // live activation rows of this sub-tile
                const int64_t m0 = int64_t(x.s0) + g * BN;
#pragma unroll 1
                for (int c0 = 0; c0 < BN && c0 < cnt; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld32(tmem + (uint32_t(quarter * 32) << 16) + slot * BN + c0, v);
                    tmem_ld_wait();
                    // live columns of this 32-column chunk (a 16-column tile loads 32: the
                    // upper 16 belong to the other accumulator)
                    const int jn = min(32, min(BN - c0, cnt - c0));
                    if constexpr (MODE == kModeFc1) {
                        // Lanes 2i / 2i+1 hold the gate / up rows of pair p: the even lane
                        // makes h for the even columns, the odd lane for the odd ones,
                        // each trading the value the other needs in one shuffle.
                        const int64_t p = x.n0 / 2 + (rr >> 1);
                        const int odd = lane & 1;
                        float bg = 0.f, bu = 0.f;  // biases of the pair's gate and up rows
                        if (a.bias && p < a.I) {
                            const auto* bp = static_cast<const typename DType<AT>::T*>(a.bias) + x.e * a.rows;
                            bg = to_f32(bp[a.inter ? 2 * p : p]);
                            bu = to_f32(bp[a.inter ? 2 * p + 1 : a.I + p]);
                        }
#pragma unroll
                        for (int j = 0; j < 32; j += 2) {
                            const float send = __uint_as_float(odd ? v[j] : v[j + 1]);  // even: gate of j+1; odd: up of j
                            const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
                            const float gate = (odd ? recv : __uint_as_float(v[j])) + bg;
                            const float up = (odd ? __uint_as_float(v[j + 1]) : recv) + bu;
                            const int col = j + odd;
                            if (col < jn && p < a.I) {
                                // h is rounded to the 16-bit activation type next, so the fast
                                // exponential and division (a few ulp of fp32) do not show
                                const float hv = __fdividef(gate, 1.0f + __expf(-gate)) * up;
                                store_from_f32(a.Y, a.y_dtype, (m0 + c0 + col) * a.ld_y + p, hv);
                            }
                        }
                    } else {
                        const int64_t n = x.n0 + rr;
                        if (a.bias && n < a.rows) {  // grouped FC2: the expert's bias of row n
                            const float b = to_f32(static_cast<const typename DType<AT>::T*>(a.bias)[x.e * a.rows + n]);
#pragma unroll
                            for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) + b);
                        }
                        if (n < a.rows && a.splits > 1) {  // fp32 partial sums of this split of K
                            float* pp = a.partials + (int64_t(x.split) * a.M + m0 + c0) * a.ld_y + n;
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                if (j < jn) pp[j * a.ld_y] = __uint_as_float(v[j]);
                        } else if (n < a.rows) {
                            if (a.y_dtype == AT) {  // 16-bit output: one strided pointer
                                using OT = typename DType<AT>::T;
                                OT* yp = static_cast<OT*>(a.Y) + (m0 + c0) * a.ld_y + n;
                                const int64_t ld = a.ld_y;
                                if (jn == 32) {
#pragma unroll
                                    for (int j = 0; j < 32; ++j) yp[j * ld] = from_f32<OT>(__uint_as_float(v[j]));
                                } else {
#pragma unroll
                                    for (int j = 0; j < 32; ++j)
                                        if (j < jn) yp[j * ld] = from_f32<OT>(__uint_as_float(v[j]));
                                }
                            } else if (a.remainder) {  // second pass of an fp32 output: add
                                float* yp = static_cast<float*>(a.Y) + (m0 + c0) * a.ld_y + n;
#pragma unroll
                                for (int j = 0; j < 32; ++j)
                                    if (j < jn) yp[j * a.ld_y] += __uint_as_float(v[j]);
                            } else {
#pragma unroll
                                for (int j = 0; j < 32; ++j)
                                    if (j < jn)
                                        store_from_f32(a.Y, a.y_dtype, (m0 + c0 + j) * a.ld_y + n, __uint_as_float(v[j]));
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[slot]);
            }
        }
    }
    if (failed) record_error(MNB_ERR_TIMEOUT);
    grid_launch_dependents();
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, a.tmem_cols);
    }
}

// ------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Ring depths: kWeightSlots dequantised-weight slots, and as many activation
// slots as fit (up to kMaxStagesTC).  A group waits on the weight slot of its
// next K step, kDequantGroups global steps after its last one; an mbarrier
// parity wait is only sound while the slot's barrier is at most one phase
// behind the awaited one, which holds exactly when that slot's previous use
// was at or before the group's last step, i.e. stages_w >= kDequantGroups.
void stages_for(int BN, int G, int bits, int* stages, int* stages_w) {
    static_assert(kWeightSlots >= kDequantGroups, "a parity wait needs a weight slot per group");
    int s = std::min(kMaxStagesTC, kWeightSlots);  // activation stages share the weight ring's barriers
    while (s > 2 && tc_plan(BN, G, s, kWeightSlots, bits).total > 227 * 1024) --s;
    *stages_w = kWeightSlots;
    *stages = s;
}

template <int BITS, int ST, int AT, int BN, int G, int MODE>
cudaError_t launch_cfg(const TcArgs& in, const void* A_rows, int64_t a_rows, int64_t a_cols, int grid,
                       bool pdl, cudaStream_t stream) {
    TcArgs a = in;
    CUtensorMap tmap;
    std::memset(&tmap, 0, sizeof tmap);
    {
        // activations [a_rows, a_cols] in BN-row tiles
        auto encode = encode_fn();
        if (!encode) return cudaErrorNotSupported;
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a_cols), static_cast<cuuint64_t>(a_rows)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a_cols * 2)};
        const cuuint32_t box[2] = {kBK, static_cast<cuuint32_t>(BN)};
        const cuuint32_t estr[2] = {1, 1};
        const CUresult cr = encode(&tmap, AT == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                                   2, const_cast<void*>(A_rows), dims, strides, box, estr,
                                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    // Packed rows and scales as [rows x bytes] tensors of all stacked matrices,
    // read in tiles of 128 rows (FC1 with separate gate/up halves: 64) by 32
    // (scales: 16) bytes; only where every row starts on a 16-byte boundary.
    CUtensorMap tmap_w, tmap_s;
    std::memset(&tmap_w, 0, sizeof tmap_w);
    std::memset(&tmap_s, 0, sizeof tmap_s);
    {
        auto encode = encode_fn();
        const int64_t ex = a.experts > 1 ? a.experts : 1;
        const int64_t all_rows = ex * a.rows;
        const cuuint32_t box_rows = (MODE == kModeFc1 && !a.inter) ? 64 : kBW;
        const int ss = ST == kF32 ? 4 : 2;
        const int64_t s_row = int64_t(a.nb) * ss;
        auto aligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
        a.w_tma = 0;
        a.s_tma = 0;
        if (all_rows < (int64_t(1) << 31) && aligned(a.B) && a.row_bytes % 16 == 0 &&
            (ex == 1 || a.w_expert_stride == a.rows * a.row_bytes)) {
            const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.row_bytes), static_cast<cuuint64_t>(all_rows)};
            const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.row_bytes)};
            const cuuint32_t box[2] = {kPackRow, box_rows};
            const cuuint32_t estr[2] = {1, 1};
            a.w_tma = encode(&tmap_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a.B), dims, strides,
                             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
        }
        if (a.w_tma && aligned(a.scales) && s_row % 16 == 0 && (ex == 1 || a.s_expert_stride == a.rows * s_row)) {
            const cuuint64_t dims[2] = {static_cast<cuuint64_t>(s_row), static_cast<cuuint64_t>(all_rows)};
            const cuuint64_t strides[1] = {static_cast<cuuint64_t>(s_row)};
            const cuuint32_t box[2] = {kSclRow, box_rows};
            const cuuint32_t estr[2] = {1, 1};
            a.s_tma = encode(&tmap_s, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(a.scales), dims, strides,
                             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
        }
    }
    // two accumulators of BN columns; the epilogue reads 32 columns at a time,
    // so a 16-column accumulator needs 16 more behind it
    uint32_t cols = 32;
    while (cols < 2u * BN + (BN < 32 ? 32u - BN : 0u)) cols <<= 1;
    a.tmem_cols = cols;
    stages_for(BN, G, BITS, &a.stages, &a.stages_w);
    const int64_t smem = tc_plan(BN, G, a.stages, a.stages_w, BITS).total;
    auto kern = gemm_tc_kernel<BITS, ST, AT, BN, G, MODE>;
    cudaError_t e = set_kernel_smem(kern, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(std::max(grid, 1)), 1, 1);
    cfg.blockDim = dim3(kThreadsTC, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, tmap, tmap_w, tmap_s, a);
}

template <int MODE, int BITS, int ST, int AT>
cudaError_t launch_bn(int BN, int G, const TcArgs& a, const void* A_rows, int64_t a_rows, int64_t a_cols, int grid,
                      bool pdl, cudaStream_t stream) {
    if constexpr (MODE == kModeFc1) {  // grouped / dense gate-up: 32 .. 256 activation rows per tile
        switch (BN) {
            case 256: return launch_cfg<BITS, ST, AT, 256, 1, MODE>(a, A_rows, a_rows, a_cols, grid, pdl, stream);
            case 128: return launch_cfg<BITS, ST, AT, 128, 1, MODE>(a, A_rows, a_rows, a_cols, grid, pdl, stream);
            case 64: return launch_cfg<BITS, ST, AT, 64, 1, MODE>(a, A_rows, a_rows, a_cols, grid, pdl, stream);
            default: return launch_cfg<BITS, ST, AT, 32, 1, MODE>(a, A_rows, a_rows, a_cols, grid, pdl, stream);
        }
    } else {
        switch (BN) {
            case 256: return launch_cfg<BITS, ST, AT, 256, 1, MODE>(a, A_rows, a_rows, a_cols, grid, pdl, stream);
            case 128: return launch_cfg<BITS, ST, AT, 128, 1, MODE>(a, A_rows, a_rows, a_cols, grid, pdl, stream);
            case 64: return launch_cfg<BITS, ST, AT, 64, 1, MODE>(a, A_rows, a_rows, a_cols, grid, pdl, stream);
            case 32: return launch_cfg<BITS, ST, AT, 32, 1, MODE>(a, A_rows, a_rows, a_cols, grid, pdl, stream);
            default: return launch_cfg<BITS, ST, AT, 16, 1, MODE>(a, A_rows, a_rows, a_cols, grid, pdl, stream);
        }
    }
}

}  // namespace

// One (mode, bit width) slice of the instantiations; each slice lives in its own
// translation unit so the slices compile in parallel.
#define MNB_GEMM_TC_SLICE(NAME, MODE, BITS)                                                                     \
    cudaError_t NAME(int scale_dtype, int a_dtype, int BN, int G, const TcArgs& a, const void* A_rows,          \
                     int64_t a_rows, int64_t a_cols, int grid, bool pdl, cudaStream_t stream) {                 \
        const bool sf = scale_dtype == kF32;                                                                     \
        if (a_dtype == kBF16)                                                                                    \
            return sf ? launch_bn<MODE, BITS, kF32, kBF16>(BN, G, a, A_rows, a_rows, a_cols, grid, pdl, stream)  \
                      : launch_bn<MODE, BITS, kBF16, kBF16>(BN, G, a, A_rows, a_rows, a_cols, grid, pdl, stream); \
        return sf ? launch_bn<MODE, BITS, kF32, kF16>(BN, G, a, A_rows, a_rows, a_cols, grid, pdl, stream)       \
                  : launch_bn<MODE, BITS, kF16, kF16>(BN, G, a, A_rows, a_rows, a_cols, grid, pdl, stream);      \
    }                                                                                                            \
    cudaError_t NAME##_take_error(unsigned int* out) { return take_unit_error(out); }

}  // namespace mnb
