// mnb_api.cu -- the extern "C" entry points declared in include/mnb.h:
// host-side metadata validation (payloads are never read on the host), plan
// selection and kernel launches on the caller's stream.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "kernels.h"
#include "qmoe.h"

namespace mnb {

namespace {

// Smallest M routed to the tensor-core GEMM (fp16/bf16 activations only).
constexpr int64_t kTcMinRows = 16;

bool valid_dtype(int d) { return d == MNB_F32 || d == MNB_F16 || d == MNB_BF16; }
bool valid_bits(int b) { return b == 3 || b == 4; }
// mnb_matmul / mnb_matmul_int8a: every width of the row-local LSB-first format
// (3 and 4 on every path; 1, 2 and 5..8 on the CUDA-core path for any M)
bool valid_bits_any(int b) { return b >= 1 && b <= 8; }
bool valid_bs(int bs) { return bs == 32 || bs == 64 || bs == 128; }
size_t dsize(int d) { return d == MNB_F32 ? 4 : 2; }
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// a * b without overflow past 2^62 (the largest byte count we accept).
bool mul_ok(int64_t a, int64_t b, int64_t* out) {
    if (a < 0 || b < 0) return false;
    if (a != 0 && b > (int64_t(1) << 62) / a) return false;
    *out = a * b;
    return true;
}

int sm_count_current() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

// Programmatic dependent launch is on unless MNB_DISABLE_PDL is set in the
// environment (for tools that replay kernels one by one).
bool pdl_enabled() {
    static const bool on = std::getenv("MNB_DISABLE_PDL") == nullptr;
    return on;
}

mnb_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return MNB_OK;
    if (e == cudaErrorNotSupported) return MNB_ERR_UNSUPPORTED;
    return MNB_ERR_CUDA;
}

// Byte counts of one packed projection [N, K]; false on overflow.
struct ProjBytes {
    int64_t nb, row_bytes, weight, scales, zp_row, zp;
};
bool proj_bytes(int64_t N, int64_t K, int bits, int bs, int sdt, ProjBytes* p) {
    p->nb = (K + bs - 1) / bs;
    p->row_bytes = p->nb * bs * bits / 8;
    p->zp_row = (p->nb * bits + 7) / 8;
    return mul_ok(N, p->row_bytes, &p->weight) && mul_ok(N, p->nb * int64_t(dsize(sdt)), &p->scales) &&
           mul_ok(N, p->zp_row, &p->zp);
}

// The version-1 prepacked row of a weight: code bytes, scale bytes, zero-point
// bytes, and the row stride rounded up to 16 bytes.
struct PpLayout {
    int64_t nb, code_bytes, scale_off, zp_off, stride, bytes;
};
bool pp_layout(int64_t N, int64_t K, int bits, int bs, int sdt, bool has_zp, PpLayout* l) {
    l->nb = (K + bs - 1) / bs;
    l->code_bytes = l->nb * bs * bits / 8;
    l->scale_off = l->code_bytes;
    const int64_t s_row = l->nb * dsize(sdt);
    const int64_t z_row = (l->nb * bits + 7) / 8;
    l->zp_off = has_zp ? l->scale_off + s_row : -1;
    l->stride = (l->code_bytes + s_row + (has_zp ? z_row : 0) + 15) / 16 * 16;
    int64_t rows;
    if (!mul_ok(N, l->stride, &rows)) return false;
    l->bytes = rows + MNB_PREPACK_HEADER_BYTES;
    return l->bytes > rows;
}

}  // namespace
}  // namespace mnb

using namespace mnb;

extern "C" {

const char* mnb_status_string(mnb_status s) {
    switch (s) {
        case MNB_OK: return "MNB_OK";
        case MNB_ERR_INVALID_ARG: return "MNB_ERR_INVALID_ARG";
        case MNB_ERR_UNSUPPORTED: return "MNB_ERR_UNSUPPORTED";
        case MNB_ERR_SIZE_OVERFLOW: return "MNB_ERR_SIZE_OVERFLOW";
        case MNB_ERR_WORKSPACE: return "MNB_ERR_WORKSPACE";
        case MNB_ERR_CUDA: return "MNB_ERR_CUDA";
        case MNB_ERR_TIMEOUT: return "MNB_ERR_TIMEOUT";
        case MNB_ERR_CONTENT: return "MNB_ERR_CONTENT";
    }
    return "MNB_ERR_UNKNOWN";
}

mnb_status mnb_get_last_device_error(mnb_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return MNB_ERR_CUDA;
    unsigned int first = 0;
    cudaError_t (*takers[])(unsigned int*) = {gemv_take_error, gemv_pp_take_error, qmoe_take_error,
                                              gemm_tc_take_error, quant_take_error, diag_take_error,
                                              qmoe_decode_take_error};
    for (auto take : takers) {
        unsigned int v = 0;
        if (take(&v) != cudaSuccess) return MNB_ERR_CUDA;
        if (first == 0) first = v;
    }
    return static_cast<mnb_status>(first);
}

mnb_status mnb_diag_wait_timeout(uint64_t limit_ns, mnb_stream_t stream) {
    if (limit_ns < 1000 || limit_ns > 1000000000ull) return MNB_ERR_INVALID_ARG;
    return from_cuda(launch_diag_wait_timeout(limit_ns, reinterpret_cast<cudaStream_t>(stream)));
}

mnb_status mnb_matmul_workspace_size(int64_t M, int64_t K, int64_t N, int bits, int block_size,
                                     mnb_dtype a_dtype, size_t* bytes) {
    if (!bytes) return MNB_ERR_INVALID_ARG;
    if (M < 1 || K < 1 || N < 1 || !valid_dtype(a_dtype)) return MNB_ERR_INVALID_ARG;
    if (!valid_bits_any(bits) || !valid_bs(block_size)) return MNB_ERR_UNSUPPORTED;
    *bytes = 0;
    if (!valid_bits(bits)) return MNB_OK;  // other widths run on CUDA cores without a workspace
    // The tensor-core path splits K when its output tiles cannot fill the GPU;
    // the size is planned for a 152-SM GB300 so that it depends only on the
    // arguments (a call given less workspace splits less, or not at all).
    if (a_dtype != MNB_F32 && M >= kTcMinRows && K % 8 == 0) *bytes = gemm_tc_workspace_bytes(M, K, N, 152);
    return MNB_OK;
}

mnb_status mnb_matmul(const void* A, mnb_dtype a_dtype, int64_t M, int64_t K, const uint8_t* B_packed,
                      const void* scales, mnb_dtype scale_dtype, const uint8_t* zero_points, int64_t N,
                      int bits, int block_size, void* Y, mnb_dtype y_dtype, void* workspace,
                      size_t workspace_bytes, mnb_stream_t stream) {
    if (!A || !B_packed || !scales || !Y) return MNB_ERR_INVALID_ARG;
    if (M < 1 || K < 1 || N < 1) return MNB_ERR_INVALID_ARG;
    if (!valid_dtype(a_dtype) || !valid_dtype(scale_dtype) || !valid_dtype(y_dtype)) return MNB_ERR_INVALID_ARG;
    if (!valid_bits_any(bits) || !valid_bs(block_size)) return MNB_ERR_UNSUPPORTED;
    if (scale_dtype != MNB_F32 && scale_dtype != a_dtype) return MNB_ERR_UNSUPPORTED;
    if (!aligned(B_packed, 16) || !aligned(scales, 16) || !aligned(A, dsize(a_dtype)) ||
        !aligned(Y, dsize(y_dtype)))
        return MNB_ERR_UNSUPPORTED;
    ProjBytes pb;
    int64_t tmp;
    if (!proj_bytes(N, K, bits, block_size, scale_dtype, &pb) || !mul_ok(M, K * 4, &tmp) ||
        !mul_ok(M, N * 4, &tmp))
        return MNB_ERR_SIZE_OVERFLOW;
    if (N > (int64_t(1) << 31)) return MNB_ERR_UNSUPPORTED;
    const int sms = sm_count_current();
    if (sms <= 0) return MNB_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

    // Tensor-core path: 3- and 4-bit weights, fp16/bf16 activations, enough
    // rows to fill an MMA column block, and a TMA-compatible activation matrix.
    if (valid_bits(bits) && a_dtype != MNB_F32 && M >= kTcMinRows && K % 8 == 0 && aligned(A, 16)) {
        GemmTcArgs g = {};
        g.A = A;
        g.a_dtype = a_dtype;
        g.M = M;
        g.K = K;
        g.B = B_packed;
        g.scales = scales;
        g.zp = zero_points;
        g.N = N;
        g.bits = bits;
        g.bs = block_size;
        g.nb = static_cast<int>(pb.nb);
        g.row_bytes = pb.row_bytes;
        g.zp_row_bytes = static_cast<int>(pb.zp_row);
        g.Y = Y;
        g.y_dtype = y_dtype;
        g.workspace = aligned(workspace, 16) ? workspace : nullptr;
        g.workspace_bytes = g.workspace ? workspace_bytes : 0;
        return from_cuda(launch_gemm_tc(g, scale_dtype, sms, pdl_enabled(), st));
    }
    if (gemv_smem_bytes(M, K, bits, block_size, scale_dtype) == 0) return MNB_ERR_UNSUPPORTED;

    GemvArgs a = {};
    a.A = A;
    a.a_dtype = a_dtype;
    a.M = M;
    a.K = K;
    a.B = B_packed;
    a.scales = scales;
    a.zp = zero_points;
    a.N = N;
    a.bits = bits;
    a.bs = block_size;
    a.nb = static_cast<int>(pb.nb);
    a.row_bytes = pb.row_bytes;
    a.zp_row_bytes = static_cast<int>(pb.zp_row);
    a.Y = Y;
    a.y_dtype = y_dtype;
    a.y_ld = N;
    a.chunks = static_cast<int>(pb.nb * block_size / 32);
    a.a_vec = aligned(A, 16) && (K * int64_t(dsize(a_dtype))) % 16 == 0;
    return from_cuda(launch_gemv(a, scale_dtype, sms, pdl_enabled(), st));
}

mnb_status mnb_matmul_int8a(const void* A, mnb_dtype a_dtype, int64_t M, int64_t K, const uint8_t* B_packed,
                            const void* scales, mnb_dtype scale_dtype, const uint8_t* zero_points, int64_t N,
                            int bits, int block_size, void* Y, mnb_dtype y_dtype, mnb_stream_t stream) {
    if (!A || !B_packed || !scales || !Y) return MNB_ERR_INVALID_ARG;
    if (M < 1 || K < 1 || N < 1) return MNB_ERR_INVALID_ARG;
    if (!valid_dtype(a_dtype) || !valid_dtype(scale_dtype) || !valid_dtype(y_dtype)) return MNB_ERR_INVALID_ARG;
    if (!valid_bits_any(bits) || !valid_bs(block_size)) return MNB_ERR_UNSUPPORTED;
    if (scale_dtype != MNB_F32 && scale_dtype != a_dtype) return MNB_ERR_UNSUPPORTED;
    if (!aligned(B_packed, 16) || !aligned(scales, 16) || !aligned(A, dsize(a_dtype)) ||
        !aligned(Y, dsize(y_dtype)))
        return MNB_ERR_UNSUPPORTED;
    ProjBytes pb;
    int64_t tmp;
    if (!proj_bytes(N, K, bits, block_size, scale_dtype, &pb) || !mul_ok(M, K * 4, &tmp) ||
        !mul_ok(M, N * 4, &tmp))
        return MNB_ERR_SIZE_OVERFLOW;
    if (N > (int64_t(1) << 31)) return MNB_ERR_UNSUPPORTED;
    if (gemv_smem_bytes(M, K, bits, block_size, scale_dtype) == 0) return MNB_ERR_UNSUPPORTED;
    const int sms = sm_count_current();
    if (sms <= 0) return MNB_ERR_CUDA;
    GemvArgs a = {};
    a.A = A;
    a.a_dtype = a_dtype;
    a.M = M;
    a.K = K;
    a.B = B_packed;
    a.scales = scales;
    a.zp = zero_points;
    a.N = N;
    a.bits = bits;
    a.bs = block_size;
    a.nb = static_cast<int>(pb.nb);
    a.row_bytes = pb.row_bytes;
    a.zp_row_bytes = static_cast<int>(pb.zp_row);
    a.Y = Y;
    a.y_dtype = y_dtype;
    a.y_ld = N;
    a.chunks = static_cast<int>(pb.nb * block_size / 32);
    a.a_vec = aligned(A, 16) && (K * int64_t(dsize(a_dtype))) % 16 == 0;
    a.int8a = 1;
    return from_cuda(launch_gemv(a, scale_dtype, sms, pdl_enabled(), reinterpret_cast<cudaStream_t>(stream)));
}

mnb_status mnb_prepack_size(int64_t N, int64_t K, int bits, int block_size, mnb_dtype scale_dtype,
                            int has_zero_points, size_t* bytes) {
    if (!bytes) return MNB_ERR_INVALID_ARG;
    *bytes = 0;
    if (N < 1 || K < 1 || !valid_dtype(scale_dtype)) return MNB_ERR_INVALID_ARG;
    if (!valid_bits(bits) || !valid_bs(block_size)) return MNB_ERR_UNSUPPORTED;
    PpLayout l;
    if (!pp_layout(N, K, bits, block_size, scale_dtype, has_zero_points != 0, &l)) return MNB_ERR_SIZE_OVERFLOW;
    *bytes = static_cast<size_t>(l.bytes);
    return MNB_OK;
}

mnb_status mnb_prepack(const uint8_t* B_packed, const void* scales, mnb_dtype scale_dtype,
                       const uint8_t* zero_points, int64_t N, int64_t K, int bits, int block_size, uint64_t identity,
                       void* dst, size_t dst_bytes, mnb_prepacked_desc* desc, mnb_stream_t stream) {
    if (!B_packed || !scales || !dst || !desc) return MNB_ERR_INVALID_ARG;
    if (N < 1 || K < 1 || !valid_dtype(scale_dtype)) return MNB_ERR_INVALID_ARG;
    if (!valid_bits(bits) || !valid_bs(block_size)) return MNB_ERR_UNSUPPORTED;
    if (!aligned(B_packed, 16) || !aligned(scales, dsize(scale_dtype)) || !aligned(dst, 16))
        return MNB_ERR_UNSUPPORTED;
    if (N > (int64_t(1) << 31)) return MNB_ERR_UNSUPPORTED;
    PpLayout l;
    ProjBytes pb;
    if (!pp_layout(N, K, bits, block_size, scale_dtype, zero_points != nullptr, &l) ||
        !proj_bytes(N, K, bits, block_size, scale_dtype, &pb))
        return MNB_ERR_SIZE_OVERFLOW;
    if (dst_bytes < static_cast<size_t>(l.bytes)) return MNB_ERR_WORKSPACE;
    // the destination must not overlap any source
    auto overlaps = [&](const void* p, int64_t n) {
        const uintptr_t a0 = reinterpret_cast<uintptr_t>(p), d0 = reinterpret_cast<uintptr_t>(dst);
        return a0 < d0 + static_cast<uintptr_t>(l.bytes) && d0 < a0 + static_cast<uintptr_t>(n);
    };
    if (overlaps(B_packed, pb.weight) || overlaps(scales, pb.scales) || (zero_points && overlaps(zero_points, pb.zp)))
        return MNB_ERR_INVALID_ARG;
    const int sms = sm_count_current();
    if (sms <= 0) return MNB_ERR_CUDA;
    mnb_prepacked_desc d = {};
    d.magic = MNB_PREPACK_MAGIC;
    d.version = MNB_PREPACK_VERSION;
    d.N = N;
    d.K = K;
    d.bits = bits;
    d.block_size = block_size;
    d.scale_dtype = scale_dtype;
    d.has_zp = zero_points != nullptr;
    d.row_stride = l.stride;
    d.scale_offset = l.scale_off;
    d.zp_offset = l.zp_off;
    d.bytes = l.bytes;
    d.identity = identity;
    const cudaError_t e = launch_prepack(B_packed, scales, scale_dtype, zero_points, N, K, bits, block_size, &d,
                                         sizeof d, static_cast<uint8_t*>(dst), l.stride, l.scale_off, l.zp_off, sms,
                                         reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return from_cuda(e);
    *desc = d;
    return MNB_OK;
}

mnb_status mnb_matmul_prepacked(const void* A, mnb_dtype a_dtype, int64_t M, int64_t K,
                                const mnb_prepacked_desc* desc, const void* prepacked, void* Y, mnb_dtype y_dtype,
                                mnb_stream_t stream) {
    if (!A || !desc || !prepacked || !Y) return MNB_ERR_INVALID_ARG;
    if (desc->magic != MNB_PREPACK_MAGIC || desc->version != MNB_PREPACK_VERSION || desc->K != K)
        return MNB_ERR_INVALID_ARG;
    const int64_t N = desc->N;
    const int bits = desc->bits, bs = desc->block_size;
    const mnb_dtype sdt = static_cast<mnb_dtype>(desc->scale_dtype);
    if (M < 1 || K < 1 || N < 1) return MNB_ERR_INVALID_ARG;
    if (!valid_dtype(a_dtype) || !valid_dtype(sdt) || !valid_dtype(y_dtype)) return MNB_ERR_INVALID_ARG;
    if (!valid_bits(bits) || !valid_bs(bs)) return MNB_ERR_INVALID_ARG;
    PpLayout l;
    if (!pp_layout(N, K, bits, bs, sdt, desc->has_zp != 0, &l)) return MNB_ERR_SIZE_OVERFLOW;
    if (l.stride != desc->row_stride || l.scale_off != desc->scale_offset || l.zp_off != desc->zp_offset ||
        l.bytes != desc->bytes)
        return MNB_ERR_INVALID_ARG;
    if (sdt != MNB_F32 && sdt != a_dtype) return MNB_ERR_UNSUPPORTED;
    if (!aligned(prepacked, 16) || !aligned(A, dsize(a_dtype)) || !aligned(Y, dsize(y_dtype)))
        return MNB_ERR_UNSUPPORTED;
    int64_t tmp;
    if (!mul_ok(M, K * 4, &tmp) || !mul_ok(M, N * 4, &tmp)) return MNB_ERR_SIZE_OVERFLOW;
    if (N > (int64_t(1) << 31)) return MNB_ERR_UNSUPPORTED;
    const int sms = sm_count_current();
    if (sms <= 0) return MNB_ERR_CUDA;
    GemvArgs a = {};
    a.A = A;
    a.a_dtype = a_dtype;
    a.M = M;
    a.K = K;
    a.B = static_cast<const uint8_t*>(prepacked) + MNB_PREPACK_HEADER_BYTES;
    a.N = N;
    a.bits = bits;
    a.bs = bs;
    a.nb = static_cast<int>(l.nb);
    a.row_bytes = l.stride;
    a.Y = Y;
    a.y_dtype = y_dtype;
    a.y_ld = N;
    a.chunks = static_cast<int>(l.nb * bs / 32);
    a.a_vec = aligned(A, 16) && (K * int64_t(dsize(a_dtype))) % 16 == 0;
    a.pp_header = prepacked;
    a.pp_identity = desc->identity;
    a.pp_scale_off = l.scale_off;
    a.pp_zp_off = l.zp_off;
    return from_cuda(launch_gemv_prepacked(a, sdt, sms, pdl_enabled(), reinterpret_cast<cudaStream_t>(stream)));
}

mnb_status mnb_gate_up_swiglu(const void* A, mnb_dtype a_dtype, int64_t M, int64_t K, const uint8_t* B_packed,
                              const void* scales, mnb_dtype scale_dtype, const uint8_t* zero_points, int64_t I,
                              int bits, int block_size, mnb_fc1_layout layout, void* Y, mnb_dtype y_dtype,
                              mnb_stream_t stream) {
    if (!A || !B_packed || !scales || !Y) return MNB_ERR_INVALID_ARG;
    if (M < 1 || K < 1 || I < 1) return MNB_ERR_INVALID_ARG;
    if (layout != MNB_FC1_INTERLEAVED && layout != MNB_FC1_CONCAT) return MNB_ERR_INVALID_ARG;
    if (!valid_dtype(a_dtype) || !valid_dtype(scale_dtype) || !valid_dtype(y_dtype)) return MNB_ERR_INVALID_ARG;
    if (!valid_bits(bits) || !valid_bs(block_size)) return MNB_ERR_UNSUPPORTED;
    if (scale_dtype != MNB_F32 && scale_dtype != a_dtype) return MNB_ERR_UNSUPPORTED;
    if (!aligned(B_packed, 16) || !aligned(scales, 16) || !aligned(A, dsize(a_dtype)) ||
        !aligned(Y, dsize(y_dtype)))
        return MNB_ERR_UNSUPPORTED;
    ProjBytes pb;
    int64_t tmp;
    if (!proj_bytes(2 * I, K, bits, block_size, scale_dtype, &pb) || !mul_ok(M, K * 4, &tmp) ||
        !mul_ok(M, I * 4, &tmp))
        return MNB_ERR_SIZE_OVERFLOW;
    if (2 * I > (int64_t(1) << 31)) return MNB_ERR_UNSUPPORTED;
    const bool inter = layout == MNB_FC1_INTERLEAVED;
    const int sms = sm_count_current();
    if (sms <= 0) return MNB_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // tensor cores: 16-bit activations and output (the SwiGLU of two 16-bit
    // products has no exact fp32 second pass)
    if (a_dtype != MNB_F32 && y_dtype == a_dtype && M >= kTcMinRows && K % 8 == 0 && aligned(A, 16)) {
        GemmTcArgs g = {};
        g.A = A;
        g.a_dtype = a_dtype;
        g.M = M;
        g.K = K;
        g.B = B_packed;
        g.scales = scales;
        g.zp = zero_points;
        g.N = 2 * I;
        g.bits = bits;
        g.bs = block_size;
        g.nb = static_cast<int>(pb.nb);
        g.row_bytes = pb.row_bytes;
        g.zp_row_bytes = static_cast<int>(pb.zp_row);
        g.Y = Y;
        g.y_dtype = y_dtype;
        return from_cuda(launch_gate_up_tc(g, I, inter, scale_dtype, sms, pdl_enabled(), st));
    }
    // CUDA cores: the gate and up halves of the concatenated layout are staged
    // by separate bulk copies, which need whole 16-byte rows
    if (!inter && (pb.row_bytes % 16 || (pb.nb * int64_t(dsize(scale_dtype))) % 16)) return MNB_ERR_UNSUPPORTED;
    if (gemv_smem_bytes(M, K, bits, block_size, scale_dtype) == 0) return MNB_ERR_UNSUPPORTED;
    GemvArgs a = {};
    a.A = A;
    a.a_dtype = a_dtype;
    a.M = M;
    a.K = K;
    a.B = B_packed;
    a.scales = scales;
    a.zp = zero_points;
    a.N = 2 * I;
    a.bits = bits;
    a.bs = block_size;
    a.nb = static_cast<int>(pb.nb);
    a.row_bytes = pb.row_bytes;
    a.zp_row_bytes = static_cast<int>(pb.zp_row);
    a.Y = Y;
    a.y_dtype = y_dtype;
    a.y_ld = I;
    a.chunks = static_cast<int>(pb.nb * block_size / 32);
    a.a_vec = aligned(A, 16) && (K * int64_t(dsize(a_dtype))) % 16 == 0;
    a.swiglu = 1;
    a.fc1_inter = inter ? 1 : 0;
    a.pairs = I;
    return from_cuda(launch_gemv(a, scale_dtype, sms, pdl_enabled(), st));
}

mnb_status mnb_unpack_codes(const uint8_t* B_packed, int64_t rows, int64_t K, int bits, int block_size,
                            uint8_t* codes, mnb_stream_t stream) {
    if (!B_packed || !codes || rows < 1 || K < 1) return MNB_ERR_INVALID_ARG;
    if (bits < 1 || bits > 8 || !valid_bs(block_size)) return MNB_ERR_UNSUPPORTED;
    ProjBytes pb;
    int64_t tmp;
    if (!proj_bytes(rows, K, bits, block_size, MNB_F32, &pb) || !mul_ok(rows, K, &tmp))
        return MNB_ERR_SIZE_OVERFLOW;
    return from_cuda(launch_unpack_codes(B_packed, rows, K, bits, block_size, codes,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

mnb_status mnb_quantize_int3(const void* W, mnb_dtype w_dtype, int64_t N, int64_t K, int block_size,
                             uint8_t* B_packed, void* scales, mnb_dtype scale_dtype, mnb_stream_t stream) {
    if (!W || !B_packed || !scales || N < 1 || K < 1) return MNB_ERR_INVALID_ARG;
    if (!valid_dtype(w_dtype) || !valid_dtype(scale_dtype)) return MNB_ERR_INVALID_ARG;
    if (!valid_bs(block_size) || K % block_size != 0) return MNB_ERR_UNSUPPORTED;
    if (!aligned(W, 16) || !aligned(B_packed, 4) || !aligned(scales, dsize(scale_dtype))) return MNB_ERR_INVALID_ARG;
    int64_t wbytes;
    if (!mul_ok(N, K, &wbytes) || !mul_ok(wbytes, int64_t(dsize(w_dtype)), &wbytes)) return MNB_ERR_SIZE_OVERFLOW;
    const int sms = sm_count_current();
    if (sms <= 0) return MNB_ERR_CUDA;
    return from_cuda(launch_quantize_int3(W, w_dtype, N, K, block_size, B_packed, scales, scale_dtype, sms,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

mnb_status mnb_pack_codes(const uint8_t* codes, int64_t rows, int64_t K, int bits, int block_size,
                          uint8_t* B_packed, mnb_stream_t stream) {
    if (!codes || !B_packed || rows < 1 || K < 1) return MNB_ERR_INVALID_ARG;
    if (bits < 1 || bits > 8 || !valid_bs(block_size)) return MNB_ERR_UNSUPPORTED;
    ProjBytes pb;
    int64_t tmp;
    if (!proj_bytes(rows, K, bits, block_size, MNB_F32, &pb) || !mul_ok(rows, K, &tmp))
        return MNB_ERR_SIZE_OVERFLOW;
    return from_cuda(launch_pack_codes(codes, rows, K, bits, block_size, B_packed,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

mnb_status qmoe_route(const float* logits, int64_t T, int64_t E, int k, int normalize_topk, int32_t* topk_idx,
                      float* topk_w, mnb_stream_t stream) {
    if (!logits || !topk_idx || !topk_w) return MNB_ERR_INVALID_ARG;
    if (T < 1 || E < 1 || k < 1 || k > E) return MNB_ERR_INVALID_ARG;
    if (E > 1024) return MNB_ERR_UNSUPPORTED;
    int64_t tmp;
    if (!mul_ok(T, E * 4, &tmp) || T > (int64_t(1) << 31)) return MNB_ERR_SIZE_OVERFLOW;
    return from_cuda(launch_route(logits, MNB_F32, T, E, k, normalize_topk ? 1 : 0, topk_idx, topk_w, nullptr,
                                  MNB_F32, reinterpret_cast<cudaStream_t>(stream), pdl_enabled()));
}

mnb_status qmoe_permute(const int32_t* topk_idx, int64_t T, int k, int64_t E, int32_t* counts, int32_t* offsets,
                        int32_t* perm, mnb_stream_t stream) {
    if (!topk_idx || !counts || !offsets || !perm) return MNB_ERR_INVALID_ARG;
    if (T < 1 || k < 1 || E < 1 || k > E) return MNB_ERR_INVALID_ARG;
    if (E > 1024) return MNB_ERR_UNSUPPORTED;
    if (T * int64_t(k) >= (int64_t(1) << 31)) return MNB_ERR_SIZE_OVERFLOW;
    return from_cuda(launch_permute(topk_idx, T, k, E, counts, offsets, perm, nullptr,
                                    reinterpret_cast<cudaStream_t>(stream), nullptr, nullptr, 0, pdl_enabled()));
}

// ------------------------------------------------------------------- QMoE

mnb_status qmoe_workspace_size(int64_t T, int64_t H, int64_t I, int64_t E, int k, mnb_dtype act_dtype,
                               size_t* bytes) {
    if (!bytes) return MNB_ERR_INVALID_ARG;
    if (T < 1 || H < 1 || I < 1 || E < 1 || k < 1 || k > E) return MNB_ERR_INVALID_ARG;
    if (act_dtype != MNB_F16 && act_dtype != MNB_BF16) return MNB_ERR_UNSUPPORTED;
    if (E > 1024) return MNB_ERR_UNSUPPORTED;
    int64_t b = 0;
    if (!qmoe_workspace_bytes(T, H, I, E, k, &b)) return MNB_ERR_SIZE_OVERFLOW;
    *bytes = static_cast<size_t>(b);
    return MNB_OK;
}

mnb_status qmoe_forward_ex(const void* X, mnb_dtype act_dtype, int64_t T, int64_t H, const void* router_logits,
                           int64_t E, int k, int normalize_topk, const uint8_t* fc1_w, const void* fc1_scales,
                           const uint8_t* fc1_zp, int fc1_bits, const uint8_t* fc2_w, const void* fc2_scales,
                           const uint8_t* fc2_zp, int fc2_bits, int64_t I, int block_size, mnb_fc1_layout fc1_layout,
                           void* Y, void* workspace, size_t workspace_bytes, const qmoe_options* options,
                           mnb_stream_t stream) {
    const qmoe_options none = {nullptr, nullptr, nullptr, MNB_F32, MNB_F32};
    const qmoe_options& op = options ? *options : none;
    if (!X || !router_logits || !fc1_w || !fc1_scales || !fc2_w || !fc2_scales || !Y) return MNB_ERR_INVALID_ARG;
    if (T < 1 || H < 1 || I < 1 || E < 1 || k < 1 || k > E) return MNB_ERR_INVALID_ARG;
    if (fc1_layout != MNB_FC1_INTERLEAVED && fc1_layout != MNB_FC1_CONCAT) return MNB_ERR_INVALID_ARG;
    if (!valid_dtype(op.logits_dtype) || !valid_dtype(op.agg_dtype)) return MNB_ERR_INVALID_ARG;
    if (act_dtype != MNB_F16 && act_dtype != MNB_BF16) return MNB_ERR_UNSUPPORTED;
    if (!valid_bits(fc1_bits) || !valid_bits(fc2_bits) || !valid_bs(block_size)) return MNB_ERR_UNSUPPORTED;
    if (H % block_size != 0 || I % block_size != 0 || E > 1024) return MNB_ERR_UNSUPPORTED;
    if (!aligned(fc1_w, 16) || !aligned(fc2_w, 16) || !aligned(fc1_scales, 16) || !aligned(fc2_scales, 16) ||
        !aligned(X, 2) || !aligned(Y, 2) || !aligned(router_logits, dsize(op.logits_dtype)) ||
        !aligned(op.fc1_bias, 2) || !aligned(op.fc2_bias, 2) || !aligned(op.agg_weights, dsize(op.agg_dtype)))
        return MNB_ERR_UNSUPPORTED;
    ProjBytes p1, p2;
    int64_t w1, w2, tmp;
    if (!proj_bytes(2 * I, H, fc1_bits, block_size, act_dtype, &p1) ||
        !proj_bytes(H, I, fc2_bits, block_size, act_dtype, &p2) || !mul_ok(E, p1.weight, &w1) ||
        !mul_ok(E, p2.weight, &w2) || !mul_ok(T, H * 4, &tmp) || !mul_ok(T, E * 4, &tmp))
        return MNB_ERR_SIZE_OVERFLOW;
    int64_t need = 0;
    if (!qmoe_workspace_bytes(T, H, I, E, k, &need)) return MNB_ERR_SIZE_OVERFLOW;
    if (!workspace || int64_t(workspace_bytes) < need) return MNB_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return MNB_ERR_UNSUPPORTED;
    const int sms = sm_count_current();
    if (sms <= 0) return MNB_ERR_CUDA;

    QmoeArgs q = {};
    q.X = X;
    q.act_dtype = act_dtype;
    q.T = T;
    q.H = H;
    q.I = I;
    q.E = E;
    q.k = k;
    q.normalize = normalize_topk ? 1 : 0;
    q.logits = router_logits;
    q.logits_dtype = op.logits_dtype;
    q.fc1_bias = op.fc1_bias;
    q.fc2_bias = op.fc2_bias;
    q.agg = op.agg_weights;
    q.agg_dtype = op.agg_dtype;
    q.fc1_w = fc1_w;
    q.fc1_s = fc1_scales;
    q.fc1_zp = fc1_zp;
    q.fc1_bits = fc1_bits;
    q.fc2_w = fc2_w;
    q.fc2_s = fc2_scales;
    q.fc2_zp = fc2_zp;
    q.fc2_bits = fc2_bits;
    q.bs = block_size;
    q.fc1_layout = fc1_layout;
    q.x_vec = aligned(X, 16) && (H * 2) % 16 == 0;
    q.Y = Y;
    q.workspace = workspace;
    q.fc1 = {p1.nb, p1.row_bytes, p1.zp_row};
    q.fc2 = {p2.nb, p2.row_bytes, p2.zp_row};
    return from_cuda(launch_qmoe(q, sms, pdl_enabled(), reinterpret_cast<cudaStream_t>(stream)));
}

mnb_status qmoe_forward(const void* X, mnb_dtype act_dtype, int64_t T, int64_t H, const float* router_logits,
                        int64_t E, int k, int normalize_topk, const uint8_t* fc1_w, const void* fc1_scales,
                        const uint8_t* fc1_zp, int fc1_bits, const uint8_t* fc2_w, const void* fc2_scales,
                        const uint8_t* fc2_zp, int fc2_bits, int64_t I, int block_size,
                        mnb_fc1_layout fc1_layout, void* Y, void* workspace, size_t workspace_bytes,
                        mnb_stream_t stream) {
    return qmoe_forward_ex(X, act_dtype, T, H, router_logits, E, k, normalize_topk, fc1_w, fc1_scales, fc1_zp,
                           fc1_bits, fc2_w, fc2_scales, fc2_zp, fc2_bits, I, block_size, fc1_layout, Y, workspace,
                           workspace_bytes, nullptr, stream);
}

// ------------------------------------------------------ host validation

static double host_scale(const void* s, int dt, int64_t i, bool* finite, bool* negative) {
    if (dt == MNB_F32) {
        float f;
        std::memcpy(&f, static_cast<const char*>(s) + 4 * i, 4);
        *finite = std::isfinite(f);
        *negative = f < 0.f;
        return f;
    }
    uint16_t h;
    std::memcpy(&h, static_cast<const char*>(s) + 2 * i, 2);
    const bool neg_sign = (h >> 15) != 0;
    if (dt == MNB_F16) {
        *finite = ((h >> 10) & 0x1F) != 0x1F;
        *negative = neg_sign && (h & 0x7FFF) != 0;
    } else {
        *finite = ((h >> 7) & 0xFF) != 0xFF;
        *negative = neg_sign && (h & 0x7FFF) != 0;
    }
    return 0.0;
}

mnb_status mnb_validate_host(const uint8_t* B_packed, const void* scales, mnb_dtype scale_dtype,
                             const uint8_t* zero_points, int64_t N, int64_t K, int bits, int block_size) {
    if (!B_packed || !scales || N < 1 || K < 1) return MNB_ERR_INVALID_ARG;
    if (!valid_dtype(scale_dtype)) return MNB_ERR_INVALID_ARG;
    if (!valid_bits_any(bits) || !valid_bs(block_size)) return MNB_ERR_UNSUPPORTED;
    ProjBytes pb;
    if (!proj_bytes(N, K, bits, block_size, scale_dtype, &pb)) return MNB_ERR_SIZE_OVERFLOW;
    for (int64_t i = 0; i < N * pb.nb; ++i) {
        bool fin = true, neg = false;
        host_scale(scales, scale_dtype, i, &fin, &neg);
        if (!fin || neg) return MNB_ERR_CONTENT;
    }
    // padding: weight stream bits [K*bits, row_bytes*8) and zero-point stream bits [nb*bits, zp_row*8)
    auto padding_clear = [](const uint8_t* row, int64_t first_bit, int64_t nbytes) {
        for (int64_t bit = first_bit; bit < nbytes * 8; ++bit)
            if ((row[bit >> 3] >> (bit & 7)) & 1) return false;
        return true;
    };
    for (int64_t n = 0; n < N; ++n) {
        if (!padding_clear(B_packed + n * pb.row_bytes, K * bits, pb.row_bytes)) return MNB_ERR_CONTENT;
        if (zero_points && !padding_clear(zero_points + n * pb.zp_row, pb.nb * bits, pb.zp_row))
            return MNB_ERR_CONTENT;
    }
    return MNB_OK;
}

}  // extern "C"
