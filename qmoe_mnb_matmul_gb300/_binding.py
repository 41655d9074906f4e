"""ctypes binding of libmnb.so: the C entry points of include/mnb.h under the
same names.  Argument marshalling only -- every step of every call runs in the
library's CUDA kernels.  There is no fallback: if the library has not been
built, loading it raises.

Tensors are torch tensors on the current CUDA device (contiguous); raw device
pointers may be passed as ints instead.  ``stream`` is a torch.cuda.Stream, a
raw cudaStream_t handle (int), or None for torch's current stream.
"""
from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
DEFAULT_LIB = os.path.join(HERE, "_build", "libmnb.so")
HEADER = os.path.join(ROOT, "include", "mnb.h")

STATUS = {0: "MNB_OK", 1: "MNB_ERR_INVALID_ARG", 2: "MNB_ERR_UNSUPPORTED", 3: "MNB_ERR_SIZE_OVERFLOW",
          4: "MNB_ERR_WORKSPACE", 5: "MNB_ERR_CUDA", 6: "MNB_ERR_TIMEOUT", 7: "MNB_ERR_CONTENT"}
F32, F16, BF16 = 0, 1, 2
FC1_INTERLEAVED, FC1_CONCAT = 0, 1


class PrepackedDesc(ctypes.Structure):
    """mnb_prepacked_desc: the host copy of a prepacked buffer's header."""
    _fields_ = [("magic", ctypes.c_uint32), ("version", ctypes.c_uint32), ("N", ctypes.c_int64),
                ("K", ctypes.c_int64), ("bits", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("scale_dtype", ctypes.c_int32), ("has_zp", ctypes.c_int32), ("row_stride", ctypes.c_int64),
                ("scale_offset", ctypes.c_int64), ("zp_offset", ctypes.c_int64), ("bytes", ctypes.c_int64),
                ("identity", ctypes.c_uint64)]


class MnbError(RuntimeError):
    def __init__(self, status: int, call: str):
        super().__init__(f"{call} failed: {STATUS.get(status, status)}")
        self.status = status
        self.call = call


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int
_SZ = ctypes.c_size_t

_SIGNATURES = {
    "mnb_matmul_workspace_size": [_I64, _I64, _I64, _I, _I, _I, ctypes.POINTER(_SZ)],
    "mnb_matmul": [_P, _I, _I64, _I64, _P, _P, _I, _P, _I64, _I, _I, _P, _I, _P, _SZ, _P],
    "mnb_matmul_int8a": [_P, _I, _I64, _I64, _P, _P, _I, _P, _I64, _I, _I, _P, _I, _P],
    "mnb_gate_up_swiglu": [_P, _I, _I64, _I64, _P, _P, _I, _P, _I64, _I, _I, _I, _P, _I, _P],
    "mnb_prepack_size": [_I64, _I64, _I, _I, _I, _I, ctypes.POINTER(_SZ)],
    "mnb_prepack": [_P, _P, _I, _P, _I64, _I64, _I, _I, ctypes.c_uint64, _P, _SZ, _P, _P],
    "mnb_matmul_prepacked": [_P, _I, _I64, _I64, _P, _P, _P, _I, _P],
    "qmoe_workspace_size": [_I64, _I64, _I64, _I64, _I, _I, ctypes.POINTER(_SZ)],
    "qmoe_forward": [_P, _I, _I64, _I64, _P, _I64, _I, _I, _P, _P, _P, _I, _P, _P, _P, _I, _I64, _I, _I,
                     _P, _P, _SZ, _P],
    "qmoe_forward_ex": [_P, _I, _I64, _I64, _P, _I64, _I, _I, _P, _P, _P, _I, _P, _P, _P, _I, _I64, _I, _I,
                        _P, _P, _SZ, _P, _P],
    "qmoe_forward_static": [_P, _I, _I64, _I64, _P, _I64, _I, _I, _P, _P, _P, _I, _P, _P, _P, _I, _I64, _I, _I,
                            _P, _P],
    "qmoe_route": [_P, _I64, _I64, _I, _I, _P, _P, _P],
    "qmoe_permute": [_P, _I64, _I, _I64, _P, _P, _P, _P],
    "mnb_unpack_codes": [_P, _I64, _I64, _I, _I, _P, _P],
    "mnb_pack_codes": [_P, _I64, _I64, _I, _I, _P, _P],
    "mnb_quantize_int3": [_P, _I, _I64, _I64, _I, _P, _P, _I, _P],
    "mnb_validate_host": [_P, _P, _I, _P, _I64, _I64, _I, _I],
    "mnb_get_last_device_error": [_P],
    "mnb_diag_wait_timeout": [ctypes.c_uint64, _P],
    "mnb_status_string": [_I],
}

_LIB = None


def header_functions() -> list[str]:
    """Names of the functions include/mnb.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)


def load_library(path: str | None = None):
    global _LIB
    if _LIB is None:
        p = path or os.environ.get("MNB_LIBRARY", DEFAULT_LIB)
        if not os.path.exists(p):
            raise ImportError(f"libmnb.so is not built ({p}); run __graft_entry__.build()")
        lib = ctypes.CDLL(p)
        for name, args in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_char_p if name == "mnb_status_string" else _I
        _LIB = lib
    return _LIB


def library_path() -> str:
    return DEFAULT_LIB


# ------------------------------------------------------------- marshalling

def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.float16:
        return F16
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, call: str):
    if status != 0:
        raise MnbError(status, call)


# ------------------------------------------------------------- entry points

def mnb_status_string(status: int) -> str:
    return load_library().mnb_status_string(status).decode()


def mnb_matmul_workspace_size(M, K, N, bits, block_size, a_dtype=F32) -> int:
    out = _SZ(0)
    _check(load_library().mnb_matmul_workspace_size(M, K, N, bits, block_size, a_dtype, ctypes.byref(out)),
           "mnb_matmul_workspace_size")
    return out.value


def mnb_matmul(A, B_packed, scales, zero_points, N, bits, block_size, Y, workspace=None, stream=None,
               *, K=None, M=None, a_dtype=None, scale_dtype=None, y_dtype=None, check=True):
    """Y[M, N] = A[M, K] . dequant(B_packed, scales, zero_points)^T."""
    if K is None:
        K = A.shape[-1]
    if M is None:
        M = A.numel() // K
    a_dtype = _dtype_code(A) if a_dtype is None else a_dtype
    scale_dtype = _dtype_code(scales) if scale_dtype is None else scale_dtype
    y_dtype = _dtype_code(Y) if y_dtype is None else y_dtype
    if workspace is None:  # the workspace the library can use (split-K partial sums), if any
        need = mnb_matmul_workspace_size(M, K, N, bits, block_size, a_dtype)
        if need:
            import torch
            workspace = torch.empty(need, dtype=torch.uint8, device=A.device)
    ws_bytes = 0 if workspace is None or isinstance(workspace, int) else workspace.numel() * workspace.element_size()
    st = load_library().mnb_matmul(_ptr(A), a_dtype, M, K, _ptr(B_packed), _ptr(scales), scale_dtype,
                                   _ptr(zero_points), N, bits, block_size, _ptr(Y), y_dtype, _ptr(workspace),
                                   ws_bytes, _stream(stream))
    if check:
        _check(st, "mnb_matmul")
    return st


def mnb_matmul_int8a(A, B_packed, scales, zero_points, N, bits, block_size, Y, stream=None, *, K=None, M=None,
                     a_dtype=None, scale_dtype=None, y_dtype=None, check=True):
    """Y[M, N] = A . dequant(B)^T with A quantised per (row, block) to int8 (accuracy_level=4)."""
    if K is None:
        K = A.shape[-1]
    if M is None:
        M = A.numel() // K
    a_dtype = _dtype_code(A) if a_dtype is None else a_dtype
    scale_dtype = _dtype_code(scales) if scale_dtype is None else scale_dtype
    y_dtype = _dtype_code(Y) if y_dtype is None else y_dtype
    st = load_library().mnb_matmul_int8a(_ptr(A), a_dtype, M, K, _ptr(B_packed), _ptr(scales), scale_dtype,
                                         _ptr(zero_points), N, bits, block_size, _ptr(Y), y_dtype, _stream(stream))
    if check:
        _check(st, "mnb_matmul_int8a")
    return st


def mnb_gate_up_swiglu(A, B_packed, scales, zero_points, I, bits, block_size, Y, stream=None, *,
                       layout=FC1_INTERLEAVED, K=None, M=None, a_dtype=None, scale_dtype=None, y_dtype=None,
                       check=True):
    """Y[M, I] = silu(A . Wgate^T) * (A . Wup^T) from the fused gate/up weight [2I, K]."""
    if K is None:
        K = A.shape[-1]
    if M is None:
        M = A.numel() // K
    a_dtype = _dtype_code(A) if a_dtype is None else a_dtype
    scale_dtype = _dtype_code(scales) if scale_dtype is None else scale_dtype
    y_dtype = _dtype_code(Y) if y_dtype is None else y_dtype
    st = load_library().mnb_gate_up_swiglu(_ptr(A), a_dtype, M, K, _ptr(B_packed), _ptr(scales), scale_dtype,
                                           _ptr(zero_points), I, bits, block_size, layout, _ptr(Y), y_dtype,
                                           _stream(stream))
    if check:
        _check(st, "mnb_gate_up_swiglu")
    return st


def mnb_prepack_size(N, K, bits, block_size, scale_dtype=F32, has_zero_points=False) -> int:
    out = _SZ(0)
    _check(load_library().mnb_prepack_size(N, K, bits, block_size, scale_dtype, int(bool(has_zero_points)),
                                           ctypes.byref(out)), "mnb_prepack_size")
    return out.value


def mnb_prepack(B_packed, scales, zero_points, N, K, bits, block_size, dst, identity=0, stream=None, *,
                scale_dtype=None, dst_bytes=None, check=True):
    """Writes the version-1 prepacked form of a row-local weight into `dst`; returns its
    PrepackedDesc (with check=False: (status, desc))."""
    scale_dtype = _dtype_code(scales) if scale_dtype is None else scale_dtype
    if dst_bytes is None:
        dst_bytes = dst.numel() * dst.element_size()
    desc = PrepackedDesc()
    st = load_library().mnb_prepack(_ptr(B_packed), _ptr(scales), scale_dtype, _ptr(zero_points), N, K, bits,
                                    block_size, ctypes.c_uint64(identity), _ptr(dst), dst_bytes, ctypes.byref(desc),
                                    _stream(stream))
    if not check:
        return st, desc
    _check(st, "mnb_prepack")
    return desc


def mnb_matmul_prepacked(A, desc, prepacked, Y, stream=None, *, K=None, M=None, a_dtype=None, y_dtype=None,
                         check=True):
    """Y[M, N] = A . W^T with W read from a prepacked buffer and its descriptor."""
    if K is None:
        K = A.shape[-1]
    if M is None:
        M = A.numel() // K
    a_dtype = _dtype_code(A) if a_dtype is None else a_dtype
    y_dtype = _dtype_code(Y) if y_dtype is None else y_dtype
    st = load_library().mnb_matmul_prepacked(_ptr(A), a_dtype, M, K, ctypes.byref(desc), _ptr(prepacked), _ptr(Y),
                                             y_dtype, _stream(stream))
    if check:
        _check(st, "mnb_matmul_prepacked")
    return st


def qmoe_workspace_size(T, H, I, E, k, act_dtype=F16) -> int:
    out = _SZ(0)
    _check(load_library().qmoe_workspace_size(T, H, I, E, k, act_dtype, ctypes.byref(out)),
           "qmoe_workspace_size")
    return out.value


def qmoe_forward(X, router_logits, k, normalize_topk, fc1_w, fc1_scales, fc1_zp, fc1_bits, fc2_w, fc2_scales,
                 fc2_zp, fc2_bits, I, block_size, Y, workspace, stream=None, *, fc1_layout=FC1_INTERLEAVED,
                 T=None, H=None, E=None, act_dtype=None, workspace_bytes=None, check=True):
    """One QMoE expert-FFN layer: Y[T, H] from X[T, H] and router_logits[T, E]."""
    if H is None:
        H = X.shape[-1]
    if T is None:
        T = X.numel() // H
    if E is None:
        E = router_logits.shape[-1]
    act_dtype = _dtype_code(X) if act_dtype is None else act_dtype
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    st = load_library().qmoe_forward(_ptr(X), act_dtype, T, H, _ptr(router_logits), E, k, int(bool(normalize_topk)),
                                     _ptr(fc1_w), _ptr(fc1_scales), _ptr(fc1_zp), fc1_bits, _ptr(fc2_w),
                                     _ptr(fc2_scales), _ptr(fc2_zp), fc2_bits, I, block_size, fc1_layout, _ptr(Y),
                                     _ptr(workspace), workspace_bytes, _stream(stream))
    if check:
        _check(st, "qmoe_forward")
    return st


class QmoeOptions(ctypes.Structure):
    """The qmoe_options struct of include/mnb.h (device pointers as ints)."""
    _fields_ = [("fc1_bias", ctypes.c_void_p), ("fc2_bias", ctypes.c_void_p), ("agg_weights", ctypes.c_void_p),
                ("agg_dtype", ctypes.c_int), ("logits_dtype", ctypes.c_int)]


def qmoe_forward_ex(X, router_logits, k, normalize_topk, fc1_w, fc1_scales, fc1_zp, fc1_bits, fc2_w, fc2_scales,
                    fc2_zp, fc2_bits, I, block_size, Y, workspace, stream=None, *, fc1_bias=None, fc2_bias=None,
                    agg_weights=None, fc1_layout=FC1_INTERLEAVED, T=None, H=None, E=None, act_dtype=None,
                    workspace_bytes=None, check=True):
    """qmoe_forward with the optional inputs: FC1/FC2 biases, aggregation weights
    [T, E], router logits of any float dtype (taken from the tensor)."""
    if H is None:
        H = X.shape[-1]
    if T is None:
        T = X.numel() // H
    if E is None:
        E = router_logits.shape[-1]
    act_dtype = _dtype_code(X) if act_dtype is None else act_dtype
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    opts = QmoeOptions(_ptr(fc1_bias), _ptr(fc2_bias), _ptr(agg_weights),
                       _dtype_code(agg_weights) if agg_weights is not None else F32, _dtype_code(router_logits))
    st = load_library().qmoe_forward_ex(_ptr(X), act_dtype, T, H, _ptr(router_logits), E, k, int(bool(normalize_topk)),
                                        _ptr(fc1_w), _ptr(fc1_scales), _ptr(fc1_zp), fc1_bits, _ptr(fc2_w),
                                        _ptr(fc2_scales), _ptr(fc2_zp), fc2_bits, I, block_size, fc1_layout, _ptr(Y),
                                        _ptr(workspace), workspace_bytes, ctypes.byref(opts), _stream(stream))
    if check:
        _check(st, "qmoe_forward_ex")
    return st


def qmoe_forward_static(X, router_logits, k, normalize_topk, fc1_w, fc1_scales, fc1_zp, fc1_bits, fc2_w,
                        fc2_scales, fc2_zp, fc2_bits, I, block_size, Y, stream=None, *, fc1_layout=FC1_INTERLEAVED,
                        T=None, H=None, E=None, act_dtype=None, check=True):
    """qmoe_forward with the library's fixed 8 MiB scratch instead of a caller workspace."""
    if H is None:
        H = X.shape[-1]
    if T is None:
        T = X.numel() // H
    if E is None:
        E = router_logits.shape[-1]
    act_dtype = _dtype_code(X) if act_dtype is None else act_dtype
    st = load_library().qmoe_forward_static(_ptr(X), act_dtype, T, H, _ptr(router_logits), E, k,
                                            int(bool(normalize_topk)), _ptr(fc1_w), _ptr(fc1_scales), _ptr(fc1_zp),
                                            fc1_bits, _ptr(fc2_w), _ptr(fc2_scales), _ptr(fc2_zp), fc2_bits, I,
                                            block_size, fc1_layout, _ptr(Y), _stream(stream))
    if check:
        _check(st, "qmoe_forward_static")
    return st


def qmoe_route(logits, k, normalize_topk, topk_idx, topk_w, stream=None, *, T=None, E=None, check=True):
    if E is None:
        E = logits.shape[-1]
    if T is None:
        T = logits.numel() // E
    st = load_library().qmoe_route(_ptr(logits), T, E, k, int(bool(normalize_topk)), _ptr(topk_idx), _ptr(topk_w),
                                   _stream(stream))
    if check:
        _check(st, "qmoe_route")
    return st


def qmoe_permute(topk_idx, E, counts, offsets, perm, stream=None, *, T=None, k=None, check=True):
    if k is None:
        k = topk_idx.shape[-1]
    if T is None:
        T = topk_idx.numel() // k
    st = load_library().qmoe_permute(_ptr(topk_idx), T, k, E, _ptr(counts), _ptr(offsets), _ptr(perm),
                                     _stream(stream))
    if check:
        _check(st, "qmoe_permute")
    return st


def mnb_unpack_codes(B_packed, rows, K, bits, block_size, codes, stream=None, *, check=True):
    st = load_library().mnb_unpack_codes(_ptr(B_packed), rows, K, bits, block_size, _ptr(codes), _stream(stream))
    if check:
        _check(st, "mnb_unpack_codes")
    return st


def mnb_pack_codes(codes, rows, K, bits, block_size, B_packed, stream=None, *, check=True):
    st = load_library().mnb_pack_codes(_ptr(codes), rows, K, bits, block_size, _ptr(B_packed), _stream(stream))
    if check:
        _check(st, "mnb_pack_codes")
    return st


def mnb_quantize_int3(W, block_size, scale_dtype, B_packed=None, scales=None, stream=None, *, check=True):
    """INT3 quantisation of the 2-D tensor W [N, K] (f32/f16/bf16); returns
    (B_packed uint8 [N, K/bs, 3*bs/8], scales [N, K/bs] in scale_dtype), allocating
    the outputs with torch when they are not given."""
    import torch
    N, K = W.shape
    nb = K // block_size
    sdt = {F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}[scale_dtype]
    if B_packed is None:
        B_packed = torch.empty((N, nb, 3 * block_size // 8), dtype=torch.uint8, device=W.device)
    if scales is None:
        scales = torch.empty((N, nb), dtype=sdt, device=W.device)
    st = load_library().mnb_quantize_int3(_ptr(W), _dtype_code(W), N, K, block_size, _ptr(B_packed), _ptr(scales),
                                          scale_dtype, _stream(stream))
    if check:
        _check(st, "mnb_quantize_int3")
    return B_packed, scales


def mnb_validate_host(B_packed, scales, scale_dtype, zero_points, N, K, bits, block_size) -> int:
    """Host buffers (numpy arrays or ctypes-compatible objects); returns the status code."""
    def hp(a):
        if a is None:
            return None
        return a.ctypes.data_as(ctypes.c_void_p)
    return load_library().mnb_validate_host(hp(B_packed), hp(scales), scale_dtype, hp(zero_points), N, K, bits,
                                            block_size)


def mnb_get_last_device_error(stream=None) -> int:
    return load_library().mnb_get_last_device_error(_stream(stream))


def mnb_diag_wait_timeout(limit_ns: int, stream=None, *, check=True) -> int:
    """Enqueue the diagnostic kernel whose bounded wait runs out after limit_ns."""
    st = load_library().mnb_diag_wait_timeout(int(limit_ns), _stream(stream))
    if check:
        _check(st, "mnb_diag_wait_timeout")
    return st
