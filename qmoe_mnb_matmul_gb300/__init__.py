"""GB300-native block-quantized weight-only matmul (MatMulNBits INT4/INT3) and
the QMoE expert FFN built on it.

The compute lives in the CUDA library ``_build/libmnb.so`` (hand-written
sm_103a kernels behind the C ABI of ``include/mnb.h``); this package is its
thin ctypes binding.  Build it with ``__graft_entry__.build()`` or
``python -m qmoe_mnb_matmul_gb300._build``.
"""
from ._binding import (BF16, F16, F32, FC1_CONCAT, FC1_INTERLEAVED, MnbError, header_functions,  # noqa: F401
                       library_path, load_library, mnb_diag_wait_timeout, mnb_get_last_device_error, mnb_gate_up_swiglu, mnb_matmul, mnb_matmul_int8a,
                       mnb_matmul_workspace_size, mnb_pack_codes, mnb_quantize_int3, mnb_status_string, mnb_unpack_codes,
                       mnb_validate_host,
                       qmoe_forward, qmoe_forward_ex, qmoe_forward_static, QmoeOptions, qmoe_permute, qmoe_route, qmoe_workspace_size)

__all__ = ["mnb_matmul", "mnb_matmul_int8a", "mnb_gate_up_swiglu", "mnb_matmul_workspace_size", "qmoe_forward", "qmoe_forward_ex", "qmoe_forward_static", "qmoe_workspace_size", "qmoe_route",
           "qmoe_permute", "mnb_unpack_codes", "mnb_pack_codes", "mnb_quantize_int3", "mnb_validate_host", "mnb_get_last_device_error", "mnb_diag_wait_timeout",
           "mnb_status_string", "load_library", "library_path", "MnbError"]
