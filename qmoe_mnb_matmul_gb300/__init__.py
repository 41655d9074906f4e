"""GB300-native block-quantized weight-only matmul (MatMulNBits INT4/INT3) and
the QMoE expert FFN built on it.

The compute lives in the CUDA library ``_build/libmnb.so`` (hand-written
sm_103a kernels behind the C ABI of ``include/mnb.h``); this package is its
thin ctypes binding.  Build it with ``__graft_entry__.build()`` or
``python -m qmoe_mnb_matmul_gb300._build``.
"""
from ._binding import (BF16, F16, F32, FC1_CONCAT, FC1_INTERLEAVED, MnbError, PrepackedDesc,  # noqa: F401
                       QmoeOptions, header_functions, library_path, load_library, mnb_diag_wait_timeout,
                       mnb_gate_up_swiglu, mnb_get_last_device_error, mnb_matmul, mnb_matmul_int8a,
                       mnb_matmul_prepacked, mnb_matmul_workspace_size, mnb_pack_codes, mnb_prepack,
                       mnb_prepack_size, mnb_quantize_int3, mnb_status_string, mnb_unpack_codes, mnb_validate_host,
                       qmoe_forward, qmoe_forward_ex, qmoe_forward_static, qmoe_permute, qmoe_route,
                       qmoe_workspace_size)

__all__ = ["mnb_matmul", "mnb_matmul_int8a", "mnb_gate_up_swiglu", "mnb_matmul_workspace_size", "mnb_prepack",
           "mnb_prepack_size", "mnb_matmul_prepacked", "PrepackedDesc", "qmoe_forward", "qmoe_forward_ex",
           "qmoe_forward_static", "qmoe_workspace_size", "qmoe_route", "qmoe_permute", "QmoeOptions",
           "mnb_unpack_codes", "mnb_pack_codes", "mnb_quantize_int3", "mnb_validate_host",
           "mnb_get_last_device_error", "mnb_diag_wait_timeout", "mnb_status_string", "load_library",
           "library_path", "MnbError"]
