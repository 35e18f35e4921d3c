"""ctypes binding of libxhc.so (include/xhc.h): argument marshalling only.

Tensors are passed as raw device pointers (``tensor.data_ptr()``) together
with the current CUDA stream; every step of the update runs in the library's
kernels.  Importing this module fails loudly when the library is missing.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
# XHC_DEBUG=1 loads the debug build (bounds-checked streaming kernels)
DEBUG = os.environ.get("XHC_DEBUG") == "1"
LIB_PATH = os.path.join(_HERE, "libxhc_debug.so" if DEBUG else "libxhc.so")

XHC_F32, XHC_BF16 = 0, 1
STATUS = {0: "XHC_OK", 1: "XHC_ERR_SHAPE", 2: "XHC_ERR_INDEX", 3: "XHC_ERR_ALIGN", 4: "XHC_ERR_DTYPE",
          5: "XHC_ERR_WORKSPACE", 6: "XHC_ERR_CUDA", 7: "XHC_ERR_TIMEOUT", 8: "XHC_ERR_ARG"}

EXPORTS = ("xhc_status_string", "xhc_last_cuda_error", "xhc_device_status", "xhc_set_wait_limit_ns",
           "xhc_debug_starve_next_projection", "xhc_debug_record", "xhc_debug_selftest", "xhc_num_logits", "xhc_coeffs", "xhc_tfa",
           "xhc_sparse_update", "xhc_fwd_workspace_bytes", "xhc_fwd_workspace_need", "xhc_sublayer_fwd", "xhc_sublayer_fwd_noalloc", "xhc_bwd_workspace_bytes",
           "xhc_sublayer_bwd", "xhc_fwd_routed_workspace_bytes", "xhc_sublayer_fwd_routed",
           "xhc_bwd_routed_workspace_bytes", "xhc_sublayer_bwd_routed", "xhc_hres_active_weights", "xhc_hres_active_grad", "xhc_copy", "xhc_timing_enable",
           "xhc_timing_collect", "xhc_stack_fwd_workspace_bytes", "xhc_stack_fwd")


class XhcShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("S", ctypes.c_int), ("N", ctypes.c_int), ("C", ctypes.c_int),
                ("k", ctypes.c_int), ("dtype", ctypes.c_int), ("sinkhorn_iters", ctypes.c_int),
                ("eps", ctypes.c_float), ("gram_schmidt", ctypes.c_int)]


class XhcError(RuntimeError):
    def __init__(self, fn, status, lib):
        msg = lib.xhc_status_string(status).decode()
        detail = ""
        if status == 6:
            detail = f" (cudaError {lib.xhc_last_cuda_error()})"
        super().__init__(f"{fn}: {STATUS.get(status, status)}: {msg}{detail}")
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{os.path.basename(LIB_PATH)} not built at {LIB_PATH}; run "
                          "`python -m residual_stream_expansion_xhc_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    sh = ctypes.POINTER(XhcShape)
    lib.xhc_status_string.restype = ctypes.c_char_p
    lib.xhc_status_string.argtypes = [I]
    lib.xhc_last_cuda_error.restype = I
    lib.xhc_last_cuda_error.argtypes = []
    lib.xhc_device_status.restype = I
    lib.xhc_device_status.argtypes = [P]
    lib.xhc_set_wait_limit_ns.restype = I
    lib.xhc_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
    lib.xhc_debug_starve_next_projection.restype = I
    lib.xhc_debug_starve_next_projection.argtypes = []
    lib.xhc_debug_record.restype = I
    lib.xhc_debug_record.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), ctypes.POINTER(ctypes.c_ulonglong)]
    lib.xhc_debug_selftest.restype = I
    lib.xhc_debug_selftest.argtypes = [P, P, P]
    lib.xhc_num_logits.restype = I
    lib.xhc_num_logits.argtypes = [sh]
    lib.xhc_coeffs.restype = I
    lib.xhc_coeffs.argtypes = [sh, P, P, P, P, P, P, P, P]
    lib.xhc_tfa.restype = I
    lib.xhc_tfa.argtypes = [sh, P, P, P, P, P, P]
    lib.xhc_sparse_update.restype = I
    lib.xhc_sparse_update.argtypes = [sh, P, P, P, P, P, P, P, P, P, P]
    lib.xhc_fwd_workspace_bytes.restype = Z
    lib.xhc_fwd_workspace_bytes.argtypes = [sh]
    lib.xhc_fwd_workspace_need.restype = Z
    lib.xhc_fwd_workspace_need.argtypes = [sh, I]
    lib.xhc_sublayer_fwd.restype = I
    lib.xhc_sublayer_fwd.argtypes = [sh, P, P, P, P, P, P, P, P, P, P, P, P, Z, P]
    lib.xhc_sublayer_fwd_noalloc.restype = I
    lib.xhc_sublayer_fwd_noalloc.argtypes = [sh, P, P, P, P, P, P, P, P, P, P, P, P]
    lib.xhc_bwd_workspace_bytes.restype = Z
    lib.xhc_bwd_workspace_bytes.argtypes = [sh]
    lib.xhc_sublayer_bwd.restype = I
    lib.xhc_sublayer_bwd.argtypes = [sh, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, Z, P]
    lib.xhc_fwd_routed_workspace_bytes.restype = Z
    lib.xhc_fwd_routed_workspace_bytes.argtypes = [sh]
    lib.xhc_sublayer_fwd_routed.restype = I
    lib.xhc_sublayer_fwd_routed.argtypes = [sh, P, P, P, P, P, P, P, P, P, I, P, P, P, P, P, P, Z, P]
    lib.xhc_bwd_routed_workspace_bytes.restype = Z
    lib.xhc_bwd_routed_workspace_bytes.argtypes = [sh]
    lib.xhc_sublayer_bwd_routed.restype = I
    lib.xhc_sublayer_bwd_routed.argtypes = [sh, P, P, P, P, P, P, P, P, P, I, P, P, P, P, P, P, P, P, P, P, P, P, P, Z,
                                            P]
    lib.xhc_hres_active_weights.restype = I
    lib.xhc_hres_active_weights.argtypes = [sh, P, P, P, P, P]
    lib.xhc_hres_active_grad.restype = I
    lib.xhc_hres_active_grad.argtypes = [sh, P, P, P, P]
    lib.xhc_stack_fwd_workspace_bytes.restype = Z
    lib.xhc_stack_fwd_workspace_bytes.argtypes = [sh]
    lib.xhc_stack_fwd.restype = I
    lib.xhc_stack_fwd.argtypes = [sh, I, P, P, P, P, P, P, P, P, P, P, Z, P]
    lib.xhc_copy.restype = I
    lib.xhc_copy.argtypes = [P, P, Z, P]
    lib.xhc_timing_enable.restype = I
    lib.xhc_timing_enable.argtypes = [I]
    lib.xhc_timing_collect.restype = I
    lib.xhc_timing_collect.argtypes = [ctypes.c_char_p, ctypes.POINTER(I), ctypes.POINTER(ctypes.c_float), I]
    return lib


LIB = _load()
