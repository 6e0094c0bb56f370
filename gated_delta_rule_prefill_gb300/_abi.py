"""ctypes view of libgdr.so (the C ABI declared in include/gdr.h).  Argument marshalling only."""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdr.so")

GDR_OK, GDR_ERR_INVALID_ARG, GDR_ERR_UNSUPPORTED, GDR_ERR_CUDA, GDR_ERR_DEVICE_CHECK = range(5)
GDR_F32, GDR_BF16 = 0, 1
GDR_GATE_SCALAR, GDR_GATE_CHANNEL = 0, 1
GDR_FLAG_FORCE_SIMT = 1
GDR_FLAG_NO_CLUSTER = 2
GDR_FLAG_PREFER_QUEUE = 4
GDR_FLAG_LAYER_PROLOGUE = 8
GDR_DEVCHECK_OK, GDR_DEVCHECK_SEQLENS, GDR_DEVCHECK_TIMEOUT = 0, 1, 2

# every symbol include/gdr.h declares
EXPORTS = ("gdr_prefill", "gdr_prefill_workspace_size", "gdr_decode_step", "gdr_linear_attn",
           "gdr_workspace_status", "gdr_status_string", "gdr_prefill_noalloc", "gdr_prefill_host",
           "gdr_prefill_host_buffer_size", "gdr_gated_linear_attn",
           "gdr_prefill_output_gate", "gdr_layer_prologue", "gdr_normalized_linear_attn",
           "gdr_gated_linear_decode_step", "gdr_normalized_linear_decode_step",
           "gdr_query_device_status", "gdr_check_wait_timeout")
GDR_NOALLOC_MAX_SEQS = 4096


class GdrShape(ctypes.Structure):
    _fields_ = [("n_seqs", ctypes.c_int32), ("H", ctypes.c_int32),
                ("total_tokens", ctypes.c_int64), ("d_k", ctypes.c_int32),
                ("d_v", ctypes.c_int32), ("dtype", ctypes.c_int32), ("gate", ctypes.c_int32),
                ("chunk_size", ctypes.c_int32), ("flags", ctypes.c_int32)]


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libgdr.so; raises if it has not been built (there is no fallback path)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError("libgdr.so is not built (%s); run __graft_entry__.build() or "
                           "python gated_delta_rule_prefill_gb300/build.py" % path)
    lib = ctypes.CDLL(path)
    P, S = ctypes.c_void_p, ctypes.POINTER(GdrShape)
    lib.gdr_prefill.argtypes = [S, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P]
    lib.gdr_prefill.restype = ctypes.c_int
    lib.gdr_linear_attn.argtypes = [S, P, P, P, P, P, P, P, P, ctypes.c_size_t, P]
    lib.gdr_linear_attn.restype = ctypes.c_int
    lib.gdr_prefill_output_gate.argtypes = [S, P, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P]
    lib.gdr_prefill_output_gate.restype = ctypes.c_int
    lib.gdr_gated_linear_attn.argtypes = [S, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P]
    lib.gdr_gated_linear_attn.restype = ctypes.c_int
    lib.gdr_normalized_linear_attn.argtypes = [S, P, P, P, ctypes.c_float, P, P, P, P, P, P, P,
                                               ctypes.c_size_t, P]
    lib.gdr_normalized_linear_attn.restype = ctypes.c_int
    lib.gdr_gated_linear_decode_step.argtypes = [S, P, P, P, P, P, P, P]
    lib.gdr_gated_linear_decode_step.restype = ctypes.c_int
    lib.gdr_normalized_linear_decode_step.argtypes = [S, P, P, P, ctypes.c_float, P, P, P, P]
    lib.gdr_normalized_linear_decode_step.restype = ctypes.c_int
    lib.gdr_layer_prologue.argtypes = [S, P, P, P, P, P, P, P, P, P]
    lib.gdr_layer_prologue.restype = ctypes.c_int
    lib.gdr_decode_step.argtypes = [S, P, P, P, P, P, P, P, P]
    lib.gdr_decode_step.restype = ctypes.c_int
    lib.gdr_prefill_workspace_size.argtypes = [S]
    lib.gdr_prefill_workspace_size.restype = ctypes.c_size_t
    lib.gdr_workspace_status.argtypes = [P, P, ctypes.POINTER(ctypes.c_int32)]
    lib.gdr_workspace_status.restype = ctypes.c_int
    lib.gdr_query_device_status.argtypes = [P]
    lib.gdr_query_device_status.restype = ctypes.c_int
    lib.gdr_check_wait_timeout.argtypes = [P, ctypes.c_uint64, P]
    lib.gdr_check_wait_timeout.restype = ctypes.c_int
    lib.gdr_prefill_noalloc.argtypes = [S, P, P, P, P, P, P, P, P, P, P]
    lib.gdr_prefill_noalloc.restype = ctypes.c_int
    lib.gdr_prefill_host.argtypes = [S, P, P, P, P, P, P, P, P, P, ctypes.c_int64, P,
                                     ctypes.c_size_t, P]
    lib.gdr_prefill_host.restype = ctypes.c_int
    lib.gdr_prefill_host_buffer_size.argtypes = [S, ctypes.c_int64]
    lib.gdr_prefill_host_buffer_size.restype = ctypes.c_size_t
    lib.gdr_status_string.argtypes = [ctypes.c_int]
    lib.gdr_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load().gdr_status_string(code).decode()


class GdrError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__("%s: %s" % (where, status_string(code)))
        self.code = code
