"""ctypes handle on the in-tree CUDA library ``libgla.so`` (C ABI in include/gla.h).

Loading never falls back to anything: if the library is missing or cannot be
loaded the error says so and names the build command.
"""

from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgla.so")

# Status codes (enum gla_status in include/gla.h).
GLA_OK = 0
GLA_ERR_ARG = 1
GLA_ERR_SHAPE = 2
GLA_ERR_DEVICE = 3
GLA_ERR_LAUNCH = 4
GLA_ERR_TIMEOUT = 5
GLA_ERR_ALLOC = 6
GLA_ERR_SCRATCH = 7

EXPORTED = ("gla_chunk_fwd", "gla_chunk_fwd_ex", "gla_chunk_fwd_plan", "gla_chunk_fwd_noalloc",
            "gla_chunk_fwd_debug",
            "gla_chunk_fwd_host", "gla_chunk_fwd_varlen", "gla_chunk_fwd_varlen_ex",
            "gla_chunk_fwd_varlen_plan", "gla_chunk_bwd", "gla_chunk_bwd_ex",
            "gla_chunk_bwd_plan", "gla_chunk_bwd_varlen", "gla_chunk_bwd_varlen_ex",
            "gla_gdn_fwd", "gla_gdn_chunk_fwd", "gla_recurrent_step", "gla_status_string",
            "gla_last_device_status", "gla_version")


class GlaChunkOptions(ctypes.Structure):
    _fields_ = [("segments", ctypes.c_int), ("dv_tile", ctypes.c_int),
                ("force_exact", ctypes.c_int), ("cta_pair", ctypes.c_int),
                ("gate_per_head", ctypes.c_int), ("reserved", ctypes.c_int * 3)]


class GlaChunkDebug(ctypes.Structure):
    """gla_chunk_debug (include/gla.h): test instrumentation of the chunked forward."""
    _fields_ = [("gamma", ctypes.c_void_p), ("block_len", ctypes.c_void_p),
                ("wait_limit_us", ctypes.c_uint), ("withhold_v", ctypes.c_int)]


class GlaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


_lock = threading.Lock()
_lib: ctypes.CDLL | None = None


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    vp, fp, i, f = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.gla_chunk_fwd.argtypes = [vp, vp, vp, fp, f, fp, vp, fp, i, i, i, i, i, vp]
    lib.gla_chunk_fwd.restype = i
    lib.gla_chunk_fwd_ex.argtypes = [vp, vp, vp, fp, f, fp, vp, fp, i, i, i, i, i,
                                     ctypes.POINTER(GlaChunkOptions), vp]
    lib.gla_chunk_fwd_ex.restype = i
    lib.gla_chunk_fwd_noalloc.argtypes = [vp, vp, vp, fp, f, fp, vp, fp, i, i, i, i, i,
                                          ctypes.POINTER(GlaChunkOptions), vp]
    lib.gla_chunk_fwd_noalloc.restype = i
    lib.gla_chunk_fwd_debug.argtypes = [vp, vp, vp, fp, f, fp, vp, fp, i, i, i, i, i,
                                        ctypes.POINTER(GlaChunkOptions),
                                        ctypes.POINTER(GlaChunkDebug), vp]
    lib.gla_chunk_fwd_debug.restype = i
    lib.gla_chunk_fwd_host.argtypes = [vp, vp, vp, fp, f, fp, vp, fp, i, i, i, i, i, vp]
    lib.gla_chunk_fwd_host.restype = i
    ip = ctypes.POINTER(ctypes.c_int)
    lib.gla_chunk_fwd_varlen_plan.argtypes = [ip, i, i, i, i, i, ctypes.POINTER(GlaChunkOptions),
                                              ip, ip, ip, ctypes.POINTER(ctypes.c_ulong)]
    lib.gla_chunk_fwd_varlen_plan.restype = i
    lib.gla_chunk_fwd_varlen.argtypes = [vp, vp, vp, fp, f, fp, vp, fp, ip, i, i, i, i, i, vp]
    lib.gla_chunk_fwd_varlen.restype = i
    lib.gla_chunk_fwd_varlen_ex.argtypes = [vp, vp, vp, fp, f, fp, vp, fp, ip, i, i, i, i, i,
                                            ctypes.POINTER(GlaChunkOptions), vp]
    lib.gla_chunk_fwd_varlen_ex.restype = i
    lib.gla_chunk_fwd_plan.argtypes = [i, i, i, i, i, ctypes.POINTER(GlaChunkOptions), ip, ip, ip,
                                       ctypes.POINTER(ctypes.c_ulong)]
    lib.gla_chunk_fwd_plan.restype = i
    bwd = [vp, vp, vp, fp, f, fp, vp, fp, vp, vp, vp, fp, fp, i, i, i, i, i]
    lib.gla_chunk_bwd.argtypes = bwd + [vp]
    lib.gla_chunk_bwd.restype = i
    lib.gla_chunk_bwd_ex.argtypes = bwd + [ctypes.POINTER(GlaChunkOptions), vp]
    lib.gla_chunk_bwd_ex.restype = i
    lib.gla_chunk_bwd_plan.argtypes = [i, i, i, i, i, ip, ip, ctypes.POINTER(ctypes.c_ulong)]
    bwdv = [vp, vp, vp, fp, f, fp, vp, fp, vp, vp, vp, fp, fp, ip, i, i, i, i, i]
    lib.gla_chunk_bwd_varlen.argtypes = bwdv + [vp]
    lib.gla_chunk_bwd_varlen.restype = i
    lib.gla_chunk_bwd_varlen_ex.argtypes = bwdv + [ctypes.POINTER(GlaChunkOptions), vp]
    lib.gla_chunk_bwd_varlen_ex.restype = i
    lib.gla_chunk_bwd_plan.restype = i
    lib.gla_gdn_fwd.argtypes = [vp, vp, vp, fp, fp, f, fp, vp, fp, i, i, i, i, i, vp]
    lib.gla_gdn_fwd.restype = i
    lib.gla_gdn_chunk_fwd.argtypes = [vp, vp, vp, fp, fp, f, fp, vp, fp, i, i, i, i, i, vp]
    lib.gla_gdn_chunk_fwd.restype = i
    lib.gla_recurrent_step.argtypes = [vp, vp, vp, fp, f, fp, vp, i, i, i, i, vp]
    lib.gla_recurrent_step.restype = i
    lib.gla_status_string.argtypes = [i]
    lib.gla_status_string.restype = ctypes.c_char_p
    lib.gla_last_device_status.argtypes = [vp]
    lib.gla_last_device_status.restype = i
    lib.gla_version.argtypes = []
    lib.gla_version.restype = i
    return lib


def lib() -> ctypes.CDLL:
    """The loaded library (loaded once per process)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m chunkwise_linear_rnn_gb300.build` (needs nvcc for sm_103a)")
            _lib = _bind(ctypes.CDLL(LIB_PATH))
        return _lib


def status_string(status: int) -> str:
    return lib().gla_status_string(int(status)).decode()


def check(status: int, what: str) -> None:
    if status != GLA_OK:
        raise GlaError(status, what)
