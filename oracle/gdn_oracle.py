"""ctypes loader for the fp64 gated-delta-rule oracle (``gdn_oracle.c``) — TEST INFRASTRUCTURE.

``forward`` takes numpy arrays (float32 inputs, the exact values a GPU run
would see) and returns float64 outputs.
"""

from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import gla_oracle

_SRC = os.path.join(os.path.dirname(os.path.abspath(__file__)), "gdn_oracle.c")
_LOCK = threading.Lock()
_LIBS: dict[str, ctypes.CDLL] = {}


def build(src: str = _SRC, out: str | None = None) -> str:
    return gla_oracle.build(src, out or gla_oracle.library_path(tag="gdn"))


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    f = ctypes.POINTER(ctypes.c_float)
    d = ctypes.POINTER(ctypes.c_double)
    lib.gdn_oracle_forward.argtypes = [f, f, f, f, f, ctypes.c_double, d, d, d, ctypes.c_int64,
                                       ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.gdn_oracle_forward.restype = ctypes.c_int
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    with _LOCK:
        path = path or build()
        if path not in _LIBS:
            _LIBS[path] = _bind(ctypes.CDLL(path))
        return _LIBS[path]


def _f32(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def forward(q, k, v, g, beta, scale: float, h0=None, *, nthreads: int = 0, lib=None):
    """Run the gated delta rule over whole sequences.

    q, k: [..., T, dk]; v: [..., T, dv]; g (log alpha), beta: [..., T];
    h0: [..., dk, dv] or None.  Returns (o float64 [..., T, dv], hT float64
    [..., dk, dv]).
    """
    lib = lib or load()
    q, k, v, g, b = _f32(q), _f32(k), _f32(v), _f32(g), _f32(beta)
    lead = q.shape[:-2]
    T, dk = q.shape[-2], q.shape[-1]
    dv = v.shape[-1]
    assert k.shape == q.shape and v.shape == lead + (T, dv)
    assert g.shape == lead + (T,) and b.shape == lead + (T,)
    BH = int(np.prod(lead, dtype=np.int64)) if lead else 1
    o = np.empty(lead + (T, dv), dtype=np.float64)
    hT = np.empty(lead + (dk, dv), dtype=np.float64)
    h0p = None
    if h0 is not None:
        h0a = np.ascontiguousarray(np.asarray(h0, dtype=np.float64))
        assert h0a.shape == lead + (dk, dv)
        h0p = h0a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
    P = lambda a, t: a.ctypes.data_as(ctypes.POINTER(t))  # noqa: E731
    rc = lib.gdn_oracle_forward(P(q, ctypes.c_float), P(k, ctypes.c_float), P(v, ctypes.c_float),
                                P(g, ctypes.c_float), P(b, ctypes.c_float), float(scale), h0p,
                                P(o, ctypes.c_double), P(hT, ctypes.c_double), BH, T, dk, dv,
                                int(nthreads))
    if rc != 0:
        raise MemoryError("oracle could not allocate its state buffers")
    return o, hT
