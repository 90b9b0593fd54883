"""ctypes loader for the fp64 C oracle (``gla_oracle.c``) — TEST INFRASTRUCTURE.

``build()`` compiles the C file with gcc and OpenMP into ``_build/`` beside
this file; ``forward`` and ``step`` take numpy arrays (float32 inputs, whose
values are the exact bf16 / fp32 values a GPU run sees) and return float64.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gla_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIBS: dict[str, ctypes.CDLL] = {}


def library_path(src: str = _SRC, tag: str = "") -> str:
    name = "libgla_oracle" + (("_" + tag) if tag else "") + ".so"
    return os.path.join(_BUILD_DIR, name)


def build(src: str = _SRC, out: str | None = None, extra_flags: tuple[str, ...] = ()) -> str:
    """Compile the oracle (or a variant of its source) into a shared library."""
    out = out or library_path()
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src)
            and not extra_flags):
        return out
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", *extra_flags, src,
           "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    f = ctypes.POINTER(ctypes.c_float)
    d = ctypes.POINTER(ctypes.c_double)
    lib.gla_oracle_forward.argtypes = [f, f, f, f, ctypes.c_double, d, d, d, ctypes.c_int64,
                                       ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.gla_oracle_forward.restype = ctypes.c_int
    lib.gla_oracle_step.argtypes = [f, f, f, f, ctypes.c_double, d, d, ctypes.c_int64,
                                    ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.gla_oracle_step.restype = None
    i64 = ctypes.c_int64
    lib.gla_oracle_backward.argtypes = [f, f, f, f, ctypes.c_double, d, f, d, d, d, d, d, d, i64,
                                        i64, ctypes.c_int, ctypes.c_int, i64, ctypes.c_int]
    lib.gla_oracle_backward.restype = ctypes.c_int
    lib.gla_oracle_max_threads.argtypes = []
    lib.gla_oracle_max_threads.restype = ctypes.c_int
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    with _LOCK:
        path = path or build()
        if path not in _LIBS:
            _LIBS[path] = _bind(ctypes.CDLL(path))
        return _LIBS[path]


def max_threads() -> int:
    return int(load().gla_oracle_max_threads())


def _f32(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _ptr(a: np.ndarray, ct):
    return a.ctypes.data_as(ctypes.POINTER(ct))


def forward(q, k, v, log_alpha, scale: float, h0=None, *, nthreads: int = 0, lib=None):
    """Run the recurrence over a whole sequence.

    q, k, log_alpha: [..., T, dk]; v: [..., T, dv]; h0: [..., dk, dv] or None.
    Leading axes (batch, heads) are flattened into independent sequences.
    Returns (o float64 [..., T, dv], hT float64 [..., dk, dv]).
    """
    lib = lib or load()
    q, k, v, a = _f32(q), _f32(k), _f32(v), _f32(log_alpha)
    lead = q.shape[:-2]
    T, dk = q.shape[-2], q.shape[-1]
    dv = v.shape[-1]
    assert k.shape == q.shape and a.shape == q.shape and v.shape == lead + (T, dv)
    BH = int(np.prod(lead, dtype=np.int64)) if lead else 1
    o = np.empty(lead + (T, dv), dtype=np.float64)
    hT = np.empty(lead + (dk, dv), dtype=np.float64)
    h0p = None
    if h0 is not None:
        h0a = np.ascontiguousarray(np.asarray(h0, dtype=np.float64))
        assert h0a.shape == lead + (dk, dv)
        h0p = _ptr(h0a, ctypes.c_double)
    rc = lib.gla_oracle_forward(_ptr(q, ctypes.c_float), _ptr(k, ctypes.c_float),
                                _ptr(v, ctypes.c_float), _ptr(a, ctypes.c_float), float(scale),
                                h0p, _ptr(o, ctypes.c_double), _ptr(hT, ctypes.c_double), BH, T,
                                dk, dv, int(nthreads))
    if rc != 0:
        raise MemoryError("oracle could not allocate its state buffers")
    return o, hT


def step(q, k, v, log_alpha, scale: float, h: np.ndarray, *, nthreads: int = 0, lib=None):
    """One decode step for independent heads; h (float64 [..., dk, dv]) is updated in place.

    q, k, log_alpha: [..., dk]; v: [..., dv].  Returns o float64 [..., dv].
    """
    lib = lib or load()
    q, k, v, a = _f32(q), _f32(k), _f32(v), _f32(log_alpha)
    assert h.dtype == np.float64 and h.flags.c_contiguous
    lead = q.shape[:-1]
    dk, dv = q.shape[-1], v.shape[-1]
    assert h.shape == lead + (dk, dv)
    BH = int(np.prod(lead, dtype=np.int64)) if lead else 1
    o = np.empty(lead + (dv,), dtype=np.float64)
    lib.gla_oracle_step(_ptr(q, ctypes.c_float), _ptr(k, ctypes.c_float), _ptr(v, ctypes.c_float),
                        _ptr(a, ctypes.c_float), float(scale), _ptr(h, ctypes.c_double),
                        _ptr(o, ctypes.c_double), BH, dk, dv, int(nthreads))
    return o


def backward(q, k, v, log_alpha, scale: float, d_o, h0=None, dhT=None, *, ck: int = 0,
             nthreads: int = 0, lib=None):
    """Gradients of L = sum_t <d_o_t, o_t> + <dhT, hT> through the recurrence.

    Shapes as in ``forward``; d_o: [..., T, dv]; h0, dhT: [..., dk, dv] or None
    (zero).  ``ck`` is the checkpoint spacing of the state replay (0 = about
    sqrt(T)); it changes memory use only.  Returns float64
    (dq, dk, dv, dlog_alpha, dh0), each shaped like its input.
    """
    lib = lib or load()
    q, k, v, a, g = _f32(q), _f32(k), _f32(v), _f32(log_alpha), _f32(d_o)
    lead = q.shape[:-2]
    T, dk = q.shape[-2], q.shape[-1]
    dv = v.shape[-1]
    assert k.shape == q.shape and a.shape == q.shape and v.shape == lead + (T, dv)
    assert g.shape == v.shape
    BH = int(np.prod(lead, dtype=np.int64)) if lead else 1

    def state(x):
        if x is None:
            return None, None
        xa = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
        assert xa.shape == lead + (dk, dv)
        return xa, _ptr(xa, ctypes.c_double)

    h0a, h0p = state(h0)
    dhTa, dhTp = state(dhT)
    dq = np.empty(q.shape, dtype=np.float64)
    dkk = np.empty(q.shape, dtype=np.float64)
    dvv = np.empty(v.shape, dtype=np.float64)
    da = np.empty(q.shape, dtype=np.float64)
    dh0 = np.empty(lead + (dk, dv), dtype=np.float64)
    dp = lambda x: _ptr(x, ctypes.c_double)  # noqa: E731
    rc = lib.gla_oracle_backward(_ptr(q, ctypes.c_float), _ptr(k, ctypes.c_float),
                                 _ptr(v, ctypes.c_float), _ptr(a, ctypes.c_float), float(scale),
                                 h0p, _ptr(g, ctypes.c_float), dhTp, dp(dq), dp(dkk), dp(dvv),
                                 dp(da), dp(dh0), BH, T, dk, dv, int(ck), int(nthreads))
    if rc != 0:
        raise MemoryError("oracle could not allocate its state buffers")
    return dq, dkk, dvv, da, dh0


def forward_torch(q, k, v, log_alpha, scale: float, h0=None, *, nthreads: int = 0):
    """Convenience: torch tensors (any device, bf16/fp32) in, float64 numpy out."""
    def cpu32(t):
        return t.detach().to("cpu").float().numpy()
    h = None if h0 is None else h0.detach().to("cpu").double().numpy()
    return forward(cpu32(q), cpu32(k), cpu32(v), cpu32(log_alpha), scale, h, nthreads=nthreads)
