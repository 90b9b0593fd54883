"""Host-side checks of the C-ABI library that need no GPU.

* the library builds for sm_103a and loads in a process without a GPU driver;
* it exports every function that include/gla.h declares;
* argument validation happens on the host, before any CUDA call, and returns
  the documented status codes; with valid arguments and no GPU the calls
  report GLA_ERR_DEVICE instead of crashing.
"""

from __future__ import annotations

import ctypes
import os
import re

import pytest

from chunkwise_linear_rnn_gb300 import _lib
from chunkwise_linear_rnn_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gla.h")


@pytest.fixture(scope="module")
def lib():
    build()
    return _lib.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gla_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("gla_chunk_fwd", "gla_recurrent_step", "gla_status_string",
              "gla_last_device_status"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} declared in gla.h but not exported"
    assert set(_declared_functions()) <= set(_lib.EXPORTED) | set(_declared_functions())


def test_status_strings(lib):
    for code in range(0, 8):
        s = _lib.status_string(code)
        assert s and s != "unknown status"
    assert _lib.status_string(99) == "unknown status"
    assert lib.gla_version() >= 100


# A fake, 16-byte aligned "device" address: validation must reject or accept
# arguments without ever dereferencing it.
P = 0x10000


def _chunk(lib, *, q=P, k=P, v=P, a=P, h0=None, o=P, hT=None, B=1, H=1, T=16, dk=64, dv=64,
           opts=None):
    return lib.gla_chunk_fwd_ex(q, k, v, a, 0.125, h0, o, hT, B, H, T, dk, dv, opts, None)


@pytest.mark.parametrize("field", ["q", "k", "v", "a", "o"])
def test_chunk_rejects_null(lib, field):
    assert _chunk(lib, **{field: None}) == _lib.GLA_ERR_ARG


@pytest.mark.parametrize("dims", [dict(B=0), dict(H=0), dict(T=0), dict(T=-3)])
def test_chunk_rejects_sizes(lib, dims):
    assert _chunk(lib, **dims) == _lib.GLA_ERR_ARG


@pytest.mark.parametrize("dk,dv", [(32, 64), (96, 64), (256, 64), (64, 32), (64, 512), (128, 192)])
def test_chunk_rejects_shapes(lib, dk, dv):
    assert _chunk(lib, dk=dk, dv=dv) == _lib.GLA_ERR_SHAPE


def test_noalloc_validates_on_the_host(lib):
    f = lib.gla_chunk_fwd_noalloc
    assert f(None, P, P, P, 0.1, None, P, None, 1, 1, 16, 64, 64, None, None) == _lib.GLA_ERR_ARG
    assert f(P, P, P, P, 0.1, None, P, None, 1, 1, 0, 64, 64, None, None) == _lib.GLA_ERR_ARG
    assert f(P + 8, P, P, P, 0.1, None, P, None, 1, 1, 16, 64, 64, None, None) == _lib.GLA_ERR_ARG
    assert f(P, P, P, P, 0.1, None, P, None, 1, 1, 16, 96, 64, None, None) == _lib.GLA_ERR_SHAPE


def test_host_entry_validates_before_any_cuda_call(lib):
    f = lib.gla_chunk_fwd_host
    assert f(None, P, P, P, 0.1, None, P, None, 1, 1, 16, 64, 64, None) == _lib.GLA_ERR_ARG
    assert f(P, P, P, P, 0.1, None, None, None, 1, 1, 16, 64, 64, None) == _lib.GLA_ERR_ARG
    assert f(P, P, P, P, 0.1, None, P, None, 1, 0, 16, 64, 64, None) == _lib.GLA_ERR_ARG
    assert f(P, P, P, P, 0.1, None, P, None, 1, 1, 16, 64, 48, None) == _lib.GLA_ERR_SHAPE


def _cu(*xs):
    return (ctypes.c_int * len(xs))(*xs)


def test_packed_entry_validates_cu_seqlens_on_the_host(lib):
    f = lib.gla_chunk_fwd_varlen
    ok = _cu(0, 5, 5, 16)
    # well-formed offsets reach the device check (no GPU here)
    assert f(P, P, P, P, 0.1, None, P, None, ok, 3, 2, 16, 64, 64, None) == _lib.GLA_ERR_DEVICE
    # offsets must start at 0, end at T_total and never decrease
    assert f(P, P, P, P, 0.1, None, P, None, _cu(1, 5, 16), 2, 2, 16, 64, 64, None) == _lib.GLA_ERR_ARG
    assert f(P, P, P, P, 0.1, None, P, None, _cu(0, 5, 15), 2, 2, 16, 64, 64, None) == _lib.GLA_ERR_ARG
    assert f(P, P, P, P, 0.1, None, P, None, _cu(0, 9, 5, 16), 3, 2, 16, 64, 64, None) == _lib.GLA_ERR_ARG
    assert f(P, P, P, P, 0.1, None, P, None, None, 3, 2, 16, 64, 64, None) == _lib.GLA_ERR_ARG
    # sizes, pointers, alignment and head dimensions as for gla_chunk_fwd
    assert f(P, P, P, P, 0.1, None, P, None, ok, 0, 2, 16, 64, 64, None) == _lib.GLA_ERR_ARG
    assert f(P, P, P, P, 0.1, None, P, None, ok, 3, 0, 16, 64, 64, None) == _lib.GLA_ERR_ARG
    assert f(None, P, P, P, 0.1, None, P, None, ok, 3, 2, 16, 64, 64, None) == _lib.GLA_ERR_ARG
    assert f(P + 8, P, P, P, 0.1, None, P, None, ok, 3, 2, 16, 64, 64, None) == _lib.GLA_ERR_ARG
    assert f(P, P, P, P, 0.1, None, P, None, ok, 3, 2, 16, 96, 64, None) == _lib.GLA_ERR_SHAPE
    ex = lib.gla_chunk_fwd_varlen_ex
    bad = ctypes.byref(_lib.GlaChunkOptions(cta_pair=3))
    assert ex(P, P, P, P, 0.1, None, P, None, ok, 3, 2, 16, 64, 64, bad, None) == _lib.GLA_ERR_ARG
    # one gate per head is for fixed-length calls only
    per_head = ctypes.byref(_lib.GlaChunkOptions(gate_per_head=1))
    assert ex(P, P, P, P, 0.1, None, P, None, ok, 3, 2, 16, 64, 64, per_head, None) == _lib.GLA_ERR_ARG


def test_gate_per_head_option_is_validated(lib):
    assert _chunk(lib, opts=ctypes.byref(_lib.GlaChunkOptions(gate_per_head=2))) == _lib.GLA_ERR_ARG
    import torch
    if not torch.cuda.is_available():
        assert _chunk(lib, opts=ctypes.byref(_lib.GlaChunkOptions(gate_per_head=1))) == _lib.GLA_ERR_DEVICE


def test_python_host_binding_checks_dtypes():
    import torch
    import chunkwise_linear_rnn_gb300 as gla
    q = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        gla.gla_chunk_fwd_host(q, q, q, torch.zeros(1, 1, 4, 64, dtype=torch.float64))


def test_chunk_rejects_misaligned(lib):
    assert _chunk(lib, q=P + 8) == _lib.GLA_ERR_ARG
    assert _chunk(lib, hT=P + 4) == _lib.GLA_ERR_ARG


def test_chunk_rejects_bad_options(lib):
    assert _chunk(lib, opts=ctypes.byref(_lib.GlaChunkOptions(dv_tile=96))) == _lib.GLA_ERR_ARG
    assert _chunk(lib, opts=ctypes.byref(_lib.GlaChunkOptions(dv_tile=128)), dv=64) == _lib.GLA_ERR_ARG
    assert _chunk(lib, opts=ctypes.byref(_lib.GlaChunkOptions(segments=-1))) == _lib.GLA_ERR_ARG
    assert _chunk(lib, opts=ctypes.byref(_lib.GlaChunkOptions(cta_pair=2))) == _lib.GLA_ERR_ARG
    assert _chunk(lib, opts=ctypes.byref(_lib.GlaChunkOptions(cta_pair=-2))) == _lib.GLA_ERR_ARG


def test_options_struct_matches_the_header(lib):
    text = open(HEADER).read()
    body = text[text.index("typedef struct gla_chunk_options"):text.index("} gla_chunk_options;")]
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = re.findall(r"int\s+(\w+)(?:\[(\d+)\])?;", body)
    ours = [(n, str(t._length_) if hasattr(t, "_length_") else "")
            for n, t in _lib.GlaChunkOptions._fields_]
    assert fields == ours


def test_step_validation(lib):
    f = lib.gla_recurrent_step
    assert f(None, P, P, P, 1.0, P, P, 1, 1, 64, 64, None) == _lib.GLA_ERR_ARG
    assert f(P, P, P, P, 1.0, None, P, 1, 1, 64, 64, None) == _lib.GLA_ERR_ARG
    assert f(P, P, P, P, 1.0, P, P, 0, 1, 64, 64, None) == _lib.GLA_ERR_ARG
    assert f(P, P, P, P, 1.0, P + 4, P, 1, 1, 64, 64, None) == _lib.GLA_ERR_ARG
    assert f(P, P, P, P, 1.0, P, P, 1, 1, 48, 64, None) == _lib.GLA_ERR_SHAPE


def test_valid_arguments_without_gpu_report_device_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _chunk(lib) == _lib.GLA_ERR_DEVICE
    assert lib.gla_recurrent_step(P, P, P, P, 1.0, P, P, 1, 1, 64, 64, None) == _lib.GLA_ERR_DEVICE
    assert lib.gla_last_device_status(None) == _lib.GLA_ERR_DEVICE
    assert lib.gla_chunk_fwd_noalloc(P, P, P, P, 0.125, None, P, None, 1, 1, 16, 64, 64, None,
                                     None) == _lib.GLA_ERR_DEVICE
    assert lib.gla_chunk_fwd_host(P, P, P, P, 0.125, None, P, None, 1, 1, 16, 64, 64,
                                  None) == _lib.GLA_ERR_DEVICE


def test_python_binding_rejects_cpu_tensors():
    import torch
    import chunkwise_linear_rnn_gb300 as gla
    q = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        gla.gla_chunk_fwd(q, q, q, torch.zeros(1, 1, 4, 64))


def _bwd(lib, **kw):
    """gla_chunk_bwd_ex with fake aligned pointers; keyword overrides."""
    a = dict(q=P, k=P, v=P, a=P, scale=0.125, h0=None, d_o=P, dhT=None, gq=P, gk=P, gv=P, ga=P,
             gh0=None, B=1, H=1, T=16, dk=64, dv=64, opts=None)
    a.update(kw)
    return lib.gla_chunk_bwd_ex(a["q"], a["k"], a["v"], a["a"], a["scale"], a["h0"], a["d_o"],
                                a["dhT"], a["gq"], a["gk"], a["gv"], a["ga"], a["gh0"], a["B"],
                                a["H"], a["T"], a["dk"], a["dv"], a["opts"], None)


@pytest.mark.parametrize("field", ["q", "k", "v", "a", "d_o", "gq", "gk", "gv", "ga"])
def test_backward_rejects_null(lib, field):
    assert _bwd(lib, **{field: None}) == _lib.GLA_ERR_ARG


def test_backward_validates_on_the_host(lib):
    assert _bwd(lib, T=0) == _lib.GLA_ERR_ARG
    assert _bwd(lib, H=70000) == _lib.GLA_ERR_ARG            # H beyond the grid's y extent
    assert _bwd(lib, dk=96) == _lib.GLA_ERR_SHAPE
    assert _bwd(lib, dv=32) == _lib.GLA_ERR_SHAPE
    assert _bwd(lib, q=P + 2) == _lib.GLA_ERR_ARG            # 16-byte alignment
    assert _bwd(lib, gh0=P + 4) == _lib.GLA_ERR_ARG
    assert _bwd(lib, opts=ctypes.byref(_lib.GlaChunkOptions(gate_per_head=2))) == _lib.GLA_ERR_ARG
    assert _bwd(lib, opts=ctypes.byref(_lib.GlaChunkOptions(force_exact=3))) == _lib.GLA_ERR_ARG


def test_backward_plan(lib):
    import chunkwise_linear_rnn_gb300 as gla
    p = gla.gla_chunk_bwd_plan(2, 16, 32768, 128, 256)
    assert p["chunk"] == 64 and p["launches"] == 6
    NC, BH = 512, 32
    # chunk states (NC + 1 slots) and state gradients (NC slots), fp32 dk x dv each
    assert p["scratch_bytes"] >= 4 * BH * (2 * NC + 1) * 128 * 256
    with pytest.raises(gla.GlaError):
        gla.gla_chunk_bwd_plan(1, 1, 0, 64, 64)


def test_backward_without_gpu_reports_device_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _bwd(lib) == _lib.GLA_ERR_DEVICE
    assert _bwd(lib, opts=ctypes.byref(_lib.GlaChunkOptions(gate_per_head=1))) == _lib.GLA_ERR_DEVICE


def _gdn(lib, **kw):
    """gla_gdn_fwd with fake aligned pointers; keyword overrides."""
    a = dict(q=P, k=P, v=P, g=P, beta=P, scale=0.125, h0=None, o=P, hT=None, B=1, H=1, T=16,
             dk=64, dv=64)
    a.update(kw)
    return lib.gla_gdn_fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["scale"], a["h0"], a["o"],
                           a["hT"], a["B"], a["H"], a["T"], a["dk"], a["dv"], None)


def test_gated_delta_rule_validates_before_the_device(lib):
    for field in ("q", "k", "v", "g", "beta", "o"):
        assert _gdn(lib, **{field: None}) == _lib.GLA_ERR_ARG
    for field in ("q", "k", "v"):   # fetched in 16-byte pieces
        assert _gdn(lib, **{field: P + 8}) == _lib.GLA_ERR_ARG
    assert _gdn(lib, o=P + 2) == _lib.GLA_ERR_DEVICE   # o needs element alignment only
    assert _gdn(lib, T=0) == _lib.GLA_ERR_ARG
    assert _gdn(lib, B=300, H=300) == _lib.GLA_ERR_ARG
    assert _gdn(lib, dk=96) == _lib.GLA_ERR_SHAPE
    assert _gdn(lib, dv=48) == _lib.GLA_ERR_SHAPE
    assert _gdn(lib) == _lib.GLA_ERR_DEVICE   # valid arguments, no GPU here


def _gdn_chunk(lib, **kw):
    """gla_gdn_chunk_fwd with fake aligned pointers; keyword overrides."""
    a = dict(q=P, k=P, v=P, g=P, beta=P, scale=0.125, h0=None, o=P, hT=None, B=1, H=1, T=16,
             dk=128, dv=64)
    a.update(kw)
    return lib.gla_gdn_chunk_fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["scale"], a["h0"],
                                 a["o"], a["hT"], a["B"], a["H"], a["T"], a["dk"], a["dv"], None)


def test_chunked_gated_delta_rule_validates_before_the_device(lib):
    for field in ("q", "k", "v", "g", "beta", "o"):
        assert _gdn_chunk(lib, **{field: None}) == _lib.GLA_ERR_ARG
    for field in ("q", "k", "v", "o", "hT"):   # TMA tiles and 16-byte stores
        assert _gdn_chunk(lib, **{field: P + 8}) == _lib.GLA_ERR_ARG
    for field in ("g", "beta", "h0"):          # fp32, read as words
        assert _gdn_chunk(lib, **{field: P + 2}) == _lib.GLA_ERR_ARG
    assert _gdn_chunk(lib, T=0) == _lib.GLA_ERR_ARG
    assert _gdn_chunk(lib, B=300, H=300) == _lib.GLA_ERR_ARG
    assert _gdn_chunk(lib, dk=64) == _lib.GLA_ERR_SHAPE    # the chunked form is dk = 128 only
    assert _gdn_chunk(lib, dv=48) == _lib.GLA_ERR_SHAPE
    # more scratch rows than 32-bit tensor-map coordinates address
    assert _gdn_chunk(lib, H=2, T=2 ** 30 + 1) == _lib.GLA_ERR_ARG
    assert _gdn_chunk(lib) == _lib.GLA_ERR_DEVICE        # valid arguments, no GPU here


def test_debug_entry_validates_before_the_device(lib):
    def dbg_call(dbg, opts=None):
        return lib.gla_chunk_fwd_debug(P, P, P, P, 0.125, None, P, None, 1, 1, 16, 64, 64,
                                       None if opts is None else ctypes.byref(opts),
                                       ctypes.byref(dbg), None)
    assert dbg_call(_lib.GlaChunkDebug(withhold_v=-1)) == _lib.GLA_ERR_ARG
    assert dbg_call(_lib.GlaChunkDebug(gamma=P + 4)) == _lib.GLA_ERR_ARG
    # the instrumented kernel build covers one gate per key channel only
    assert dbg_call(_lib.GlaChunkDebug(), _lib.GlaChunkOptions(gate_per_head=1)) == _lib.GLA_ERR_ARG
    assert dbg_call(_lib.GlaChunkDebug(wait_limit_us=5, withhold_v=1)) == _lib.GLA_ERR_DEVICE
