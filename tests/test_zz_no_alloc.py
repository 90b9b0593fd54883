"""gla_chunk_fwd_noalloc, through the C ABI, against the fp64 oracle and against
gla_chunk_fwd_ex.

gla_chunk_fwd_noalloc is for callers that cannot let a library allocate
device memory: runtimes that reserve and account for all of HBM themselves,
or that run without the stream-ordered memory pool.  It takes the scratch of
the sequence-split path from a fixed array inside the library instead of
cudaMallocAsync.  The checks use shapes whose launch plan splits sequences,
so that the array is really used, and make two calls in a row with different
inputs (the array keeps the previous call's contents).  Each result is checked
against the oracle, which shares nothing with either entry point, and against
the allocating entry point's result.

This file is named so that pytest collects it after every other test.
"""

from __future__ import annotations

import ctypes
import os
import re

import pytest
import torch

import chunkwise_linear_rnn_gb300 as gla
from chunkwise_linear_rnn_gb300 import _lib
from oracle import gla_oracle as og
from synth import make_chunk_inputs
from tolerance import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def lib():
    from chunkwise_linear_rnn_gb300.build import build
    build()
    og.build()
    return _lib.lib()


def _oracle_check(o, h, q, k, v, a, h0, what, heads=None):
    """o, hT of a call against the fp64 oracle, on every head or the listed (b, h)."""
    B, H = q.shape[:2]
    heads = heads if heads is not None else [(b, hh) for b in range(B) for hh in range(H)]
    sel = lambda t: torch.stack([t[b, hh] for b, hh in heads])  # noqa: E731
    cpu = lambda t: sel(t).float().cpu().numpy()  # noqa: E731
    o_ref, h_ref = og.forward(cpu(q), cpu(k), cpu(v), cpu(a), float(q.shape[-1] ** -0.5),
                              None if h0 is None else sel(h0).double().cpu().numpy())
    assert_close(sel(o).float().cpu().numpy(), o_ref, f"{what} o vs oracle", bf16_output=True)
    assert_close(sel(h).cpu().numpy(), h_ref, f"{what} hT vs oracle")


def _abi_call(fn, q, k, v, a, h0, o, hT, opts=None):
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), a.data_ptr(), float(dk ** -0.5),
              None if h0 is None else h0.data_ptr(), o.data_ptr(), hT.data_ptr(), B, H, T, dk,
              dv, None if opts is None else ctypes.byref(opts), stream)


@pytest.mark.parametrize("shape", [(1, 2, 4096, 128, 256), (1, 3, 2500, 64, 128)])
def test_noalloc_matches_the_allocating_entry_point_on_two_calls(lib, shape):
    B, H, T, dk, dv = shape
    plan = gla.gla_chunk_fwd_plan(B, H, T, dk, dv)
    assert plan["segments"] > 1 and 0 < plan["scratch_bytes"] <= _lib_scratch_limit()
    for seed in (0, 1):
        q, k, v, a, h0 = make_chunk_inputs(B, H, T, dk, dv, sigma_h0=0.1, seed=seed, device=DEV)
        o_ref = torch.empty(B, H, T, dv, dtype=torch.bfloat16, device=DEV)
        h_ref = torch.empty(B, H, dk, dv, dtype=torch.float32, device=DEV)
        o = torch.full_like(o_ref, float("nan"))
        h = torch.full_like(h_ref, float("nan"))
        assert _abi_call(lib.gla_chunk_fwd_ex, q, k, v, a, h0, o_ref, h_ref) == _lib.GLA_OK
        assert _abi_call(lib.gla_chunk_fwd_noalloc, q, k, v, a, h0, o, h) == _lib.GLA_OK
        torch.cuda.synchronize()
        assert lib.gla_last_device_status(None) == _lib.GLA_OK
        _oracle_check(o, h, q, k, v, a, h0, f"noalloc, call {seed + 1}")
        _oracle_check(o_ref, h_ref, q, k, v, a, h0, f"allocating, call {seed + 1}")
        assert_close(o.float().cpu().numpy(), o_ref.double().cpu().numpy(),
                     f"noalloc o vs allocating, call {seed + 1}", bf16_output=True)
        assert_close(h.cpu().numpy(), h_ref.double().cpu().numpy(),
                     f"noalloc hT vs allocating, call {seed + 1}")


def _lib_scratch_limit() -> int:
    """GLA_NOALLOC_SCRATCH_BYTES as the public header defines it."""
    header = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                          "include", "gla.h")
    m = re.search(r"#define\s+GLA_NOALLOC_SCRATCH_BYTES\s+\(([^)]*)\)", open(header).read())
    assert m, "GLA_NOALLOC_SCRATCH_BYTES not found in include/gla.h"
    return int(eval(m.group(1).replace("u", ""), {"__builtins__": {}}))  # e.g. 16 * 1024 * 1024


def test_noalloc_rejects_plans_beyond_its_scratch(lib):
    B, H, T, dk, dv = 2, 16, 8192, 128, 256
    opts = _lib.GlaChunkOptions(segments=64)
    plan = gla.gla_chunk_fwd_plan(B, H, T, dk, dv, segments=64)
    assert plan["scratch_bytes"] > _lib_scratch_limit()
    q, k, v, a, h0 = make_chunk_inputs(B, H, T, dk, dv, seed=2, device=DEV)
    o = torch.zeros(B, H, T, dv, dtype=torch.bfloat16, device=DEV)
    h = torch.zeros(B, H, dk, dv, dtype=torch.float32, device=DEV)
    assert _abi_call(lib.gla_chunk_fwd_noalloc, q, k, v, a, None, o, h, opts) == _lib.GLA_ERR_SCRATCH
    torch.cuda.synchronize()
    assert torch.count_nonzero(o).item() == 0 and torch.count_nonzero(h).item() == 0


def test_automatic_plans_beyond_the_scratch_take_longer_segments(lib):
    # many sequences of a few dozen chunks: the allocating plan cuts them into
    # segments whose scratch exceeds the fixed array; the no-allocation call
    # takes longer segments instead of failing.  100 sequences of 32 chunks on
    # 152 SMs: ranges of 22 chunks, up to 3 segments per sequence, 3 x 100 states
    # of 64 KB = 19.7 MB of scratch (still 3 segments on any GPU with 108 to 200
    # SMs, one 128x128 tile per CTA)
    B, H, T, dk, dv = 50, 2, 4096, 128, 128
    plan = gla.gla_chunk_fwd_plan(B, H, T, dk, dv)
    assert plan["scratch_bytes"] > _lib_scratch_limit(), (
        f"the allocating plan fits the fixed scratch: {plan}; pick a shape that does not")
    q, k, v, a, h0 = make_chunk_inputs(B, H, T, dk, dv, sigma_h0=0.1, seed=3, device=DEV)
    o_ref = torch.empty(B, H, T, dv, dtype=torch.bfloat16, device=DEV)
    h_ref = torch.empty(B, H, dk, dv, dtype=torch.float32, device=DEV)
    o = torch.full_like(o_ref, float("nan"))
    h = torch.full_like(h_ref, float("nan"))
    assert _abi_call(lib.gla_chunk_fwd_ex, q, k, v, a, h0, o_ref, h_ref) == _lib.GLA_OK
    assert _abi_call(lib.gla_chunk_fwd_noalloc, q, k, v, a, h0, o, h) == _lib.GLA_OK
    torch.cuda.synchronize()
    assert lib.gla_last_device_status(None) == _lib.GLA_OK
    heads = [(0, 0), (17, 1), (33, 0), (49, 1)]
    _oracle_check(o, h, q, k, v, a, h0, "longer segments", heads)
    assert_close(o.float().cpu().numpy(), o_ref.double().cpu().numpy(),
                 "longer segments o vs allocating", bf16_output=True)
    assert_close(h.cpu().numpy(), h_ref.double().cpu().numpy(), "longer segments hT vs allocating")
