"""gla_chunk_fwd_noalloc, through the C ABI, against gla_chunk_fwd.

gla_chunk_fwd_noalloc is for callers that cannot let a library allocate
device memory: runtimes that reserve and account for all of HBM themselves,
or that run without the stream-ordered memory pool.  It takes the scratch of
the sequence-split path from a fixed array inside the library instead of
cudaMallocAsync.  The checks use shapes whose launch plan splits sequences,
so that the array is really used, and make two calls in a row with different
inputs (the array keeps the previous call's contents).

This file is named so that pytest collects it after every other test.
"""

from __future__ import annotations

import ctypes

import pytest
import torch

import chunkwise_linear_rnn_gb300 as gla
from chunkwise_linear_rnn_gb300 import _lib
from synth import make_chunk_inputs
from tolerance import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def lib():
    from chunkwise_linear_rnn_gb300.build import build
    build()
    return _lib.lib()


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
        assert_close(o.float().cpu().numpy(), o_ref.double().cpu().numpy(),
                     f"noalloc o, call {seed + 1}", bf16_output=True)
        assert_close(h.cpu().numpy(), h_ref.double().cpu().numpy(), f"noalloc hT, call {seed + 1}")


def _lib_scratch_limit() -> int:
    return 16 * 1024 * 1024  # GLA_NOALLOC_SCRATCH_BYTES in include/gla.h


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
    # takes longer segments instead of failing
    B, H, T, dk, dv = 50, 2, 4096, 128, 128
    plan = gla.gla_chunk_fwd_plan(B, H, T, dk, dv)
    if plan["scratch_bytes"] <= _lib_scratch_limit():
        pytest.skip(f"the allocating plan fits the fixed scratch on this device ({plan})")
    q, k, v, a, h0 = make_chunk_inputs(B, H, T, dk, dv, sigma_h0=0.1, seed=3, device=DEV)
    o_ref = torch.empty(B, H, T, dv, dtype=torch.bfloat16, device=DEV)
    h_ref = torch.empty(B, H, dk, dv, dtype=torch.float32, device=DEV)
    o = torch.full_like(o_ref, float("nan"))
    h = torch.full_like(h_ref, float("nan"))
    assert _abi_call(lib.gla_chunk_fwd_ex, q, k, v, a, h0, o_ref, h_ref) == _lib.GLA_OK
    assert _abi_call(lib.gla_chunk_fwd_noalloc, q, k, v, a, h0, o, h) == _lib.GLA_OK
    torch.cuda.synchronize()
    assert lib.gla_last_device_status(None) == _lib.GLA_OK
    assert_close(o.float().cpu().numpy(), o_ref.double().cpu().numpy(), "longer segments o",
                 bf16_output=True)
    assert_close(h.cpu().numpy(), h_ref.double().cpu().numpy(), "longer segments hT")
