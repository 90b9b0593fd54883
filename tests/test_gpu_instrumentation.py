"""Looking inside the chunked forward through gla_chunk_fwd_debug (C ABI).

gla_chunk_fwd_debug runs the instrumented build of the forward kernel: the
same template with its test hooks compiled in (the production entry points
run the build without them).  The outputs of every instrumented call are
still checked against the oracle.

1. The in-chunk prefix sums (GLA page, "Cumulative Decay Representation"): the
   preparation stage's Gamma, dumped by the kernel, against an fp64 cumulative
   sum of the same fp32 gates, and the block length each chunk took against
   the rule that picks it (one 128-token block while every |Gamma| <= 30 over
   the chunk, else the longest power-of-two sub-chunk whose every block keeps
   its clamped prefix sums within 30).  An error in Gamma that only moves
   rounding in the outputs is caught here and by no end-to-end test.
2. A bounded device wait made to expire on purpose: the loader withholds one
   value tile, the waits for it give up after a short limit, the CTA frees its
   TMEM and returns, gla_last_device_status reports GLA_ERR_TIMEOUT, and the
   next normal call on the device is correct.  No fault, trap or hang: every
   wait in the kernel is bounded and nothing is in flight on the withheld
   barrier.
"""

from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from chunkwise_linear_rnn_gb300 import _lib
from oracle import gla_oracle as og
from synth import make_chunk_inputs
from tolerance import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"
BOUND = 30.0


@pytest.fixture(scope="module")
def lib():
    from chunkwise_linear_rnn_gb300.build import build
    build()
    og.build()
    return _lib.lib()


def _call(lib, q, k, v, a, h0, o, hT, opts=None, dbg=None):
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.gla_chunk_fwd_debug(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), a.data_ptr(), float(dk ** -0.5),
        None if h0 is None else h0.data_ptr(), o.data_ptr(), hT.data_ptr(), B, H, T, dk, dv,
        None if opts is None else ctypes.byref(opts), None if dbg is None else ctypes.byref(dbg),
        stream)


def _expected_blocks(a: np.ndarray):
    """Per (sequence, chunk): the block length the rule picks and the prefix sums
    relative to each token's block reference, in fp64 from the fp32 gates."""
    B, H, T, dk = a.shape
    nch = (T + 127) // 128
    blk = np.zeros((B, H, nch), dtype=np.int64)
    gam = np.zeros(a.shape, dtype=np.float64)
    for b in range(B):
        for h in range(H):
            for c in range(nch):
                seg = a[b, h, 128 * c:128 * (c + 1)].astype(np.float64)
                g = np.cumsum(seg, axis=0)
                if np.max(np.abs(g)) <= BOUND:
                    blk[b, h, c] = 128
                    gam[b, h, 128 * c:128 * c + len(seg)] = g
                    continue
                cl = np.clip(seg, -BOUND, BOUND)
                cs = 64
                while cs > 1:
                    ok = all(np.max(np.abs(np.cumsum(cl[s:s + cs], axis=0))) <= BOUND
                             for s in range(0, len(cl), cs))
                    if ok:
                        break
                    cs //= 2
                blk[b, h, c] = cs
                for s in range(0, len(cl), cs):
                    gam[b, h, 128 * c + s:128 * c + s + cs][:len(cl[s:s + cs])] = \
                        np.cumsum(cl[s:s + cs], axis=0)
    return blk, gam


def _inputs(B, H, T, dk, dv, seed, spikes=False):
    q, k, v, a, h0 = make_chunk_inputs(B, H, T, dk, dv, sigma_h0=0.1, seed=seed, device="cpu")
    if spikes:
        # gates far past the bound in a few chunks and channels (one channel
        # block only in one of them), so that those chunks take sub-chunks
        a[..., 10, 0:64] = -80.0
        a[..., 300:310, min(100, dk - 1)] = -40.0
        a[0, 0, 700, :] = -35.0
    return tuple(None if t is None else t.to(DEV) for t in (q, k, v, a, h0))


@pytest.mark.parametrize("cta_pair,dk,dv,spikes,force", [
    (-1, 128, 128, False, False), (-1, 128, 128, True, False), (-1, 64, 64, True, False),
    (1, 128, 256, False, False), (1, 128, 256, True, False), (-1, 128, 128, False, True),
    (1, 128, 256, False, True)])
def test_prefix_sums_match_fp64_cumsum(lib, cta_pair, dk, dv, spikes, force):
    B, H, T = 2, 2, 777          # six full chunks and a ragged tail
    q, k, v, a, h0 = _inputs(B, H, T, dk, dv, seed=7 + dk + dv, spikes=spikes)
    nch = (T + 127) // 128
    gamma = torch.full((B, H, T, dk), float("nan"), dtype=torch.float32, device=DEV)
    blk = torch.full((B * H * nch,), -1, dtype=torch.int32, device=DEV)
    o = torch.empty(B, H, T, dv, dtype=torch.bfloat16, device=DEV)
    hT = torch.empty(B, H, dk, dv, dtype=torch.float32, device=DEV)
    opts = _lib.GlaChunkOptions(cta_pair=cta_pair, force_exact=1 if force else 0)
    dbg = _lib.GlaChunkDebug(gamma=gamma.data_ptr(), block_len=blk.data_ptr())
    assert _call(lib, q, k, v, a, h0, o, hT, opts, dbg) == _lib.GLA_OK
    torch.cuda.synchronize()
    assert lib.gla_last_device_status(None) == _lib.GLA_OK
    want_blk, want_gam = _expected_blocks(a.cpu().numpy())
    got_blk = blk.cpu().numpy().reshape(B, H, nch)
    if force:
        # every chunk is cut into sub-chunks; the gates here keep 64-token blocks
        # within the bound, so the rule picks 64 for every chunk
        assert np.all(got_blk == 64), got_blk
        want_gam = np.zeros_like(want_gam)
        an = a.cpu().numpy().astype(np.float64)
        for s in range(0, T, 64):
            want_gam[:, :, s:s + 64] = np.cumsum(np.clip(an[:, :, s:s + 64], -BOUND, BOUND), axis=2)
    else:
        np.testing.assert_array_equal(got_blk, want_blk)
        if spikes:
            assert np.any(want_blk < 128) and np.any(want_blk == 128)
    got = gamma.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got)), "a token's prefix sum was not written"
    # fp32 running sums in log2 units over at most 128 terms
    err = np.abs(got - want_gam)
    tol = 2e-5 * (1.0 + np.abs(want_gam)) + 2e-6 * 128
    assert np.all(err <= tol), f"max |Gamma - fp64 cumsum| {err.max():.3e}"
    # and the outputs of the instrumented call are the forward's, against the oracle
    scale = dk ** -0.5
    o_ref, h_ref = og.forward(q.float().cpu().numpy(), k.float().cpu().numpy(),
                              v.float().cpu().numpy(), a.cpu().numpy(), scale,
                              h0.double().cpu().numpy())
    assert_close(o.float().cpu().numpy(), o_ref, "instrumented o", bf16_output=True)
    assert_close(hT.cpu().numpy(), h_ref, "instrumented hT")


@pytest.mark.parametrize("cta_pair,dk,dv", [(-1, 64, 64), (-1, 128, 128)])
def test_bounded_wait_expires_and_the_device_recovers(lib, cta_pair, dk, dv):
    B, H, T = 1, 2, 1024
    q, k, v, a, h0 = _inputs(B, H, T, dk, dv, seed=11)
    o = torch.zeros(B, H, T, dv, dtype=torch.bfloat16, device=DEV)
    hT = torch.zeros(B, H, dk, dv, dtype=torch.float32, device=DEV)
    opts = _lib.GlaChunkOptions(cta_pair=cta_pair)
    # the second value tile of every CTA is never loaded; every wait gives up
    # after 2 ms instead of 2 s
    dbg = _lib.GlaChunkDebug(wait_limit_us=2000, withhold_v=2)
    assert lib.gla_last_device_status(None) == _lib.GLA_OK
    assert _call(lib, q, k, v, a, h0, o, hT, opts, dbg) == _lib.GLA_OK
    torch.cuda.synchronize()
    assert lib.gla_last_device_status(None) == _lib.GLA_ERR_TIMEOUT
    # the word was cleared by the read, and the context is usable: a normal call
    assert lib.gla_last_device_status(None) == _lib.GLA_OK
    assert _call(lib, q, k, v, a, h0, o, hT, opts, None) == _lib.GLA_OK
    torch.cuda.synchronize()
    assert lib.gla_last_device_status(None) == _lib.GLA_OK
    o_ref, h_ref = og.forward(q.float().cpu().numpy(), k.float().cpu().numpy(),
                              v.float().cpu().numpy(), a.cpu().numpy(), dk ** -0.5,
                              h0.double().cpu().numpy())
    assert_close(o.float().cpu().numpy(), o_ref, "after the timeout o", bf16_output=True)
    assert_close(hT.cpu().numpy(), h_ref, "after the timeout hT")


def test_debug_entry_rejects_a_negative_withheld_tile(lib):
    q, k, v, a, h0 = _inputs(1, 1, 128, 64, 64, seed=12)
    o = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device=DEV)
    hT = torch.zeros(1, 1, 64, 64, dtype=torch.float32, device=DEV)
    dbg = _lib.GlaChunkDebug(withhold_v=-1)
    assert _call(lib, q, k, v, a, h0, o, hT, None, dbg) == _lib.GLA_ERR_ARG
