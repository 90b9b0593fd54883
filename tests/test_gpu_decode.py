"""GPU parity of gla_recurrent_step (through the C ABI) against the fp64 oracle."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import chunkwise_linear_rnn_gb300 as gla
from oracle import gla_oracle as og
from synth import DECODE_CONFIG, make_chunk_inputs, make_decode_inputs
from tolerance import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunkwise_linear_rnn_gb300.build import build
    build()
    og.build()


def _np32(t):
    return t.detach().float().cpu().numpy()


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (64, 256), (128, 64), (128, 128),
                                   (128, 256)])
def test_step_shapes(dk, dv):
    B, H, steps = 3, 5, 12
    h0, q, k, v, a = make_decode_inputs(B, H, dk, dv, steps, seed=dk * 7 + dv, device=DEV)
    h = h0.clone()
    href = h0.double().cpu().numpy().copy()
    for s in range(steps):
        o = gla.gla_recurrent_step(q[s], k[s], v[s], a[s], h)
        o_ref = og.step(_np32(q[s]), _np32(k[s]), _np32(v[s]), _np32(a[s]), dk ** -0.5, href)
        assert_close(_np32(o), o_ref, f"step {s} o", bf16_output=True)
    assert_close(h.cpu().numpy(), href, "final state")
    assert gla.gla_last_device_status() == 0


def test_decode_equals_chunked_prefill():
    B, H, T, dk, dv = 2, 3, 150, 128, 128
    q, k, v, a, h0 = make_chunk_inputs(B, H, T, dk, dv, sigma_h0=0.1, seed=11, device=DEV)
    o_pf, h_pf = gla.gla_chunk_fwd(q, k, v, a, None, h0)
    h = h0.clone()
    outs = []
    for t in range(T):
        outs.append(gla.gla_recurrent_step(q[:, :, t].contiguous(), k[:, :, t].contiguous(),
                                           v[:, :, t].contiguous(), a[:, :, t].contiguous(), h))
    o_dec = torch.stack(outs, dim=2)
    # Both paths against the oracle (two independently rounded bf16 outputs may
    # differ by a whole bf16 step, so they are not compared with each other).
    o_ref, h_ref = og.forward(_np32(q), _np32(k), _np32(v), _np32(a), dk ** -0.5,
                              h0.double().cpu().numpy())
    assert_close(_np32(o_dec), o_ref, "decode o", bf16_output=True)
    assert_close(_np32(o_pf), o_ref, "prefill o", bf16_output=True)
    assert_close(h.cpu().numpy(), h_ref, "decode state")
    assert_close(h_pf.cpu().numpy(), h_ref, "prefill state")
    # fp32 states of the two paths agree far inside the bar
    assert np.abs(h.cpu().numpy() - h_pf.cpu().numpy()).max() <= 1e-3 * np.sqrt(np.mean(h_ref ** 2))


def test_decode_config_sampled_heads_every_128_steps():
    cfg = DECODE_CONFIG
    h0, q, k, v, a = make_decode_inputs(cfg.B, cfg.H, cfg.dk, cfg.dv, cfg.steps,
                                        sigma_z=cfg.sigma_z, tau=cfg.tau, sigma_h0=cfg.sigma_h0,
                                        device=DEV)
    heads = [(0, 0), (17, 5), (101, 31), (255, 16), (128, 0), (64, 12)]
    bi = torch.tensor([b for b, _ in heads], device=DEV)
    hi = torch.tensor([h for _, h in heads], device=DEV)
    href = h0[bi, hi].double().cpu().numpy().copy()
    sq, sk, sv, sa = (_np32(t[:, bi, hi]) for t in (q, k, v, a))
    h = h0.clone()
    for s in range(cfg.steps):
        o = gla.gla_recurrent_step(q[s], k[s], v[s], a[s], h)
        o_ref = og.step(sq[s], sk[s], sv[s], sa[s], cfg.scale, href)
        if (s + 1) % cfg.check_every == 0:
            assert_close(_np32(o[bi, hi]), o_ref, f"step {s + 1} o", bf16_output=True)
            assert_close(h[bi, hi].cpu().numpy(), href, f"step {s + 1} state")
    assert gla.gla_last_device_status() == 0
