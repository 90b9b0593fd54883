"""GPU parity of the chunked forward with one gate per token and head (log_alpha [B, H, T]).

The gate of every key channel is the token's one gate: the oracle runs on
that gate broadcast over the channels.  The per-head case is also compared
with the per-channel kernel fed the broadcast gate, which computes exactly
the same operations (same prefix sums, same rescaling), so the two outputs
agree bit for bit.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import chunkwise_linear_rnn_gb300 as gla
from oracle import gla_oracle as og
from synth import make_chunk_inputs
from tolerance import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunkwise_linear_rnn_gb300.build import build
    build()
    og.build()


def _inputs(B, H, T, dk, dv, *, seed=0, sigma_z=1.0, tau=16.0, h0=True):
    q, k, v, a, s0 = make_chunk_inputs(B, H, T, dk, dv, sigma_z=sigma_z, tau=tau,
                                       sigma_h0=0.1 if h0 else None, seed=seed)
    g = a[..., 0].contiguous()          # one gate per (b, h, t): the first channel's draw
    return q, k, v, g, s0


def _check(q, k, v, g, s0, what, **kw):
    dk = q.shape[-1]
    scale = dk ** -0.5
    dev = lambda t: None if t is None else t.to(DEV)  # noqa: E731
    o, hT = gla.gla_chunk_fwd(dev(q), dev(k), dev(v), dev(g), scale, dev(s0), **kw)
    torch.cuda.synchronize()
    assert gla.gla_last_device_status() == 0
    a4 = g[..., None].expand(*g.shape, dk).contiguous()
    cpu = lambda t: t.float().numpy()  # noqa: E731
    o_ref, h_ref = og.forward(cpu(q), cpu(k), cpu(v), cpu(a4), scale,
                              None if s0 is None else s0.double().numpy())
    assert_close(o.float().cpu().numpy(), o_ref, f"{what} o", bf16_output=True)
    assert_close(hT.cpu().numpy(), h_ref, f"{what} hT")
    return o, hT


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64), (128, 128), (128, 256)])
def test_head_dims(dk, dv):
    _check(*_inputs(1, 2, 300, dk, dv, seed=dk + dv), f"dk={dk} dv={dv}")


@pytest.mark.parametrize("T", [1, 129, 257])
def test_ragged_lengths(T):
    _check(*_inputs(2, 2, T, 128, 256, seed=T), f"T={T}")


def test_independent_tiles():
    _check(*_inputs(1, 2, 300, 128, 256, seed=3), "cta_pair=-1", cta_pair=-1)


@pytest.mark.parametrize("segments", [2, 3])
def test_segments(segments):
    _check(*_inputs(1, 2, 2100, 128, 128, seed=10 + segments), f"segments={segments}",
           segments=segments)


def test_pair_segments():
    _check(*_inputs(1, 2, 1500, 128, 256, seed=20), "pair segments=3", segments=3)


def test_sub_chunk_path():
    _check(*_inputs(1, 2, 300, 128, 128, seed=21, sigma_z=2.0), "force_exact", force_exact=True)


def test_constant_decay_per_head():
    # RetNet: a fixed decay per head, gamma_h = 1 - 2^-(5 + h)
    q, k, v, _, s0 = _inputs(1, 4, 640, 128, 128, seed=22)
    gam = torch.tensor([1.0 - 2.0 ** -(5 + h) for h in range(4)])
    g = torch.log(gam)[None, :, None].expand(1, 4, 640).contiguous().float()
    _check(q, k, v, g, s0, "retnet decays")


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 256)])
def test_equals_the_per_channel_kernel_on_the_broadcast_gate(dk, dv):
    q, k, v, g, s0 = _inputs(1, 2, 700, dk, dv, seed=30 + dk)
    a4 = g[..., None].expand(*g.shape, dk).contiguous()
    dev = lambda t: t.to(DEV)  # noqa: E731
    o1, h1 = gla.gla_chunk_fwd(dev(q), dev(k), dev(v), dev(g), None, dev(s0))
    o2, h2 = gla.gla_chunk_fwd(dev(q), dev(k), dev(v), dev(a4), None, dev(s0))
    torch.cuda.synchronize()
    assert gla.gla_last_device_status() == 0
    assert torch.equal(o1, o2)
    assert torch.equal(h1, h2)
