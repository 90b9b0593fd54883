"""GPU parity of gla_chunk_fwd_host (host buffers, copies pipelined with the
forward) against the fp64 oracle, through the C ABI."""

from __future__ import annotations

import pytest
import torch

import chunkwise_linear_rnn_gb300 as gla
from oracle import gla_oracle as og
from synth import make_chunk_inputs
from tolerance import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunkwise_linear_rnn_gb300.build import build
    build()
    og.build()


def _oracle(q, k, v, a, scale, h0):
    f = lambda t: t.float().numpy()  # noqa: E731
    return og.forward(f(q), f(k), f(v), f(a), scale, None if h0 is None else h0.double().numpy())


def _run(q, k, v, a, h0, what, pin=True, **kw):
    if pin:
        q, k, v, a = (t.pin_memory() for t in (q, k, v, a))
        h0 = None if h0 is None else h0.pin_memory()
    scale = q.shape[-1] ** -0.5
    o, hT = gla.gla_chunk_fwd_host(q, k, v, a, scale, h0, **kw)
    torch.cuda.synchronize()
    assert gla.gla_last_device_status() == 0
    o_ref, h_ref = _oracle(q, k, v, a, scale, h0)
    assert_close(o.float().numpy(), o_ref, f"{what} o", bf16_output=True)
    if hT is not None:
        assert_close(hT.numpy(), h_ref, f"{what} hT")
    return o, hT


@pytest.mark.parametrize("B,H,T,dk,dv", [(2, 3, 300, 128, 256), (1, 9, 257, 64, 128),
                                         (1, 1, 129, 128, 128), (4, 4, 200, 128, 64)])
def test_host_entry_matches_oracle(B, H, T, dk, dv):
    q, k, v, a, h0 = make_chunk_inputs(B, H, T, dk, dv, sigma_h0=0.1, seed=B * 100 + H + T)
    _run(q, k, v, a, h0, f"host B{B} H{H} T{T} {dk}/{dv}")


def test_host_entry_pageable_buffers():
    q, k, v, a, h0 = make_chunk_inputs(2, 2, 200, 128, 128, sigma_h0=0.1, seed=3)
    _run(q, k, v, a, h0, "pageable", pin=False)


def test_host_entry_without_states():
    q, k, v, a, _ = make_chunk_inputs(1, 5, 140, 128, 256, seed=4)
    o, hT = _run(q, k, v, a, None, "no h0 / no hT", output_final_state=False)
    assert hT is None


def test_host_entry_state_in_place():
    q, k, v, a, h0 = make_chunk_inputs(1, 10, 190, 64, 64, sigma_h0=0.1, seed=5)
    h = h0.clone().pin_memory()
    q, k, v, a = (t.pin_memory() for t in (q, k, v, a))
    o_ref, h_ref = _oracle(q, k, v, a, 64 ** -0.5, h0)
    o, hT = gla.gla_chunk_fwd_host(q, k, v, a, None, h, final_state=h)
    torch.cuda.synchronize()
    assert hT.data_ptr() == h.data_ptr()
    assert_close(o.float().numpy(), o_ref, "in-place o", bf16_output=True)
    assert_close(h.numpy(), h_ref, "in-place hT")


def test_host_entry_agrees_with_device_entry():
    q, k, v, a, h0 = make_chunk_inputs(2, 8, 1024, 128, 256, sigma_z=2.0, sigma_h0=0.1, seed=6)
    o_h, h_h = gla.gla_chunk_fwd_host(q.pin_memory(), k.pin_memory(), v.pin_memory(),
                                      a.pin_memory(), None, h0.pin_memory())
    o_d, h_d = gla.gla_chunk_fwd(q.cuda(), k.cuda(), v.cuda(), a.cuda(), None, h0.cuda())
    torch.cuda.synchronize()
    o_ref, h_ref = _oracle(q, k, v, a, 128 ** -0.5, h0)
    assert_close(o_h.float().numpy(), o_ref, "host o", bf16_output=True)
    assert_close(o_d.float().cpu().numpy(), o_ref, "device o", bf16_output=True)
    assert_close(h_h.numpy(), h_ref, "host hT")
    assert_close(h_d.cpu().numpy(), h_ref, "device hT")
