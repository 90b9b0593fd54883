"""The seeded input generators (``synth/``) keep their stated recipes.

Both sides of every parity test are fed from these functions, so their
determinism, draw order, value domains and the workload table are checked
here on the CPU: the same seed gives the same tensors, the documented draw
order reproduces them from a fresh generator, gates are log-values of
numbers in (0, 1), write strengths lie in (0, 1), the gated delta rule's keys
have unit norm up to bf16 rounding, and the bench workload has the sizes it
is quoted with.
"""

from __future__ import annotations

import torch
import torch.nn.functional as F

from synth import (CHUNK_CONFIGS, DECODE_CONFIG, make_backward_grads, make_chunk_inputs,
                   make_config_inputs, make_decode_inputs, make_gdn_inputs)


def _same(a, b):
    return all((x is None and y is None) or torch.equal(x, y) for x, y in zip(a, b))


def test_same_seed_same_tensors_other_seed_other_tensors():
    for make in (lambda s: make_chunk_inputs(1, 2, 40, 8, 4, sigma_h0=0.1, seed=s),
                 lambda s: make_gdn_inputs(1, 2, 40, 8, 4, sigma_h0=0.1, seed=s),
                 lambda s: make_decode_inputs(2, 2, 8, 4, 3, seed=s),
                 lambda s: make_backward_grads(1, 2, 40, 8, 4, sigma_dhT=0.1, seed=s)):
        assert _same(make(3), make(3))
        assert not torch.equal(make(3)[0], make(4)[0])


def test_chunk_inputs_follow_the_stated_draw_order():
    B, H, T, dk, dv, sz, tau = 1, 2, 33, 8, 4, 2.0, 16.0
    q, k, v, a, h0 = make_chunk_inputs(B, H, T, dk, dv, sigma_z=sz, tau=tau, sigma_h0=0.1, seed=5)
    g = torch.Generator().manual_seed(5)
    z = torch.randn(B, H, T, dk, generator=g) * sz
    assert torch.equal(q, torch.randn(B, H, T, dk, generator=g).to(torch.bfloat16))
    assert torch.equal(k, torch.randn(B, H, T, dk, generator=g).to(torch.bfloat16))
    assert torch.equal(v, torch.randn(B, H, T, dv, generator=g).to(torch.bfloat16))
    assert torch.equal(h0, torch.randn(B, H, dk, dv, generator=g) * 0.1)
    torch.testing.assert_close(a, F.logsigmoid(z) / tau, rtol=0, atol=0)


def test_backward_gradients_use_the_next_seed():
    d_o, dhT = make_backward_grads(1, 2, 9, 8, 4, sigma_dhT=0.1, seed=7)
    g = torch.Generator().manual_seed(8)
    assert torch.equal(d_o, torch.randn(1, 2, 9, 4, generator=g).to(torch.bfloat16))
    assert torch.equal(dhT, torch.randn(1, 2, 8, 4, generator=g) * 0.1)


def test_domains_and_types():
    q, k, v, a, h0 = make_chunk_inputs(2, 3, 50, 16, 8, sigma_z=3.0, seed=1)
    assert q.dtype == k.dtype == v.dtype == torch.bfloat16 and a.dtype == torch.float32
    assert h0 is None and torch.isfinite(a).all() and (a < 0).all()
    qg, kg, vg, gg, bg, hg = make_gdn_inputs(2, 3, 50, 16, 8, sigma_z=3.0, sigma_h0=0.5, seed=1)
    assert qg.dtype == kg.dtype == vg.dtype == torch.bfloat16
    assert gg.shape == bg.shape == (2, 3, 50) and gg.dtype == bg.dtype == torch.float32
    assert torch.isfinite(gg).all() and (gg < 0).all() and (bg > 0).all() and (bg < 1).all()
    norms = kg.float().norm(dim=-1)
    assert ((norms - 1).abs() <= 2 ** -7).all()      # unit keys, up to the bf16 rounding of each entry
    assert hg.shape == (2, 3, 16, 8) and hg.dtype == torch.float32


def test_workload_table():
    long = CHUNK_CONFIGS["long"]
    assert (long.B, long.H, long.T, long.dk, long.dv) == (2, 16, 32768, 128, 256)
    assert long.sigma_h0 == 0.1 and long.tau == 16
    assert long.tokens == 2 * 16 * 32768 and abs(long.scale - 128 ** -0.5) < 1e-12
    small = CHUNK_CONFIGS["small"]
    assert (small.B, small.H, small.T, small.dk, small.dv) == (1, 2, 256, 64, 64)
    assert (DECODE_CONFIG.B, DECODE_CONFIG.H, DECODE_CONFIG.dk, DECODE_CONFIG.dv) == (256, 32, 128, 128)
    q, _, _, _, h0 = make_config_inputs(small, seed=0)
    assert q.shape == (1, 2, 256, 64) and h0 is None
