"""GPU parity of gla_gdn_fwd (the gated delta rule, token-recurrent) and gla_gdn_chunk_fwd
(the same rule by chunks on the tensor cores) against the fp64 oracle.

The oracle walks the same recurrence in double on the exact bf16/fp32 input
values; the CUDA path keeps each state column in fp32 registers split over
lanes.  Outputs o (bf16) and hT (fp32) are held to the forward's bar:
relative L2 <= 1e-2 and max-abs <= 2e-2 * RMS.

Cases: every (dk, dv) pair with a ragged last round of staged tokens, a single
token, fewer tokens than one staged round, absent initial state and final
state, strong forgetting, writes at full strength, the degenerate gates
(beta = 0 leaves only the decay of h0), and sampled heads of the long
workload computed at full size.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import chunkwise_linear_rnn_gb300 as gla
from oracle import gdn_oracle as gd
from synth import make_gdn_inputs
from tolerance import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunkwise_linear_rnn_gb300.build import build
    build()
    gd.build()


def _gpu(q, k, v, g, b, h0, scale, **kw):
    dev = lambda t: None if t is None else t.to(DEV)  # noqa: E731
    o, hT = gla.gla_gdn_fwd(dev(q), dev(k), dev(v), dev(g), dev(b), scale, dev(h0), **kw)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), None if hT is None else hT.cpu().numpy()


def _oracle(q, k, v, g, b, h0, scale):
    return gd.forward(q.float().numpy(), k.float().numpy(), v.float().numpy(), g.numpy(),
                      b.numpy(), scale, None if h0 is None else h0.double().numpy())


def _check(case, scale, what, **kw):
    o, hT = _gpu(*case, scale, **kw)
    ro, rhT = _oracle(*case, scale)
    assert_close(o, ro, f"{what} o", bf16_output=True)
    if hT is not None:
        assert_close(hT, rhT, f"{what} hT")
    return o, hT, ro, rhT


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (64, 256), (128, 64), (128, 128),
                                   (128, 256)])
def test_head_dims_with_ragged_tail(dk, dv):
    T = 200  # six whole rounds of 32 staged tokens and a tail of 8
    case = make_gdn_inputs(2, 3, T, dk, dv, sigma_h0=0.1, seed=dk + dv)
    _check(case, dk ** -0.5, f"dk={dk} dv={dv}")


@pytest.mark.parametrize("T", [1, 5, 31, 33])
def test_short_sequences(T):
    case = make_gdn_inputs(1, 2, T, 128, 128, sigma_h0=0.1, seed=T)
    _check(case, 128 ** -0.5, f"T={T}")


def test_no_initial_state_and_no_final_state():
    q, k, v, g, b, _ = make_gdn_inputs(1, 4, 100, 64, 128, seed=3)
    o, hT = _gpu(q, k, v, g, b, None, 0.125, output_final_state=False)
    assert hT is None
    ro, _ = _oracle(q, k, v, g, b, None, 0.125)
    assert_close(o, ro, "no h0 o", bf16_output=True)


def test_strong_forgetting_and_full_writes():
    q, k, v, g, b, h0 = make_gdn_inputs(1, 2, 160, 128, 256, tau=1.0, sigma_z=3.0, sigma_h0=1.0,
                                        seed=11)
    _check((q, k, v, g, b, h0), 128 ** -0.5, "tau=1")
    _check((q, k, v, g, torch.ones_like(b), h0), 128 ** -0.5, "beta=1")


def test_beta_zero_only_decays_the_initial_state():
    q, k, v, g, b, h0 = make_gdn_inputs(1, 2, 70, 64, 64, sigma_h0=1.0, seed=5)
    o, hT, ro, rhT = _check((q, k, v, g, torch.zeros_like(b), h0), 0.125, "beta=0")
    decay = np.exp(g.double().numpy().sum(axis=-1))[..., None, None]
    np.testing.assert_allclose(hT, decay * h0.double().numpy(), rtol=1e-4, atol=1e-7)


def test_bad_arguments_are_rejected():
    q, k, v, g, b, h0 = make_gdn_inputs(1, 1, 8, 64, 64, seed=0)
    dev = lambda t: t.to(DEV)  # noqa: E731
    with pytest.raises(Exception):
        gla.gla_gdn_fwd(dev(q)[..., :48].contiguous(), dev(k)[..., :48].contiguous(), dev(v),
                        dev(g), dev(b))
    with pytest.raises(Exception):
        gla.gla_gdn_fwd(dev(q), dev(k), dev(v), dev(g).double(), dev(b))
    # q one element off a 16-byte boundary: refused on the host, nothing launched
    flat = torch.empty(q.numel() + 8, dtype=torch.bfloat16, device=DEV)
    q_off = flat[1:1 + q.numel()].view(q.shape)
    q_off.copy_(dev(q))
    with pytest.raises(Exception):
        gla.gla_gdn_fwd(q_off, dev(k), dev(v), dev(g), dev(b))


def test_long_workload_sampled_heads():
    B, H, T, dk, dv = 2, 16, 32768, 128, 256
    q, k, v, g, b, h0 = make_gdn_inputs(B, H, T, dk, dv, sigma_h0=0.1, seed=7, device=DEV)
    o, hT = gla.gla_gdn_fwd(q, k, v, g, b, dk ** -0.5, h0)
    torch.cuda.synchronize()
    for n, h in ((0, 0), (1, 13)):
        ro, rhT = gd.forward(q[n, h].float().cpu().numpy(), k[n, h].float().cpu().numpy(),
                             v[n, h].float().cpu().numpy(), g[n, h].cpu().numpy(),
                             b[n, h].cpu().numpy(), dk ** -0.5, h0[n, h].double().cpu().numpy())
        assert_close(o[n, h].float().cpu().numpy(), ro, f"long ({n},{h}) o", bf16_output=True)
        assert_close(hT[n, h].cpu().numpy(), rhT, f"long ({n},{h}) hT")


# ---- gla_gdn_chunk_fwd: the same recurrence by the four-step chunk algorithm on
# the tensor cores (64-token chunks, dk = 128), against the same oracle.

@pytest.mark.parametrize("dv", [64, 128, 256])
@pytest.mark.parametrize("T", [1, 37, 63, 64, 65, 200, 1000])
def test_chunked_matches_oracle(dv, T):
    case = make_gdn_inputs(1, 3, T, 128, dv, sigma_h0=0.1, seed=T + dv)
    _check(case, 128 ** -0.5, f"chunked T={T} dv={dv}", chunked=True)


def test_chunked_without_states_and_with_several_batches():
    q, k, v, g, b, _ = make_gdn_inputs(3, 2, 300, 128, 128, seed=21)
    o, hT = _gpu(q, k, v, g, b, None, 0.1, output_final_state=False, chunked=True)
    assert hT is None
    ro, _ = _oracle(q, k, v, g, b, None, 0.1)
    assert_close(o, ro, "chunked no h0 o", bf16_output=True)


def test_chunked_strong_forgetting_full_writes_and_beta_zero():
    q, k, v, g, b, h0 = make_gdn_inputs(1, 2, 260, 128, 256, tau=1.0, sigma_z=3.0, sigma_h0=1.0,
                                        seed=23)
    _check((q, k, v, g, b, h0), 128 ** -0.5, "chunked tau=1", chunked=True)
    _check((q, k, v, g, torch.ones_like(b), h0), 128 ** -0.5, "chunked beta=1", chunked=True)
    # beta = 0 on the default gates: the state only decays (the gates above would take it
    # below the fp32 range within these 260 tokens)
    q, k, v, g, b, h0 = make_gdn_inputs(1, 2, 260, 128, 128, sigma_h0=1.0, seed=24)
    o, hT, ro, rhT = _check((q, k, v, g, torch.zeros_like(b), h0), 128 ** -0.5,
                            "chunked beta=0", chunked=True)
    decay = np.exp(g.double().numpy().sum(axis=-1))[..., None, None]
    np.testing.assert_allclose(hT, decay * h0.double().numpy(), rtol=1e-4, atol=1e-7)


def test_chunked_more_sequential_ctas_than_sms():
    # B*H = 64 heads at dv = 256: 256 sequential-kernel CTAs (one per head and
    # 64-column tile, one per SM) run in two waves; the WY pre-pass has 1,280
    # CTAs; a ragged last chunk
    q, k, v, g, b, h0 = make_gdn_inputs(4, 16, 300, 128, 256, sigma_h0=0.1, seed=26)
    o, hT = _gpu(q, k, v, g, b, h0, 128 ** -0.5, chunked=True)
    ro, rhT = _oracle(q, k, v, g, b, h0, 128 ** -0.5)
    assert_close(o, ro, "chunked 64 heads o", bf16_output=True)
    assert_close(hT, rhT, "chunked 64 heads hT")


def test_chunked_agrees_with_the_token_recurrent_kernel():
    case = make_gdn_inputs(2, 2, 500, 128, 128, sigma_h0=0.1, seed=25)
    o_c, h_c = _gpu(*case, 128 ** -0.5, chunked=True)
    o_t, h_t = _gpu(*case, 128 ** -0.5)
    assert_close(o_c, o_t.astype(np.float64), "chunked vs token o", bf16_output=True)
    assert_close(h_c, h_t.astype(np.float64), "chunked vs token hT")


def test_chunked_rejects_other_key_widths():
    q, k, v, g, b, h0 = make_gdn_inputs(1, 1, 8, 64, 64, seed=0)
    dev = lambda t: t.to(DEV)  # noqa: E731
    with pytest.raises(Exception):
        gla.gla_gdn_fwd(dev(q), dev(k), dev(v), dev(g), dev(b), chunked=True)


def test_chunked_long_workload_sampled_heads():
    B, H, T, dk, dv = 2, 16, 32768, 128, 256
    q, k, v, g, b, h0 = make_gdn_inputs(B, H, T, dk, dv, sigma_h0=0.1, seed=7, device=DEV)
    o, hT = gla.gla_gdn_fwd(q, k, v, g, b, dk ** -0.5, h0, chunked=True)
    torch.cuda.synchronize()
    for n, h in ((0, 0), (1, 13)):
        ro, rhT = gd.forward(q[n, h].float().cpu().numpy(), k[n, h].float().cpu().numpy(),
                             v[n, h].float().cpu().numpy(), g[n, h].cpu().numpy(),
                             b[n, h].cpu().numpy(), dk ** -0.5, h0[n, h].double().cpu().numpy())
        assert_close(o[n, h].float().cpu().numpy(), ro, f"chunked long ({n},{h}) o",
                     bf16_output=True)
        assert_close(hT[n, h].cpu().numpy(), rhT, f"chunked long ({n},{h}) hT")
