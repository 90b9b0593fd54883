"""GPU parity of gla_chunk_bwd (the chunkwise backward) against the fp64 oracle.

The oracle differentiates the token-by-token recurrence in reverse mode; the
CUDA path recomputes chunk-start states, runs the state-gradient pass and
then every chunk's gradients independently.  Each of the five gradients
(dq, dk, dv in bf16; dlog_alpha and dh0 in fp32) is held to the same bar as
the forward's outputs: relative L2 <= 1e-2 and max-abs <= 2e-2 * RMS.

The cases cover every (dk, dv) pair, ragged last chunks, sequences shorter
than one chunk, absent initial and final-state gradients, the exact
in-chunk decay path (forced, and taken by itself under near-zero gates), the
differentiable wrapper, and sampled heads of the long workload at full size.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import chunkwise_linear_rnn_gb300 as gla
from oracle import gla_oracle as og
from synth import make_backward_grads, make_chunk_inputs
from tolerance import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"
NAMES = ("dq", "dk", "dv", "dlog_alpha", "dh0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunkwise_linear_rnn_gb300.build import build
    build()
    og.build()


def _inputs(B, H, T, dk, dv, *, sigma_z=1.0, tau=16.0, h0=True, dhT=True, seed=0):
    q, k, v, a, s0 = make_chunk_inputs(B, H, T, dk, dv, sigma_z=sigma_z, tau=tau,
                                       sigma_h0=0.1 if h0 else None, seed=seed)
    d_o, g = make_backward_grads(B, H, T, dk, dv, sigma_dhT=0.1 if dhT else None, seed=seed)
    return q, k, v, a, s0, d_o, g


def _gpu(q, k, v, a, s0, d_o, g, scale, **kw):
    dev = lambda t: None if t is None else t.to(DEV)  # noqa: E731
    out = gla.gla_chunk_bwd(dev(q), dev(k), dev(v), dev(a), dev(d_o), scale, dev(s0), dev(g), **kw)
    torch.cuda.synchronize()
    return [None if x is None else x.float().cpu().numpy() for x in out]


def _oracle(q, k, v, a, s0, d_o, g, scale):
    np64 = lambda t: None if t is None else t.double().numpy()  # noqa: E731
    return og.backward(q.float().numpy(), k.float().numpy(), v.float().numpy(), a.numpy(), scale,
                       d_o.float().numpy(), np64(s0), np64(g))


def _compare(got, want, what):
    for name, x, ref in zip(NAMES, got, want):
        if x is None:
            continue
        assert_close(x, ref, f"{what} {name}", bf16_output=name in ("dq", "dk", "dv"))


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (64, 256), (128, 64), (128, 128),
                                   (128, 256)])
def test_head_dims_with_ragged_tail(dk, dv):
    T = 300  # four whole chunks of 64 and a tail of 44
    case = _inputs(1, 2, T, dk, dv, seed=dk + dv)
    scale = dk ** -0.5
    _compare(_gpu(*case, scale), _oracle(*case, scale), f"dk={dk} dv={dv}")


@pytest.mark.parametrize("T", [1, 37, 64, 65, 129])
def test_short_sequences(T):
    case = _inputs(2, 2, T, 64, 128, seed=T)
    _compare(_gpu(*case, 0.125), _oracle(*case, 0.125), f"T={T}")


def test_without_initial_state_or_final_gradient():
    case = _inputs(1, 3, 200, 128, 128, h0=False, dhT=False, seed=5)
    got = _gpu(*case, 0.1)
    _compare(got, _oracle(*case, 0.1), "no h0 / dhT")


def test_dh0_not_requested():
    case = _inputs(1, 2, 100, 64, 64, seed=6)
    got = _gpu(*case, 0.125, need_dh0=False)
    assert got[4] is None
    _compare(got, _oracle(*case, 0.125), "no dh0")


@pytest.mark.parametrize("sigma_z,tau", [(1.0, 16.0), (4.0, 1.0)])
def test_forced_exact_path(sigma_z, tau):
    case = _inputs(1, 2, 260, 128, 256, sigma_z=sigma_z, tau=tau, seed=7)
    scale = 128 ** -0.5
    want = _oracle(*case, scale)
    _compare(_gpu(*case, scale, force_exact=True), want, f"forced exact sz={sigma_z}")
    _compare(_gpu(*case, scale), want, f"automatic sz={sigma_z}")


def test_vanishing_gates_take_the_exact_path():
    """log alpha = -30 on some chunks: their decay spans far beyond 2^120."""
    q, k, v, a, s0, d_o, g = _inputs(1, 2, 256, 64, 128, seed=8)
    a = a.clone()
    a[:, :, 64:128] = -30.0
    a[:, 1, 200:210] = -30.0
    case = (q, k, v, a, s0, d_o, g)
    _compare(_gpu(*case, 0.125), _oracle(*case, 0.125), "vanishing gates")


def test_strong_decay_workload_spread():
    """The long workload's gate spread (sigma_z = 2) at a size the oracle covers in full."""
    case = _inputs(2, 2, 1000, 128, 256, sigma_z=2.0, seed=9)
    _compare(_gpu(*case, 128 ** -0.5), _oracle(*case, 128 ** -0.5), "sigma_z=2")


def test_differentiable_wrapper_matches_the_c_call():
    q, k, v, a, s0, d_o, g = [None if t is None else t.to(DEV) for t in _inputs(1, 2, 150, 64, 128,
                                                                               seed=10)]
    leaves = [t.clone().requires_grad_(True) for t in (q, k, v, a, s0)]
    o, hT = gla.gla_chunk(*leaves[:4], 0.125, leaves[4])
    ((o.float() * d_o.float()).sum() + (hT * g).sum()).backward()
    want = gla.gla_chunk_bwd(q, k, v, a, d_o, 0.125, s0, g)
    torch.cuda.synchronize()
    for name, leaf, ref in zip(NAMES, leaves, want):
        assert torch.equal(leaf.grad, ref), name


def test_full_size_long_workload_sampled_heads():
    """B2 H16 T32768 dk128 dv256 on the GPU; two heads checked in full against the oracle."""
    B, H, T, dk, dv = 2, 16, 32768, 128, 256
    q, k, v, a, s0 = make_chunk_inputs(B, H, T, dk, dv, sigma_z=2.0, sigma_h0=0.1, seed=0,
                                       device=DEV)
    d_o, g = make_backward_grads(B, H, T, dk, dv, sigma_dhT=0.1, seed=0, device=DEV)
    scale = dk ** -0.5
    out = gla.gla_chunk_bwd(q, k, v, a, d_o, scale, s0, g)
    torch.cuda.synchronize()
    for b, h in ((0, 0), (1, 15)):
        sl = lambda t: t[b:b + 1, h:h + 1].cpu()  # noqa: E731
        want = _oracle(sl(q), sl(k), sl(v), sl(a), sl(s0), sl(d_o), sl(g), scale)
        got = [x[b:b + 1, h:h + 1].float().cpu().numpy() for x in out]
        _compare(got, want, f"long workload head ({b},{h})")


def test_argument_errors():
    q, k, v, a, s0, d_o, g = [None if t is None else t.to(DEV) for t in _inputs(1, 1, 8, 64, 64)]
    with pytest.raises(ValueError):
        gla.gla_chunk_bwd(q, k, v, a, d_o[..., :32].contiguous(), 0.1)
    with pytest.raises(TypeError):
        gla.gla_chunk_bwd(q, k, v, a, d_o.float(), 0.1)


@pytest.mark.parametrize("dk,dv,T", [(64, 128, 300), (128, 256, 200), (128, 64, 65)])
def test_one_gate_per_head(dk, dv, T):
    """log_alpha [B,H,T]: one gate per token and head, used for every key channel.

    The oracle runs on the gate broadcast over the channels; the head gate's
    gradient is then the sum of the channel gates' gradients (chain rule)."""
    q, k, v, a, s0, d_o, g = _inputs(1, 2, T, dk, dv, sigma_z=2.0, seed=11 + dk + T)
    a1 = a[..., 0].contiguous()
    a_full = a1[..., None].expand(-1, -1, -1, dk).contiguous()
    scale = dk ** -0.5
    got = _gpu(q, k, v, a1, s0, d_o, g, scale)
    want = list(_oracle(q, k, v, a_full, s0, d_o, g, scale))
    want[3] = want[3].sum(axis=-1)
    assert got[3].shape == want[3].shape
    _compare(got, want, f"gate per head dk={dk} dv={dv} T={T}")


def test_differentiable_wrapper_with_one_gate_per_head():
    q, k, v, a, s0, d_o, g = [None if t is None else t.to(DEV) for t in _inputs(1, 2, 130, 64, 64,
                                                                               seed=12)]
    a1 = a[..., 0].contiguous()
    leaves = [t.clone().requires_grad_(True) for t in (q, k, v, a1, s0)]
    o, hT = gla.gla_chunk(*leaves[:4], 0.125, leaves[4])
    ((o.float() * d_o.float()).sum() + (hT * g).sum()).backward()
    want = gla.gla_chunk_bwd(q, k, v, a1, d_o, 0.125, s0, g)
    torch.cuda.synchronize()
    for name, leaf, ref in zip(NAMES, leaves, want):
        assert torch.equal(leaf.grad, ref), name


def _packed_case(lens, H, dk, dv, *, seed, states=True):
    T_total = int(sum(lens))
    q, k, v, a, _ = make_chunk_inputs(1, H, max(T_total, 1), dk, dv, sigma_z=2.0, seed=seed)
    q, k, v, a = (t[0, :, :T_total].contiguous() for t in (q, k, v, a))
    d_o, _ = make_backward_grads(1, H, max(T_total, 1), dk, dv, seed=seed)
    d_o = d_o[0, :, :T_total].contiguous()
    gen = torch.Generator().manual_seed(seed + 77)
    h0 = torch.randn(len(lens), H, dk, dv, generator=gen).mul_(0.1) if states else None
    dhT = torch.randn(len(lens), H, dk, dv, generator=gen).mul_(0.1) if states else None
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64).tolist()
    return q, k, v, a, d_o, h0, dhT, cu


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (128, 256)])
@pytest.mark.parametrize("states", [True, False])
def test_packed_sequences(dk, dv, states):
    """gla_chunk_bwd_varlen: each packed sequence against the oracle on its own rows."""
    lens = [1, 127, 0, 200, 65, 64, 513]
    q, k, v, a, d_o, h0, dhT, cu = _packed_case(lens, 2, dk, dv, seed=dk + dv, states=states)
    scale = dk ** -0.5
    dev = lambda t: None if t is None else t.to(DEV)  # noqa: E731
    out = gla.gla_chunk_bwd_varlen(dev(q), dev(k), dev(v), dev(a), dev(d_o), cu, scale, dev(h0),
                                   dev(dhT))
    torch.cuda.synchronize()
    out = [x.float().cpu().numpy() for x in out]
    for n in range(len(lens)):
        b, e = cu[n], cu[n + 1]
        if e == b:
            want = np.zeros((2, dk, dv)) if dhT is None else dhT[n].numpy()
            np.testing.assert_array_equal(out[4][n], want.astype(np.float32))
            continue
        sl = lambda t: t[:, b:e].unsqueeze(0)  # noqa: E731
        st = lambda t: None if t is None else t[n:n + 1]  # noqa: E731
        want = _oracle(sl(q), sl(k), sl(v), sl(a), st(h0), sl(d_o), st(dhT), scale)
        got = [out[0][:, b:e][None], out[1][:, b:e][None], out[2][:, b:e][None],
               out[3][:, b:e][None], out[4][n:n + 1]]
        if not np.any(want[3]):
            # one token from a zero state with no final-state gradient: q dq = k dk
            # exactly, so dlog_alpha is 0 and the RMS-relative bar degenerates; the
            # kernel's value is the fp32 rounding of that difference of O(1) terms
            assert np.max(np.abs(got[3])) <= 1e-5, f"packed seq {n}: dlog_alpha not ~0"
            got[3], want = None, list(want)
        _compare(got, want, f"packed seq {n} (len {e - b}) dk={dk} dv={dv}")


@pytest.mark.parametrize("name", ["medium", "very_long"])
def test_full_size_other_workloads_sampled_heads(name):
    """The medium (B8 H16 T2048 dk=dv=128) and very long (B1 H32 T262144 dk=dv=128)
    workloads at full size on the GPU; one head of each checked against the oracle."""
    from synth import CHUNK_CONFIGS
    cfg = CHUNK_CONFIGS[name]
    q, k, v, a, s0 = make_chunk_inputs(cfg.B, cfg.H, cfg.T, cfg.dk, cfg.dv, sigma_z=cfg.sigma_z,
                                       tau=cfg.tau, sigma_h0=cfg.sigma_h0, seed=0, device=DEV)
    d_o, g = make_backward_grads(cfg.B, cfg.H, cfg.T, cfg.dk, cfg.dv, seed=0, device=DEV)
    out = gla.gla_chunk_bwd(q, k, v, a, d_o, cfg.scale, s0, g)
    torch.cuda.synchronize()
    b, h = cfg.B - 1, cfg.H - 1
    sl = lambda t: None if t is None else t[b:b + 1, h:h + 1].cpu()  # noqa: E731
    want = _oracle(sl(q), sl(k), sl(v), sl(a), sl(s0), sl(d_o), sl(g), cfg.scale)
    got = [x[b:b + 1, h:h + 1].float().cpu().numpy() for x in out]
    _compare(got, want, f"{name} workload head ({b},{h})")


def test_gates_of_one():
    """log alpha = 0 (alpha = 1): causal linear attention with no decay at all."""
    q, k, v, a, s0, d_o, g = _inputs(1, 2, 200, 64, 128, seed=13)
    a = torch.zeros_like(a)
    case = (q, k, v, a, s0, d_o, g)
    _compare(_gpu(*case, 0.125), _oracle(*case, 0.125), "alpha = 1")


def test_many_heads_one_token():
    """B * H = 70,000 (beyond one grid dimension's 65,535) with T = 1."""
    q, k, v, a, s0, d_o, g = _inputs(7000, 10, 1, 64, 64, seed=14)
    case = (q, k, v, a, s0, d_o, g)
    _compare(_gpu(*case, 0.125), _oracle(*case, 0.125), "B*H = 70000, T = 1")


def test_differentiable_packed_wrapper_matches_the_c_call():
    lens = [70, 0, 130, 5]
    q, k, v, a, d_o, h0, dhT, cu = _packed_case(lens, 2, 64, 128, seed=15)
    q, k, v, a, d_o, h0, dhT = (t.to(DEV) for t in (q, k, v, a, d_o, h0, dhT))
    leaves = [t.clone().requires_grad_(True) for t in (q, k, v, a, h0)]
    o, hT = gla.gla_chunk_varlen(*leaves[:4], cu, 0.125, leaves[4])
    ((o.float() * d_o.float()).sum() + (hT * dhT).sum()).backward()
    want = gla.gla_chunk_bwd_varlen(q, k, v, a, d_o, cu, 0.125, h0, dhT)
    torch.cuda.synchronize()
    for name, leaf, ref in zip(NAMES, leaves, want):
        assert torch.equal(leaf.grad, ref), name
