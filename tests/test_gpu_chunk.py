"""GPU parity of gla_chunk_fwd (through the C ABI) against the fp64 oracle.

Small and ragged cases are compared element by element over every head; the
full-size workloads are compared on sampled heads (heads are independent
sequences, so the oracle runs those heads in full, every token).
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import chunkwise_linear_rnn_gb300 as gla
from oracle import gla_oracle as og
from synth import CHUNK_CONFIGS, make_chunk_inputs, make_config_inputs
from tolerance import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunkwise_linear_rnn_gb300.build import build
    build()
    og.build()


def _oracle(q, k, v, a, scale, h0, heads=None):
    """Oracle on the exact GPU inputs; heads = list of (b, h) or None for all."""
    def cpu(t):
        return t.detach().float().cpu().numpy()
    if heads is None:
        return og.forward(cpu(q), cpu(k), cpu(v), cpu(a), scale,
                          None if h0 is None else h0.double().cpu().numpy())
    sel = lambda t: torch.stack([t[b, h] for b, h in heads])  # noqa: E731
    o, hT = og.forward(cpu(sel(q)), cpu(sel(k)), cpu(sel(v)), cpu(sel(a)), scale,
                       None if h0 is None else sel(h0).double().cpu().numpy())
    return o, hT


def _run_and_check(q, k, v, a, h0, what, heads=None, **kw):
    scale = q.shape[-1] ** -0.5
    o, hT = gla.gla_chunk_fwd(q, k, v, a, scale, h0, **kw)
    torch.cuda.synchronize()
    assert gla.gla_last_device_status() == 0
    o_ref, h_ref = _oracle(q, k, v, a, scale, h0, heads)
    if heads is not None:
        o = torch.stack([o[b, h] for b, h in heads])
        hT = torch.stack([hT[b, h] for b, h in heads])
    r1 = assert_close(o.float().cpu().numpy(), o_ref, f"{what} o", bf16_output=True)
    r2 = assert_close(hT.cpu().numpy(), h_ref, f"{what} hT")
    return r1, r2


def _inputs(B, H, T, dk, dv, *, h0=False, sigma_z=1.0, tau=16.0, seed=0):
    q, k, v, a, s0 = make_chunk_inputs(B, H, T, dk, dv, sigma_z=sigma_z, tau=tau,
                                       sigma_h0=0.1 if h0 else None, seed=seed, device="cpu")
    to = lambda t: None if t is None else t.to(DEV)  # noqa: E731
    return to(q), to(k), to(v), to(a), to(s0)


def test_small_config_all_heads():
    cfg = CHUNK_CONFIGS["small"]
    q, k, v, a, h0 = (None if t is None else t.to(DEV) for t in make_config_inputs(cfg))
    _run_and_check(q, k, v, a, h0, cfg.name)


@pytest.mark.parametrize("T", [1, 2, 63, 127, 128, 129, 255, 300, 513])
def test_ragged_lengths(T):
    q, k, v, a, h0 = _inputs(2, 3, T, 64, 64, h0=True, seed=T)
    _run_and_check(q, k, v, a, h0, f"T={T}")


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (64, 256), (128, 64), (128, 128),
                                   (128, 256)])
def test_head_dims(dk, dv):
    q, k, v, a, h0 = _inputs(1, 2, 200, dk, dv, h0=True, seed=dk + dv)
    _run_and_check(q, k, v, a, h0, f"dk={dk} dv={dv}")


@pytest.mark.parametrize("dv_tile", [64, 128])
def test_dv_tile_does_not_change_results(dv_tile):
    q, k, v, a, h0 = _inputs(1, 2, 300, 128, 256, h0=True, seed=5)
    _run_and_check(q, k, v, a, h0, f"dv_tile={dv_tile}", dv_tile=dv_tile)


def test_no_initial_state_and_no_final_state():
    q, k, v, a, _ = _inputs(2, 2, 130, 128, 128, seed=3)
    o, hT = gla.gla_chunk_fwd(q, k, v, a, None, None, output_final_state=False)
    assert hT is None
    o_ref, _ = _oracle(q, k, v, a, 128 ** -0.5, None)
    assert_close(o.float().cpu().numpy(), o_ref, "no h0 / no hT", bf16_output=True)


def test_final_state_may_alias_initial_state():
    q, k, v, a, h0 = _inputs(1, 3, 257, 64, 128, h0=True, seed=4)
    h = h0.clone()
    o_ref, h_ref = _oracle(q, k, v, a, 64 ** -0.5, h0)
    o, hT = gla.gla_chunk_fwd(q, k, v, a, None, h, final_state=h)
    assert hT.data_ptr() == h.data_ptr()
    assert_close(o.float().cpu().numpy(), o_ref, "aliased o", bf16_output=True)
    assert_close(h.cpu().numpy(), h_ref, "aliased hT")


def test_vanishing_gates_take_the_exact_path():
    # log alpha = -30 per token: the in-chunk decay leaves the fast path's bounded domain.
    q, k, v, a, h0 = _inputs(1, 2, 200, 64, 64, h0=True, seed=6)
    a = torch.full_like(a, -30.0)
    _run_and_check(q, k, v, a, h0, "log alpha = -30")


def test_gate_of_one_is_linear_attention():
    q, k, v, a, h0 = _inputs(1, 2, 256, 128, 64, h0=True, seed=7)
    a = torch.zeros_like(a)
    _run_and_check(q, k, v, a, h0, "alpha = 1")


def test_forced_sub_chunk_rescaling_matches_oracle():
    q, k, v, a, h0 = _inputs(1, 2, 300, 128, 128, h0=True, seed=8, sigma_z=2.0)
    _run_and_check(q, k, v, a, h0, "force_exact", force_exact=True)


def test_gates_beyond_the_exponent_bound_are_exact():
    # single tokens with log alpha far below -30: sub-chunks of one token, clamped gate
    q, k, v, a, h0 = _inputs(1, 2, 260, 64, 128, h0=True, seed=12)
    a[..., 5, :] = -200.0
    a[..., 130:140, 3] = -45.0
    _run_and_check(q, k, v, a, h0, "log alpha = -200 / -45 spikes")


@pytest.mark.parametrize("segments", [2, 3, 5])
def test_sequence_segments_match_oracle(segments):
    q, k, v, a, h0 = _inputs(1, 2, 2600, 128, 128, h0=True, seed=20 + segments)
    _run_and_check(q, k, v, a, h0, f"segments={segments}", segments=segments)


def test_segments_with_slow_decay_recompute_whole_segments():
    # alpha = 1: the start state never fades, every segment is recomputed from the scan
    q, k, v, a, h0 = _inputs(1, 2, 1100, 64, 64, h0=True, seed=31)
    a = torch.zeros_like(a)
    _run_and_check(q, k, v, a, h0, "alpha=1 segments=4", segments=4)


def test_segments_with_aliased_state():
    q, k, v, a, h0 = _inputs(2, 1, 1500, 128, 256, h0=True, seed=32)
    h = h0.clone()
    o_ref, h_ref = _oracle(q, k, v, a, 128 ** -0.5, h0)
    o, hT = gla.gla_chunk_fwd(q, k, v, a, None, h, final_state=h, segments=3)
    assert_close(o.float().cpu().numpy(), o_ref, "segments aliased o", bf16_output=True)
    assert_close(h.cpu().numpy(), h_ref, "segments aliased hT")


def test_segment_count_does_not_change_results_beyond_tolerance():
    q, k, v, a, h0 = _inputs(1, 1, 2048, 128, 128, h0=True, seed=33)
    outs = [gla.gla_chunk_fwd(q, k, v, a, None, h0, segments=s) for s in (1, 2, 4)]
    o_ref, h_ref = _oracle(q, k, v, a, 128 ** -0.5, h0)
    for o, hT in outs:
        assert_close(o.float().cpu().numpy(), o_ref, "segment sweep o", bf16_output=True)
        assert_close(hT.cpu().numpy(), h_ref, "segment sweep hT")


def test_mixed_fast_and_exact_chunks():
    q, k, v, a, h0 = _inputs(1, 1, 640, 128, 128, h0=True, seed=9)
    a[..., 128:256, :] = -1.0     # chunk 1 leaves the bounded domain, its neighbours do not
    _run_and_check(q, k, v, a, h0, "mixed chunks")


def test_split_sequence_equals_one_call():
    q, k, v, a, h0 = _inputs(1, 2, 400, 128, 128, h0=True, seed=10)
    o, hT = gla.gla_chunk_fwd(q, k, v, a, None, h0)
    T1 = 200  # not a chunk boundary
    o1, h1 = gla.gla_chunk_fwd(q[:, :, :T1].contiguous(), k[:, :, :T1].contiguous(),
                               v[:, :, :T1].contiguous(), a[:, :, :T1].contiguous(), None, h0)
    o2, h2 = gla.gla_chunk_fwd(q[:, :, T1:].contiguous(), k[:, :, T1:].contiguous(),
                               v[:, :, T1:].contiguous(), a[:, :, T1:].contiguous(), None, h1)
    ref_o, ref_h = _oracle(q, k, v, a, 128 ** -0.5, h0)
    assert_close(torch.cat([o1, o2], dim=2).float().cpu().numpy(), ref_o, "split o",
                 bf16_output=True)
    assert_close(h2.cpu().numpy(), ref_h, "split hT")
    assert_close(o.float().cpu().numpy(), ref_o, "whole o", bf16_output=True)


# ---- CTA pairs: dk = 128 with two value-column tiles (dv = 256, or dv = 128 at
# tile 64) runs each head's tiles as a 2-CTA cluster that splits the key-side
# preparation between them.  Each case is checked against the oracle, with and
# without pairs.

@pytest.mark.parametrize("cta_pair", [0, -1])
@pytest.mark.parametrize("dv,dv_tile,T", [(256, 0, 300), (256, 128, 129), (128, 64, 513),
                                          (256, 0, 1)])
def test_cta_pair_matches_oracle(dv, dv_tile, T, cta_pair):
    q, k, v, a, h0 = _inputs(2, 2, T, 128, dv, h0=True, seed=40 + T + dv)
    _run_and_check(q, k, v, a, h0, f"pair={cta_pair} dv={dv} tile={dv_tile} T={T}",
                   dv_tile=dv_tile, cta_pair=cta_pair)


def test_cta_pair_one_half_breaks_the_bound():
    # gate spikes only in key channels 0-63 (the first CTA's half) and only in
    # channels 64-127 in a later chunk: both CTAs must take the sub-chunk path
    q, k, v, a, h0 = _inputs(1, 2, 520, 128, 256, h0=True, seed=41)
    a[..., 10, 0:64] = -80.0
    a[..., 300:310, 100] = -40.0
    _run_and_check(q, k, v, a, h0, "pair spikes")


def test_cta_pair_forced_sub_chunks():
    q, k, v, a, h0 = _inputs(1, 2, 300, 128, 256, h0=True, seed=42, sigma_z=2.0)
    _run_and_check(q, k, v, a, h0, "pair force_exact", force_exact=True)


@pytest.mark.parametrize("segments", [2, 4])
def test_cta_pair_segments(segments):
    q, k, v, a, h0 = _inputs(1, 2, 2300, 128, 256, h0=True, seed=43 + segments)
    _run_and_check(q, k, v, a, h0, f"pair segments={segments}", segments=segments)


def test_cta_pair_segments_without_decay():
    # alpha = 1 in every channel: the correction window spans whole segments
    q, k, v, a, h0 = _inputs(1, 1, 1100, 128, 256, h0=True, seed=45)
    a = torch.zeros_like(a)
    _run_and_check(q, k, v, a, h0, "pair alpha=1 segments=3", segments=3)


def test_cta_pair_window_closes_in_one_half_first():
    # channels 64-127 decay fast, channels 0-63 slowly: the window stays open
    # until the slow half has decayed too, a decision both CTAs must share
    q, k, v, a, h0 = _inputs(1, 1, 2600, 128, 256, h0=True, seed=46)
    a[..., 0:64] = -0.002
    a[..., 64:128] = -0.5
    _run_and_check(q, k, v, a, h0, "pair split window", segments=3)


def test_cta_pair_aliased_state():
    q, k, v, a, h0 = _inputs(2, 1, 700, 128, 256, h0=True, seed=47)
    h = h0.clone()
    o_ref, h_ref = _oracle(q, k, v, a, 128 ** -0.5, h0)
    o, hT = gla.gla_chunk_fwd(q, k, v, a, None, h, final_state=h, segments=2)
    assert_close(o.float().cpu().numpy(), o_ref, "pair aliased o", bf16_output=True)
    assert_close(h.cpu().numpy(), h_ref, "pair aliased hT")


def test_medium_config_all_heads():
    cfg = CHUNK_CONFIGS["medium"]
    q, k, v, a, h0 = make_config_inputs(cfg, device=DEV)
    _run_and_check(q, k, v, a, h0, cfg.name)


def test_long_config_sampled_heads():
    cfg = CHUNK_CONFIGS["long"]
    q, k, v, a, h0 = make_config_inputs(cfg, device=DEV)
    _run_and_check(q, k, v, a, h0, cfg.name, heads=[(0, 0), (1, 7), (1, 15)])


def test_very_long_config_sampled_heads():
    cfg = CHUNK_CONFIGS["very_long"]
    q, k, v, a, h0 = make_config_inputs(cfg, device=DEV)
    _run_and_check(q, k, v, a, h0, cfg.name, heads=[(0, 3), (0, 30)])
