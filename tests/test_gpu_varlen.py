"""GPU parity of gla_chunk_fwd_varlen (packed variable-length batches) against the oracle.

Each packed sequence is an independent recurrence with its own initial and
final state, so the oracle runs on each sequence's slice on its own, every
token, and the kernel's rows for that sequence are compared element by
element.  The cases cover lengths that end inside a chunk (their tail tile
holds the next sequence's rows), empty sequences, the CTA-pair and
single-CTA paths, sequences cut into segments, and the sub-chunk path.
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


def _packed_inputs(lens, H, dk, dv, *, h0=True, seed=0, sigma_z=1.0):
    """Inputs for a packed batch: [H, T_total, d] tensors and cu_seqlens."""
    T_total = int(sum(lens))
    q, k, v, a, _ = make_chunk_inputs(1, H, max(T_total, 1), dk, dv, sigma_z=sigma_z, seed=seed)
    q, k, v, a = (t[0, :, :T_total].contiguous() for t in (q, k, v, a))
    s0 = None
    if h0:
        g = torch.Generator().manual_seed(seed + 1000)
        s0 = torch.randn(len(lens), H, dk, dv, generator=g).mul_(0.1)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64).tolist()
    return q, k, v, a, s0, cu


def _check(q, k, v, a, s0, cu, what, **kw):
    H, T_total, dk = q.shape
    dv = v.shape[-1]
    scale = dk ** -0.5
    dev = lambda t: None if t is None else t.to(DEV)  # noqa: E731
    o, hT = gla.gla_chunk_fwd_varlen(dev(q), dev(k), dev(v), dev(a), cu, scale, dev(s0), **kw)
    torch.cuda.synchronize()
    assert gla.gla_last_device_status() == 0
    o = o.float().cpu().numpy()
    hT = hT.cpu().numpy()
    for n in range(len(cu) - 1):
        b, e = cu[n], cu[n + 1]
        if e == b:
            want = np.zeros((H, dk, dv)) if s0 is None else s0[n].double().numpy()
            np.testing.assert_array_equal(hT[n], want.astype(np.float32))
            continue
        sl = lambda t: t[:, b:e].unsqueeze(0).float().numpy()  # noqa: E731
        o_ref, h_ref = og.forward(sl(q), sl(k), sl(v), sl(a), scale,
                                  None if s0 is None else s0[n:n + 1].double().numpy())
        assert_close(o[:, b:e][None], o_ref, f"{what} seq {n} (len {e - b}) o", bf16_output=True)
        assert_close(hT[n:n + 1], h_ref, f"{what} seq {n} (len {e - b}) hT")
    return o, hT


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (128, 256)])
def test_mixed_lengths(dk, dv):
    lens = [1, 127, 128, 129, 300, 65, 513]
    q, k, v, a, s0, cu = _packed_inputs(lens, 2, dk, dv, seed=dk + dv)
    _check(q, k, v, a, s0, cu, f"dk={dk} dv={dv}")


def test_empty_sequences_pass_the_state_through():
    lens = [0, 200, 0, 0, 130, 0]
    q, k, v, a, s0, cu = _packed_inputs(lens, 2, 64, 128, seed=3)
    _check(q, k, v, a, s0, cu, "empty sequences")


def test_no_initial_state():
    lens = [90, 260, 5]
    q, k, v, a, _, cu = _packed_inputs(lens, 3, 128, 128, h0=False, seed=4)
    _check(q, k, v, a, None, cu, "no h0")


def test_one_sequence_equals_the_fixed_length_call():
    lens = [777]
    q, k, v, a, s0, cu = _packed_inputs(lens, 2, 128, 256, seed=5)
    o_v, h_v = gla.gla_chunk_fwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), a.to(DEV), cu, None,
                                        s0.to(DEV))
    o_f, h_f = gla.gla_chunk_fwd(q[None].to(DEV), k[None].to(DEV), v[None].to(DEV),
                                 a[None].to(DEV), None, s0.to(DEV))
    torch.cuda.synchronize()
    assert gla.gla_last_device_status() == 0
    # the same chunks through the same kernel (one sequence, whole chunks)
    assert torch.equal(o_v, o_f[0])
    assert torch.equal(h_v, h_f)


@pytest.mark.parametrize("segments", [2, 3])
def test_long_sequences_cut_into_segments(segments):
    lens = [2100, 300, 1500, 129]
    q, k, v, a, s0, cu = _packed_inputs(lens, 2, 128, 128, seed=10 + segments)
    _check(q, k, v, a, s0, cu, f"segments={segments}", segments=segments)


def test_pair_path_with_segments_and_tails():
    lens = [1000, 77, 640, 3]
    q, k, v, a, s0, cu = _packed_inputs(lens, 2, 128, 256, seed=21)
    _check(q, k, v, a, s0, cu, "pair segments", segments=3)


@pytest.mark.parametrize("cta_pair", [0, -1])
def test_pair_and_independent_tiles(cta_pair):
    lens = [333, 64, 190]
    q, k, v, a, s0, cu = _packed_inputs(lens, 2, 128, 256, seed=22)
    _check(q, k, v, a, s0, cu, f"cta_pair={cta_pair}", cta_pair=cta_pair)


def test_sub_chunk_path_on_tails():
    lens = [150, 40, 260]
    q, k, v, a, s0, cu = _packed_inputs(lens, 2, 128, 128, seed=23, sigma_z=2.0)
    _check(q, k, v, a, s0, cu, "force_exact", force_exact=True)


def test_many_short_sequences():
    rng = np.random.default_rng(7)
    lens = rng.integers(1, 260, size=60).tolist()
    q, k, v, a, s0, cu = _packed_inputs(lens, 2, 64, 64, seed=24)
    _check(q, k, v, a, s0, cu, "60 short sequences")


def test_final_state_may_alias_initial_state():
    lens = [300, 129]
    q, k, v, a, s0, cu = _packed_inputs(lens, 2, 128, 256, seed=25)
    h = s0.to(DEV).clone()
    o, hT = gla.gla_chunk_fwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), a.to(DEV), cu, None, h,
                                     final_state=h)
    torch.cuda.synchronize()
    assert hT.data_ptr() == h.data_ptr()
    for n in range(2):
        b, e = cu[n], cu[n + 1]
        sl = lambda t: t[:, b:e].unsqueeze(0).float().numpy()  # noqa: E731
        _, h_ref = og.forward(sl(q), sl(k), sl(v), sl(a), 128 ** -0.5,
                              s0[n:n + 1].double().numpy())
        assert_close(h[n:n + 1].cpu().numpy(), h_ref, f"aliased hT seq {n}")
