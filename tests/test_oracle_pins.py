"""Pins of the fp64 CPU oracle against what the pages and the mathematics fix.

Every check below compares the oracle (the token-by-token recurrence in C) with
something that is not the oracle: a hand-worked example, the dual attention
form by brute force, textbook special cases, the chunkwise equations, closed
forms, limits and invariants.  ``test_mutants_are_rejected`` then plants
plausible mistakes in a copy of the oracle's source and requires that at least
one of these pins rejects each of them.
"""

from __future__ import annotations

import json
import os
import re
import shutil

import numpy as np
import pytest

import oracle
from oracle import gla_oracle as og
import pins

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "hand_examples.json")
RTOL = 1e-11  # fp64 against fp64 in a different summation order


def _rng(seed):
    return np.random.default_rng(seed)


def _seq(rng, T, dk, dv, *, gate_spread=2.0, tau=2.0, h0=False):
    """Small random sequence with strongly varying gates (alpha in (0, 1))."""
    z = rng.normal(0.0, gate_spread, size=(T, dk))
    a = (-np.logaddexp(0.0, -z) / tau).astype(np.float32)       # log sigmoid(z) / tau
    q = rng.normal(size=(T, dk)).astype(np.float32)
    k = rng.normal(size=(T, dk)).astype(np.float32)
    v = rng.normal(size=(T, dv)).astype(np.float32)
    s0 = rng.normal(0.0, 0.5, size=(dk, dv)) if h0 else None
    return q, k, v, a, s0


class Oracle:
    """The oracle bound to one compiled library (the real one, or a mutant)."""

    def __init__(self, lib=None):
        self.lib = lib

    def fwd(self, q, k, v, a, scale, h0=None):
        return og.forward(q, k, v, a, scale, h0, lib=self.lib)

    def step(self, q, k, v, a, scale, h):
        return og.step(q, k, v, a, scale, h, lib=self.lib)


def _close(x, ref, rtol=RTOL, what=""):
    err = pins.rel_err(x, ref)
    assert err <= rtol, f"{what}: relative error {err:.3e} > {rtol:.1e}"


# --------------------------------------------------------------------------- pins

def pin_hand_examples(orc: Oracle):
    cases = json.load(open(GOLDEN))["cases"]
    for c in cases:
        a = np.log(np.asarray(c["alpha"], dtype=np.float64)).astype(np.float32)
        h0 = None if c["h0"] is None else np.asarray(c["h0"], dtype=np.float64)
        o, hT = orc.fwd(np.float32(c["q"]), np.float32(c["k"]), np.float32(c["v"]), a,
                        c["scale"], h0)
        np.testing.assert_allclose(o, c["o"], rtol=1e-6, atol=1e-6, err_msg=c["name"])
        np.testing.assert_allclose(hT, c["hT"], rtol=1e-6, atol=1e-6, err_msg=c["name"])


def pin_dual_form(orc: Oracle):
    rng = _rng(1)
    for T, dk, dv, h0 in [(19, 5, 3, False), (23, 4, 6, True), (1, 3, 2, True), (40, 8, 8, False)]:
        q, k, v, a, s0 = _seq(rng, T, dk, dv, h0=h0)
        o, _ = orc.fwd(q, k, v, a, 0.37, s0)
        _close(o, pins.dual_form(q, k, v, a, 0.37, s0), what=f"dual form T={T} h0={h0}")


def pin_linear_attention(orc: Oracle):
    rng = _rng(2)
    for h0 in (False, True):
        q, k, v, _, s0 = _seq(rng, 31, 6, 5, h0=h0)
        a = np.zeros_like(q)  # alpha = 1
        o, hT = orc.fwd(q, k, v, a, 0.5, s0)
        o_ref, s_ref = pins.causal_linear_attention(q, k, v, 0.5, s0)
        _close(o, o_ref, what="alpha=1 output")
        _close(hT, s_ref, what="alpha=1 state")


def pin_retention(orc: Oracle):
    rng = _rng(3)
    gamma = np.float32(0.9)
    for h0 in (False, True):
        q, k, v, _, s0 = _seq(rng, 37, 4, 7, h0=h0)
        a = np.full_like(q, np.log(gamma))
        g = float(np.exp(np.float64(np.log(gamma))))  # the exact alpha the oracle sees
        o, hT = orc.fwd(q, k, v, a, 1.0, s0)
        o_ref, s_ref = pins.retention(q, k, v, g, 1.0, s0)
        _close(o, o_ref, what="retention output")
        _close(hT, s_ref, what="retention state")


def pin_chunk_form(orc: Oracle):
    rng = _rng(4)
    q, k, v, a, s0 = _seq(rng, 45, 6, 5, h0=True)
    o, hT = orc.fwd(q, k, v, a, 0.25, s0)
    for C in (1, 2, 3, 5, 8, 16, 45, 64):
        o_c, s_c = pins.chunk_form(q, k, v, a, 0.25, s0, C=C)
        _close(o, o_c, what=f"chunk form C={C} output")
        _close(hT, s_c, what=f"chunk form C={C} state")


def pin_state_passing(orc: Oracle):
    rng = _rng(5)
    q, k, v, a, s0 = _seq(rng, 50, 5, 4, h0=True)
    o, hT = orc.fwd(q, k, v, a, 0.5, s0)
    for T1 in (1, 7, 16, 33, 49):
        o1, h1 = orc.fwd(q[:T1], k[:T1], v[:T1], a[:T1], 0.5, s0)
        o2, h2 = orc.fwd(q[T1:], k[T1:], v[T1:], a[T1:], 0.5, h1)
        _close(np.concatenate([o1, o2]), o, what=f"split at {T1} output")
        _close(h2, hT, what=f"split at {T1} state")


def pin_single_token(orc: Oracle):
    rng = _rng(6)
    q, k, v, a, s0 = _seq(rng, 1, 7, 3, h0=True)
    o, hT = orc.fwd(q, k, v, a, 0.3, s0)
    s1 = (np.exp(a[0].astype(np.float64))[:, None] * s0
          + np.outer(k[0].astype(np.float64), v[0].astype(np.float64)))
    _close(hT, s1, what="T=1 state")
    _close(o[0], 0.3 * (q[0].astype(np.float64) @ s1), what="T=1 output")


def pin_vanishing_gate(orc: Oracle):
    # log alpha = -30: alpha ~ 9.4e-14, so every token forgets the past.
    rng = _rng(7)
    q, k, v, _, s0 = _seq(rng, 12, 4, 3, h0=True)
    a = np.full_like(q, -30.0)
    o, hT = orc.fwd(q, k, v, a, 0.5, s0)
    qd, kd, vd = (x.astype(np.float64) for x in (q, k, v))
    o_lim = 0.5 * (qd * kd).sum(1)[:, None] * vd
    np.testing.assert_allclose(o, o_lim, rtol=0, atol=1e-10)
    np.testing.assert_allclose(hT, np.outer(kd[-1], vd[-1]), rtol=0, atol=1e-10)


def pin_linearity(orc: Oracle):
    rng = _rng(8)
    q, k, v1, a, h1 = _seq(rng, 20, 5, 4, h0=True)
    v2 = rng.normal(size=v1.shape).astype(np.float32)
    h2 = rng.normal(size=h1.shape)
    oa, sa = orc.fwd(q, k, v1, a, 0.5, h1)
    ob, sb = orc.fwd(q, k, v2, a, 0.5, h2)
    oc, sc = orc.fwd(q, k, (v1 + 2 * v2).astype(np.float64), a, 0.5, h1 + 2 * h2)
    # v1 + 2 v2 is rounded to float32 inside the oracle wrapper: compare loosely.
    _close(oc, oa + 2 * ob, rtol=1e-6, what="linearity output")
    _close(sc, sa + 2 * sb, rtol=1e-6, what="linearity state")
    # v = 0: only the decayed initial state is read out, o_t = (q_t * exp(sum_{m<=t} A_m)) h0.
    o0, _ = orc.fwd(q, k, np.zeros_like(v1), a, 0.5, h1)
    decay = np.exp(np.cumsum(a.astype(np.float64), axis=0))
    _close(o0, 0.5 * (q * decay) @ h1, what="v=0 output")


def pin_contraction(orc: Oracle):
    # alpha in (0,1) makes diag(alpha) a contraction ("Context Length
    # Extrapolation"): ||S_T||_F <= ||h0||_F + sum_j ||k_j|| ||v_j||.
    rng = _rng(9)
    q, k, v, a, s0 = _seq(rng, 300, 6, 6, h0=True, gate_spread=0.5, tau=40.0)
    _, hT = orc.fwd(q, k, v, a, 1.0, s0)
    bound = np.linalg.norm(s0) + sum(np.linalg.norm(k[j].astype(np.float64)) *
                                     np.linalg.norm(v[j].astype(np.float64)) for j in range(300))
    assert np.linalg.norm(hT) <= bound * (1 + 1e-12)
    # and it is not vacuous: with slow decay the state norm is a sizeable part of the bound.
    assert np.linalg.norm(hT) > 0.02 * bound


def pin_step_matches_forward(orc: Oracle):
    rng = _rng(10)
    q, k, v, a, s0 = _seq(rng, 9, 5, 6, h0=True)
    o, hT = pins.chunk_form(q, k, v, a, 0.7, s0, C=4)
    h = s0.copy()
    for t in range(9):
        ot = orc.step(q[t], k[t], v[t], a[t], 0.7, h)
        _close(ot, o[t], what=f"decode step {t}")
    _close(h, hT, what="decode final state")


PINS = [pin_hand_examples, pin_dual_form, pin_linear_attention, pin_retention, pin_chunk_form,
        pin_state_passing, pin_single_token, pin_vanishing_gate, pin_linearity, pin_contraction,
        pin_step_matches_forward]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(Oracle())


def test_batched_heads_are_independent():
    rng = _rng(11)
    B, H, T, dk, dv = 2, 3, 17, 4, 5
    seqs = [_seq(rng, T, dk, dv, h0=True) for _ in range(B * H)]
    stack = [np.stack([s[i] for s in seqs]).reshape(B, H, *seqs[0][i].shape) for i in range(5)]
    o, hT = og.forward(*stack[:4], 0.5, stack[4])
    for n, (q, k, v, a, s0) in enumerate(seqs):
        b, h = divmod(n, H)
        o_ref, s_ref = pins.chunk_form(q, k, v, a, 0.5, s0, C=5)
        _close(o[b, h], o_ref, what=f"head {n} output")
        _close(hT[b, h], s_ref, what=f"head {n} state")


def test_thread_count_does_not_change_results():
    rng = _rng(12)
    seqs = [_seq(rng, 33, 6, 4, h0=True) for _ in range(8)]
    stack = [np.stack([s[i] for s in seqs]) for i in range(5)]
    o1, h1 = og.forward(*stack[:4], 0.5, stack[4], nthreads=1)
    o4, h4 = og.forward(*stack[:4], 0.5, stack[4], nthreads=4)
    assert np.array_equal(o1, o4) and np.array_equal(h1, h4)


# --------------------------------------------------------------------------- mutants

_TOKEN_UPDATE = "row[c] = alpha * row[c] + kd * (double)v[c];"
MUTANTS = {
    "gate_sign": ("exp((double)a[d])", "exp(-(double)a[d])"),
    "gate_dropped": (_TOKEN_UPDATE, "row[c] = row[c] + kd * (double)v[c];"),
    "gate_wrong_channel": ("exp((double)a[d])", "exp((double)a[0])"),
    "gate_after_write": (_TOKEN_UPDATE, "row[c] = alpha * (row[c] + kd * (double)v[c]);"),
    "value_index": (_TOKEN_UPDATE, "row[c] = alpha * row[c] + kd * (double)v[0];"),
    "readout_transposed": ("S[(int64_t)d * dv + c]", "S[(int64_t)c * dk + d]"),
    "readout_uses_k": ("acc += (double)q[d] *", "acc += (double)k[d] *"),
    "scale_dropped": ("o[c] = scale * acc;", "o[c] = acc;"),
    "h0_ignored": ("if (h0) memcpy", "if (0) memcpy"),
    "previous_token_gate": ("log_alpha + rk, scale", "log_alpha + (t > 0 ? rk - dk : rk), scale"),
    "readout_before_update": None,  # block swap, see below
}


def _mutate(src: str, name: str) -> str:
    if name == "readout_before_update":
        m = re.search(r"(    for \(int d = 0; d < dk; \+\+d\) \{.*?\n    \}\n)"
                      r"(    for \(int c = 0; c < dv; \+\+c\) \{.*?\n    \}\n)", src, re.S)
        assert m, "token-function blocks not found"
        return src[: m.start()] + m.group(2) + m.group(1) + src[m.end():]
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    return src.replace(old, new)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutants_are_rejected(name, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(og._SRC).read()
    mutant = _mutate(src, name)
    assert mutant != src
    path = tmp_path / f"mut_{name}.c"
    path.write_text(mutant)
    lib = og._bind(__import__("ctypes").CDLL(og.build(str(path), str(tmp_path / f"mut_{name}.so"))))
    orc = Oracle(lib)
    caught = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(orc)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
