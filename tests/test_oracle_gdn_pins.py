"""Pins of the gated-delta-rule oracle (``oracle/gdn_oracle.c``), row F4's reference.

The oracle is the token loop S_t = alpha_t (I - beta_t k_t^T k_t) S_{t-1} +
beta_t k_t^T v_t, o_t = scale q_t S_t ("Qwen Team Releases FlashQLA ...",
"Core Technical Principles", in the standard gated-delta-rule reading).
Each check compares it with something else: two cases worked by hand
(tests/golden/gdn_hand_examples.json), the four-step chunk algorithm
of the same page (``pins.gdn_chunk_form``) at every chunk length, the
decay-only closed form (beta = 0), the delta rule's defining overwrite
(alpha = beta = 1, unit key: reading with the written key returns the
written value), the vanishing-gate limit (only the current write survives),
linearity in (v, h0), the contraction bound that unit keys and gates in
(0, 1] give, the page's sequence-parallel correction (segments from zero
state, corrected by products of per-chunk dk x dk transition matrices) and
its sliding-window bound.  ``test_gdn_mutants_are_rejected`` plants
mistakes in a copy of the oracle.
"""

from __future__ import annotations

import ctypes
import json
import os
import shutil

import numpy as np
import pytest

from oracle import gdn_oracle as gd
import pins

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "gdn_hand_examples.json")


def _case(seed, BH, T, dk, dv, *, g_spread=1.0, tau=4.0, h0=True):
    rng = np.random.default_rng(seed)
    z = rng.normal(0.0, g_spread, size=(BH, T))
    g = (-np.logaddexp(0.0, -z) / tau).astype(np.float32)            # log alpha in (-inf, 0)
    beta = (1.0 / (1.0 + np.exp(-rng.normal(size=(BH, T))))).astype(np.float32)
    q = rng.normal(size=(BH, T, dk)).astype(np.float32)
    k = rng.normal(size=(BH, T, dk))
    k = (k / np.linalg.norm(k, axis=-1, keepdims=True)).astype(np.float32)   # L2-normalised keys
    v = rng.normal(size=(BH, T, dv)).astype(np.float32)
    s0 = rng.normal(0.0, 0.5, size=(BH, dk, dv)) if h0 else None
    return q, k, v, g, beta, s0


class Orc:
    def __init__(self, lib=None):
        self.lib = lib

    def fwd(self, q, k, v, g, b, scale, h0=None):
        return gd.forward(q, k, v, g, b, scale, h0, lib=self.lib)


def _rel(x, ref):
    x, ref = np.asarray(x, np.float64), np.asarray(ref, np.float64)
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300))


def pin_hand_examples(orc: Orc):
    """Cases worked by hand (tests/golden/gdn_hand_examples.json, derivations included)."""
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        q = np.asarray(c["q"], np.float32)[None]
        k = np.asarray(c["k"], np.float32)[None]
        v = np.asarray(c["v"], np.float32)[None]
        g = np.log(np.asarray(c["alpha"], np.float64)).astype(np.float32)[None]
        b = np.asarray(c["beta"], np.float32)[None]
        h0 = None if c["h0"] is None else np.asarray(c["h0"], np.float64)[None]
        o, hT = orc.fwd(q, k, v, g, b, c["scale"], h0)
        np.testing.assert_allclose(o[0], np.asarray(c["o"]), rtol=1e-6, atol=1e-6,
                                   err_msg=c["name"] + " o")
        np.testing.assert_allclose(hT[0], np.asarray(c["hT"]), rtol=1e-6, atol=1e-6,
                                   err_msg=c["name"] + " hT")


def pin_chunk_form(orc: Orc):
    q, k, v, g, b, s0 = _case(1, 2, 37, 6, 5)
    o, hT = orc.fwd(q, k, v, g, b, 0.4, s0)
    for C in (1, 3, 8, 37, 64):
        for n in range(2):
            o_ref, s_ref = pins.gdn_chunk_form(q[n], k[n], v[n], g[n], b[n], 0.4, s0[n], C)
            assert _rel(o[n], o_ref) <= 1e-11, f"C={C} head {n} o"
            assert _rel(hT[n], s_ref) <= 1e-11, f"C={C} head {n} hT"


def pin_decay_only(orc: Orc):
    """beta = 0: nothing is written or erased; S_t = (prod alpha) h0."""
    q, k, v, g, b, s0 = _case(2, 2, 20, 4, 3)
    b = np.zeros_like(b)
    o, hT = orc.fwd(q, k, v, g, b, 0.7, s0)
    cum = np.exp(np.cumsum(g.astype(np.float64), axis=1))            # [BH, T]
    want = 0.7 * cum[:, :, None] * np.einsum("ntd,nde->nte", q.astype(np.float64), s0)
    assert _rel(o, want) <= 1e-12
    assert _rel(hT, cum[:, -1, None, None] * s0) <= 1e-12


def pin_overwrite(orc: Orc):
    """alpha = beta = 1 and a unit key: the write replaces what the key reads,
    so querying with that key returns exactly the value just written."""
    q, k, v, g, b, s0 = _case(3, 2, 15, 8, 4)
    g, b = np.zeros_like(g), np.ones_like(b)
    q = k.copy()
    o, _ = orc.fwd(q, k, v, g, b, 1.0, s0)
    # k is float32-normalised; its norm differs from 1 by float32 rounding only
    assert _rel(o, v.astype(np.float64)) <= 1e-6


def pin_linearity(orc: Orc):
    """o and hT are jointly linear in (v, h0) for fixed q, k, gates."""
    q, k, v, g, b, s0 = _case(4, 2, 25, 5, 4)
    v2 = np.random.default_rng(9).normal(size=v.shape).astype(np.float32)
    s2 = np.random.default_rng(10).normal(size=s0.shape)
    o1, h1 = orc.fwd(q, k, v, g, b, 0.3, s0)
    o2, h2 = orc.fwd(q, k, v2, g, b, 0.3, s2)
    o3, h3 = orc.fwd(q, k, (v.astype(np.float64) + v2).astype(np.float32), g, b, 0.3, s0 + s2)
    vsum = v.astype(np.float64) + v2
    exact = np.array_equal(vsum.astype(np.float32).astype(np.float64), vsum)
    tol = 1e-11 if exact else 1e-6
    assert _rel(o3, o1 + o2) <= tol and _rel(h3, h1 + h2) <= tol


def pin_contraction(orc: Orc):
    """Unit keys, beta in [0, 1], alpha <= 1: |S_t|_F <= |S_{t-1}|_F + beta_t |v_t|."""
    q, k, v, g, b, s0 = _case(5, 3, 60, 6, 5, g_spread=0.2, tau=50.0)
    _, hT = orc.fwd(q, k, v, g, b, 1.0, s0)
    bound = np.linalg.norm(s0, axis=(1, 2)) + np.sum(
        b * np.linalg.norm(v.astype(np.float64), axis=-1), axis=1)
    assert np.all(np.linalg.norm(hT, axis=(1, 2)) <= bound * (1 + 1e-9))


def pin_vanishing_gate(orc: Orc):
    """alpha = e^-30: everything before the current token is gone, so
    S_t = beta_t k_t^T v_t + O(e^-30) and o_t = scale beta_t (q_t . k_t) v_t."""
    q, k, v, g, b, s0 = _case(7, 2, 12, 5, 4)
    g = np.full_like(g, -30.0)
    o, hT = orc.fwd(q, k, v, g, b, 0.6, s0)
    q64, k64, v64 = (x.astype(np.float64) for x in (q, k, v))
    want = 0.6 * (b * np.sum(q64 * k64, axis=-1))[:, :, None] * v64
    assert np.max(np.abs(o - want)) <= 1e-9 * max(1.0, float(np.max(np.abs(want))))
    want_h = b[:, -1, None, None] * np.einsum("nd,ne->nde", k64[:, -1], v64[:, -1])
    assert np.max(np.abs(hT - want_h)) <= 1e-9


def pin_segment_correction(orc: Orc):
    """Segments started from zero and corrected by the products of their chunks'
    dk x dk transition matrices (the page's sequence-parallel scheme) give the
    loop's outputs and final state, for segment and chunk lengths on and off
    the sequence length."""
    q, k, v, g, b, s0 = _case(11, 2, 45, 6, 5)
    o, hT = orc.fwd(q, k, v, g, b, 0.5, s0)
    for C, seg in ((1, 7), (4, 1), (4, 3), (8, 2), (16, 1), (64, 1)):
        for n in range(2):
            o_ref, s_ref = pins.gdn_segment_form(q[n], k[n], v[n], g[n], b[n], 0.5, s0[n], C, seg)
            assert _rel(o[n], o_ref) <= 1e-10, f"C={C} seg={seg} head {n} o"
            assert _rel(hT[n], s_ref) <= 1e-10, f"C={C} seg={seg} head {n} hT"


def pin_sliding_window(orc: Orc):
    """Each step maps a state difference D to alpha_t (I - beta_t k_t^T k_t) D,
    whose norm is at most alpha_t |D| for unit keys and beta in [0, 1]: a state
    rebuilt from zero over the last w tokens differs from the true one by at
    most (product of alpha over the window) x |true state before the window|
    (the sliding-window property of the same page)."""
    q, k, v, g, b, s0 = _case(12, 3, 90, 6, 5, g_spread=1.0, tau=3.0)
    p = 80
    for w in (1, 5, 20, 40):
        _, s_true = orc.fwd(q[:, :p], k[:, :p], v[:, :p], g[:, :p], b[:, :p], 1.0, s0)
        _, s_before = orc.fwd(q[:, :p - w], k[:, :p - w], v[:, :p - w], g[:, :p - w],
                              b[:, :p - w], 1.0, s0)
        _, s_win = orc.fwd(q[:, p - w:p], k[:, p - w:p], v[:, p - w:p], g[:, p - w:p],
                           b[:, p - w:p], 1.0, None)
        decay = np.exp(np.sum(g[:, p - w:p].astype(np.float64), axis=1))
        err = np.linalg.norm(s_true - s_win, axis=(1, 2))
        bound = decay * np.linalg.norm(s_before, axis=(1, 2))
        assert np.all(err <= bound * (1 + 1e-9) + 1e-12), (w, err, bound)
        assert np.all(err >= 0.01 * bound) or w > 20   # the bound is not vacuous at short windows


GDN_PINS = [pin_hand_examples, pin_chunk_form, pin_decay_only, pin_overwrite, pin_linearity, pin_contraction,
            pin_vanishing_gate, pin_segment_correction, pin_sliding_window]


@pytest.mark.parametrize("pin", GDN_PINS, ids=[p.__name__ for p in GDN_PINS])
def test_gdn_pin(pin):
    pin(Orc())


def test_threads_and_batching_do_not_change_results():
    q, k, v, g, b, s0 = _case(6, 5, 30, 4, 3)
    o1, h1 = gd.forward(q, k, v, g, b, 0.5, s0, nthreads=1)
    o4, h4 = gd.forward(q, k, v, g, b, 0.5, s0, nthreads=4)
    assert np.array_equal(o1, o4) and np.array_equal(h1, h4)
    for n in range(5):
        on, hn = gd.forward(q[n], k[n], v[n], g[n], b[n], 0.5, s0[n])
        assert np.array_equal(on, o1[n]) and np.array_equal(hn, h1[n])


GDN_MUTANTS = {
    "gate_on_write_too": ("row[c] = alpha * (row[c] - beta * kd * kS[c]) + beta * kd * (double)v[c];",
                          "row[c] = alpha * (row[c] - beta * kd * kS[c] + beta * kd * (double)v[c]);"),
    "erase_not_gated": ("row[c] = alpha * (row[c] - beta * kd * kS[c]) + beta * kd * (double)v[c];",
                        "row[c] = alpha * row[c] - beta * kd * kS[c] + beta * kd * (double)v[c];"),
    "erase_sign": ("row[c] = alpha * (row[c] - beta * kd * kS[c]) + beta * kd * (double)v[c];",
                   "row[c] = alpha * (row[c] + beta * kd * kS[c]) + beta * kd * (double)v[c];"),
    "write_without_beta": ("row[c] = alpha * (row[c] - beta * kd * kS[c]) + beta * kd * (double)v[c];",
                           "row[c] = alpha * (row[c] - beta * kd * kS[c]) + kd * (double)v[c];"),
    "erase_reads_with_q": ("for (int d = 0; d < dk; ++d) acc += (double)k[d] * S[(int64_t)d * dv + c];\n        kS[c] = acc;",
                           "for (int d = 0; d < dk; ++d) acc += (double)q[d] * S[(int64_t)d * dv + c];\n        kS[c] = acc;"),
    "gate_sign": ("const double alpha = exp(g);", "const double alpha = exp(-g);"),
    "scale_dropped": ("o[c] = scale * acc;", "o[c] = acc;"),
    "h0_ignored": ("if (h0) memcpy", "if (0) memcpy"),
}


@pytest.mark.parametrize("name", sorted(GDN_MUTANTS))
def test_gdn_mutants_are_rejected(name, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(gd._SRC).read()
    old, new = GDN_MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path = tmp_path / f"gdn_{name}.c"
    path.write_text(src.replace(old, new))
    lib = gd._bind(ctypes.CDLL(gd.build(str(path), str(tmp_path / f"gdn_{name}.so"))))
    caught = []
    for pin in GDN_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(Orc(lib))
        except (AssertionError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
