"""Pins of the oracle's backward pass against what the mathematics fixes.

The backward (``oracle.backward``) is reverse-mode differentiation of the
token loop.  Nothing below re-derives it; each check compares it with
something else:

* central differences of the forward oracle (itself pinned by
  ``test_oracle_pins.py``), along random directions for every input, and
  entry by entry on a tiny case;
* autograd (torch, float64) through the unrolled dual attention form of
  "Gated Linear Attention (GLA) ...", section "The Gated Recurrent Update",
  a different algorithm that reaches the same gradients;
* the log-gate identity: shifting log alpha_t by e shifts the cumulative
  log-gates of every token from t on, so
  dL/dlog_alpha_t = sum_{tau >= t} (q_tau * dq_tau - k_tau * dk_tau)
                    + rowsum(dhT * hT);
* the chunk-form gradient equations (``pins.chunk_form_backward``, the form
  the backward kernels evaluate) at every chunk length from 1 to T;
* independence from the checkpoint spacing and the thread count.

``test_backward_mutants_are_rejected`` plants plausible mistakes in a copy of
the backward's source and requires that a pin rejects each.
"""

from __future__ import annotations

import ctypes
import shutil

import numpy as np
import pytest

from oracle import gla_oracle as og

torch = pytest.importorskip("torch")


def _case(seed, BH, T, dk, dv, *, spread=2.0, tau=4.0, states=True):
    rng = np.random.default_rng(seed)
    z = rng.normal(0.0, spread, size=(BH, T, dk))
    a = (-np.logaddexp(0.0, -z) / tau).astype(np.float32)
    f = lambda *s: rng.normal(size=s).astype(np.float32)  # noqa: E731
    q, k, v, do = f(BH, T, dk), f(BH, T, dk), f(BH, T, dv), f(BH, T, dv)
    h0 = rng.normal(0.0, 0.5, size=(BH, dk, dv)) if states else None
    dhT = rng.normal(0.0, 0.5, size=(BH, dk, dv)) if states else None
    return q, k, v, a, do, h0, dhT


class Orc:
    def __init__(self, lib=None):
        self.lib = lib

    def fwd(self, q, k, v, a, scale, h0):
        return og.forward(q, k, v, a, scale, h0, lib=self.lib)

    def bwd(self, q, k, v, a, scale, do, h0, dhT, ck=0):
        return og.backward(q, k, v, a, scale, do, h0, dhT, ck=ck, lib=self.lib)


def _loss(orc, q, k, v, a, scale, do, h0, dhT):
    o, hT = orc.fwd(q, k, v, a, scale, h0)
    L = float(np.sum(o * do, dtype=np.float64))
    if dhT is not None:
        L += float(np.sum(hT * dhT, dtype=np.float64))
    return L


def _rel(x, ref):
    x, ref = np.asarray(x, np.float64), np.asarray(ref, np.float64)
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300))


NAMES = ("q", "k", "v", "log_alpha", "h0")


def pin_directional_differences(orc: Orc):
    """<grad, d> against (L(x + e d) - L(x - e d)) / 2e for every input."""
    q, k, v, a, do, h0, dhT = _case(1, 2, 37, 6, 5)
    scale = 0.4
    grads = orc.bwd(q, k, v, a, scale, do, h0, dhT, ck=5)
    rng = np.random.default_rng(2)
    base = [q, k, v, a, h0]
    for i, name in enumerate(NAMES):
        x = base[i]
        d = rng.normal(size=x.shape)
        eps = 1e-3 * float(np.sqrt(np.mean(np.square(x, dtype=np.float64))))
        if name == "h0":
            xp, xm = x + eps * d, x - eps * d
        else:  # the forward takes float32: use the exactly representable steps
            xp = (x + eps * d).astype(np.float32)
            xm = (x - eps * d).astype(np.float32)
        args_p, args_m = list(base), list(base)
        args_p[i], args_m[i] = xp, xm
        lp = _loss(orc, *args_p[:4], scale, do, args_p[4], dhT)
        lm = _loss(orc, *args_m[:4], scale, do, args_m[4], dhT)
        want = lp - lm
        got = float(np.sum(grads[i] * (np.asarray(xp, np.float64) - np.asarray(xm, np.float64))))
        assert abs(got - want) <= 1e-6 * max(abs(want), 1e-3), f"{name}: {got} vs {want}"


def pin_entrywise_differences(orc: Orc):
    """Every entry of every gradient of a tiny case, by central differences."""
    q, k, v, a, do, h0, dhT = _case(3, 1, 4, 2, 3)
    scale = 0.7
    grads = orc.bwd(q, k, v, a, scale, do, h0, dhT)
    base = [q, k, v, a, h0]
    for i, name in enumerate(NAMES):
        x = base[i]
        num = np.zeros(x.shape)
        for idx in np.ndindex(*x.shape):
            xp, xm = np.array(x, copy=True), np.array(x, copy=True)
            step = 1e-3 * max(abs(float(x[idx])), 0.1)
            xp[idx] += step
            xm[idx] -= step
            dx = float(xp[idx]) - float(xm[idx])
            args_p, args_m = list(base), list(base)
            args_p[i], args_m[i] = xp, xm
            num[idx] = (_loss(orc, *args_p[:4], scale, do, args_p[4], dhT)
                        - _loss(orc, *args_m[:4], scale, do, args_m[4], dhT)) / dx
        err = float(np.max(np.abs(grads[i] - num)))
        assert err <= 1e-6 * max(float(np.max(np.abs(num))), 1.0), f"{name}: max err {err:.3e}"


def _dual_form_grads(q, k, v, a, scale, do, h0, dhT):
    """Autograd of the dual form O = scale ((Q e^b)(K e^-b)^T * tril) V + scale (Q e^b) h0,
    hT = diag(e^{b_T}) (h0 + (K e^-b)^T V), b = cumulative log-gates."""
    t = lambda x: torch.tensor(np.asarray(x, np.float64), requires_grad=True)  # noqa: E731
    Q, K, V, A, H0 = t(q), t(k), t(v), t(a), t(h0)
    b = torch.cumsum(A, dim=0)
    Qt, Kt = Q * torch.exp(b), K * torch.exp(-b)
    P = torch.tril(Qt @ Kt.T)
    O = scale * (P @ V + Qt @ H0)
    hT = torch.exp(b[-1])[:, None] * (H0 + Kt.T @ V)
    L = (O * torch.tensor(np.asarray(do, np.float64))).sum() + \
        (hT * torch.tensor(np.asarray(dhT, np.float64))).sum()
    g = torch.autograd.grad(L, (Q, K, V, A, H0))
    return [x.numpy() for x in g]


def pin_dual_form_autograd(orc: Orc):
    for seed, T, dk, dv in ((4, 1, 3, 2), (5, 23, 5, 4), (6, 40, 4, 7)):
        q, k, v, a, do, h0, dhT = _case(seed, 3, T, dk, dv, spread=1.0, tau=8.0)
        scale = 0.3
        grads = orc.bwd(q, k, v, a, scale, do, h0, dhT)
        for n in range(3):
            want = _dual_form_grads(q[n], k[n], v[n], a[n], scale, do[n], h0[n], dhT[n])
            for i, name in enumerate(NAMES):
                err = _rel(grads[i][n], want[i])
                assert err <= 1e-10, f"T={T} head {n} {name}: rel err {err:.2e}"


def pin_log_gate_identity(orc: Orc):
    q, k, v, a, do, h0, dhT = _case(7, 2, 50, 6, 5, spread=3.0, tau=2.0)
    scale = 0.5
    dq, dk, _, da, _ = orc.bwd(q, k, v, a, scale, do, h0, dhT)
    _, hT = orc.fwd(q, k, v, a, scale, h0)
    term = q * dq - k * dk                                    # [BH, T, dk]
    tail = np.flip(np.cumsum(np.flip(term, axis=1), axis=1), axis=1)
    want = tail + np.sum(dhT * hT, axis=2)[:, None, :]
    err = _rel(da, want)
    assert err <= 1e-10, f"log-gate identity: rel err {err:.2e}"


def pin_no_states(orc: Orc):
    """Absent h0 / dhT are zero: same gradients as explicit zeros."""
    q, k, v, a, do, _, _ = _case(8, 2, 19, 4, 3, states=False)
    z = np.zeros((2, 4, 3))
    g_none = orc.bwd(q, k, v, a, 0.6, do, None, None)
    g_zero = orc.bwd(q, k, v, a, 0.6, do, z, z)
    for i, name in enumerate(NAMES):
        assert np.array_equal(g_none[i], g_zero[i]), name
    # and with zero states, the gradients match the dual form
    want = _dual_form_grads(q[0], k[0], v[0], a[0], 0.6, do[0], z[0], z[0])
    for i, name in enumerate(NAMES):
        assert _rel(g_none[i][0], want[i]) <= 1e-10, name


def pin_chunk_form(orc: Orc):
    """The chunk-form gradient equations (every chunk length, incl. 1 and T) equal the
    reverse-mode gradients."""
    import pins
    q, k, v, a, do, h0, dhT = _case(10, 2, 29, 5, 4, spread=2.0, tau=3.0)
    scale = 0.45
    grads = orc.bwd(q, k, v, a, scale, do, h0, dhT)
    for C in (1, 4, 7, 29, 64):
        for n in range(2):
            want = pins.chunk_form_backward(q[n], k[n], v[n], a[n], scale, do[n], h0[n], dhT[n], C)
            for i, name in enumerate(NAMES):
                err = _rel(grads[i][n], want[i])
                assert err <= 1e-10, f"C={C} head {n} {name}: rel err {err:.2e}"


BWD_PINS = [pin_directional_differences, pin_entrywise_differences, pin_dual_form_autograd,
            pin_log_gate_identity, pin_no_states, pin_chunk_form]


@pytest.mark.parametrize("pin", BWD_PINS, ids=[p.__name__ for p in BWD_PINS])
def test_backward_pin(pin):
    pin(Orc())


def test_checkpoint_spacing_and_threads_do_not_change_results():
    q, k, v, a, do, h0, dhT = _case(9, 6, 45, 5, 4)
    ref = og.backward(q, k, v, a, 0.5, do, h0, dhT, nthreads=1)
    for ck, nt in ((1, 4), (7, 2), (45, 3), (100, 1)):
        got = og.backward(q, k, v, a, 0.5, do, h0, dhT, ck=ck, nthreads=nt)
        for x, y in zip(got, ref):
            assert np.array_equal(x, y), (ck, nt)


def test_empty_sequence():
    q = np.zeros((2, 0, 4), np.float32)
    v = np.zeros((2, 0, 3), np.float32)
    dhT = np.random.default_rng(0).normal(size=(2, 4, 3))
    dq, dk, dv, da, dh0 = og.backward(q, q, v, q, 0.5, v, None, dhT)
    assert dq.shape == (2, 0, 4) and dv.shape == (2, 0, 3)
    np.testing.assert_array_equal(dh0, dhT)


# --------------------------------------------------------------------------- mutants

BWD_MUTANTS = {
    "adjoint_scale_dropped": ("const double sq = scale * (double)qt[d];",
                              "const double sq = (double)qt[d];"),
    "adjoint_not_decayed": ("for (int c = 0; c < dv; ++c) row[c] *= alpha;",
                            "for (int c = 0; c < dv; ++c) row[c] *= 1.0;"),
    "dq_reads_previous_state": ("aq += srow[c] * (double)dot[c];",
                                "aq += prow[c] * (double)dot[c];"),
    "dq_scale_dropped": ("gq[d] = scale * aq;", "gq[d] = aq;"),
    "dk_uses_output_grad": ("ak += grow[c] * (double)vt[c];", "ak += grow[c] * (double)dot[c];"),
    "dv_uses_query": ("acc += (double)kt[d] * G[(int64_t)d * dv + c];",
                      "acc += (double)qt[d] * G[(int64_t)d * dv + c];"),
    "dv_transposed": ("acc += (double)kt[d] * G[(int64_t)d * dv + c];",
                      "acc += (double)kt[d] * G[(int64_t)c * dk + d];"),
    "gate_grad_missing_alpha": ("ga[d] = exp((double)at[d]) * aa;", "ga[d] = aa;"),
    "gate_grad_uses_new_state": ("aa += grow[c] * prow[c];", "aa += grow[c] * srow[c];"),
    "final_adjoint_ignored": ("if (dhT) memcpy(G,", "if (0) memcpy(G,"),
    "replay_skips_first_token": ("for (int64_t t = t0; t < t1; ++t) {\n                double *nxt",
                                 "for (int64_t t = t0; t < t1; ++t) {\n                if (t == t0 && t > 0) continue;\n                double *nxt"),
}


@pytest.mark.parametrize("name", sorted(BWD_MUTANTS))
def test_backward_mutants_are_rejected(name, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(og._SRC).read()
    old, new = BWD_MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path = tmp_path / f"bwd_{name}.c"
    path.write_text(src.replace(old, new))
    lib = og._bind(ctypes.CDLL(og.build(str(path), str(tmp_path / f"bwd_{name}.so"))))
    orc = Orc(lib)
    caught = []
    for pin in BWD_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(orc)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every backward pin"
