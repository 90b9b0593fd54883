"""The chunked gated-delta-rule kernels' rearrangement of the page's chunk
algorithm, checked in fp64 against the oracle (no GPU).

"Qwen Team Releases FlashQLA for High-Performance Linear Attention", "Core
Technical Principles", gives four steps per chunk (``pins.gdn_chunk_form``
restates them).  The two CUDA kernels compute the same quantities in a
rearranged form so that the raw bf16 tiles of K and V are the products'
operands:

* the pre-pass stores W = (T diag(beta gamma)) K and (T - I) diag(beta);
* the sequential kernel forms U = beta_t v_t + ((T - I) diag(beta) V)_t, with
  the diagonal term exact, and D = U - W S;
* the state update takes the decay to the chunk's end on D instead of K:
  S_C = gamma_C S + K^T D', D' = diag(gamma_C / gamma) D;
* the output is O = scale (diag(gamma) Q S + tril(Q K^T gamma_t / gamma_i) D).

The rearrangement below is that algebra written out in plain NumPy, in the
kernels' order and in fp64, with no rounding of operands: it must equal the
token-loop oracle to rounding.  A slip in it (the diagonal term dropped or
counted twice, the decay on the wrong side, the wrong power of gamma) fails
here without a GPU.
"""

from __future__ import annotations

import numpy as np
import pytest

from oracle import gdn_oracle as gd


def kernel_algebra(q, k, v, g, beta, scale, h0, C=64, *, mutant=None):
    """One sequence: q, k [T, dk], v [T, dv], g, beta [T], h0 [dk, dv] or None.
    ``mutant`` plants one slip (for the detection tests)."""
    q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
    g, beta = np.asarray(g, np.float64), np.asarray(beta, np.float64)
    T, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if h0 is None else np.asarray(h0, np.float64).copy()
    o = np.zeros((T, dv))
    for t0 in range(0, T, C):
        qc, kc, vc = q[t0:t0 + C], k[t0:t0 + C], v[t0:t0 + C]
        n = kc.shape[0]
        G = np.cumsum(g[t0:t0 + C])                 # in-chunk inclusive prefix sums (log)
        gam = np.exp(G)
        b = beta[t0:t0 + C]
        # pre-pass: L, T, then what it stores
        L = np.tril(b[:, None] * np.exp(G[:, None] - G[None, :]) * (kc @ kc.T), -1)
        Tm = np.linalg.inv(np.eye(n) + L)
        W = (Tm * (b * gam)[None, :]) @ kc          # (T diag(beta gamma)) K
        Toff = (Tm - np.eye(n)) * b[None, :]        # (T - I) diag(beta)
        # sequential kernel
        U = b[:, None] * vc + Toff @ vc             # exact diagonal term plus the rest
        if mutant == "no_diagonal":
            U = Toff @ vc
        D = U - W @ S
        Dp = (np.exp(G[-1] - G))[:, None] * D       # decay to the chunk's end on D
        if mutant == "decay_from_start":
            Dp = gam[:, None] * D
        P = np.tril((qc @ kc.T) * np.exp(G[:, None] - G[None, :]))
        o[t0:t0 + n] = scale * (gam[:, None] * (qc @ S) + P @ D)
        S = np.exp(G[-1]) * S + kc.T @ Dp
    return o, S


def _case(seed, T, dk, dv, tau=4.0):
    rng = np.random.default_rng(seed)
    z = rng.normal(size=T)
    g = -np.logaddexp(0.0, -z) / tau                            # log alpha in (-inf, 0)
    beta = 1.0 / (1.0 + np.exp(-rng.normal(size=T)))
    q = rng.normal(size=(T, dk))
    k = rng.normal(size=(T, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)              # unit keys
    v = rng.normal(size=(T, dv))
    h0 = rng.normal(0.0, 0.5, size=(dk, dv))
    return q, k, v, g, beta, h0


@pytest.fixture(scope="module", autouse=True)
def _built():
    gd.build()


@pytest.mark.parametrize("T,C", [(1, 64), (37, 64), (64, 64), (150, 64), (150, 16), (257, 32)])
def test_kernel_algebra_equals_the_oracle(T, C):
    q, k, v, g, beta, h0 = _case(T + C, T, 16, 8)
    ro, rS = gd.forward(q[None].astype(np.float32), k[None].astype(np.float32),
                        v[None].astype(np.float32), g[None].astype(np.float32),
                        beta[None].astype(np.float32), 0.3, h0[None])
    # the oracle reads fp32 copies of the inputs: compare on those same values
    q32, k32, v32 = (x.astype(np.float32).astype(np.float64) for x in (q, k, v))
    g32, b32 = g.astype(np.float32).astype(np.float64), beta.astype(np.float32).astype(np.float64)
    o, S = kernel_algebra(q32, k32, v32, g32, b32, 0.3, h0, C)
    np.testing.assert_allclose(o, ro[0], rtol=1e-9, atol=1e-10)
    np.testing.assert_allclose(S, rS[0], rtol=1e-9, atol=1e-10)


@pytest.mark.parametrize("mutant", ["no_diagonal", "decay_from_start"])
def test_planted_slips_are_detected(mutant):
    q, k, v, g, beta, h0 = _case(3, 100, 16, 8)
    ro, _ = gd.forward(q[None].astype(np.float32), k[None].astype(np.float32),
                       v[None].astype(np.float32), g[None].astype(np.float32),
                       beta[None].astype(np.float32), 0.3, h0[None])
    q, k, v = (x.astype(np.float32).astype(np.float64) for x in (q, k, v))
    g, beta = g.astype(np.float32).astype(np.float64), beta.astype(np.float32).astype(np.float64)
    o, _ = kernel_algebra(q, k, v, g, beta, 0.3, h0, mutant=mutant)
    assert np.linalg.norm(o - ro[0]) / np.linalg.norm(ro[0]) > 1e-3
