"""Independent formulations that pin the fp64 oracle (test helpers, numpy fp64).

None of these calls the oracle or shares code with it; each is another way the
pages (or a textbook) state the same result:

* ``dual_form``: "Gated Linear Attention (GLA): Mathematical Foundations, ..."
  (llms.blog), section "The Gated Recurrent Update", the unrolled state and the
  dual attention form o_t = sum_j ((q_t * k_j) . Lambda_{j,t}) v_j with
  Lambda_{j,t} = prod_{m=j+1..t} alpha_m, evaluated by brute force.  The h0
  term comes from the same unrolling with a non-zero S_0.
* ``chunk_form``: same page, sections "Cumulative Decay Representation",
  "Intra-Chunk Matrix Multiplications" and "Inter-Chunk Recurrence and Output
  Projection": Gamma = in-chunk inclusive prefix sum of A = log alpha;
  M = (Q K^T) * D with the decay inside the key-channel contraction;
  O = M V + (Q * exp(Gamma)) S_prev;
  S = diag(exp(Gamma_C)) S_prev + (K * exp(Gamma_C - Gamma))^T V.
* ``causal_linear_attention``: the alpha = 1 case, same page, section
  "Linearized Attention as Associative Memory": O = tril(Q K^T) V.
* ``retention``: the fixed-decay case, same page, section "The Retention and
  Recall Degradation Problem": S_i = gamma S_{i-1} + k_i^T v_i, whose parallel
  form is O = ((Q K^T) * D) V with D_{t,j} = gamma^(t-j) for t >= j.

All take float arrays for one sequence: q, k, a=log_alpha [T, dk], v [T, dv],
h0 [dk, dv] or None, and return o [T, dv] (times ``scale``) and, where the
formulation yields one, the final state.
"""

from __future__ import annotations

import numpy as np


def _d(x):
    return np.asarray(x, dtype=np.float64)


def dual_form(q, k, v, a, scale, h0=None):
    q, k, v, a = _d(q), _d(k), _d(v), _d(a)
    T, dk = q.shape
    dv = v.shape[1]
    alpha = np.exp(a)  # [T, dk]
    o = np.zeros((T, dv))
    lam = np.zeros((T, dk))     # lam[j] = Lambda_{j,t} for the current t (rows j <= t)
    lam0 = np.ones(dk)          # prod_{m=1..t} alpha_m, the decay applied to S_0
    for t in range(T):
        lam[:t] *= alpha[t]     # extend every product by alpha_t
        lam[t] = 1.0            # empty product: Lambda_{t,t} = 1
        lam0 = lam0 * alpha[t]
        w = ((q[t][None, :] * k[: t + 1]) * lam[: t + 1]).sum(axis=1)  # [t+1]
        o[t] = w @ v[: t + 1]
        if h0 is not None:
            o[t] += (q[t] * lam0) @ _d(h0)
    return scale * o


def chunk_form(q, k, v, a, scale, h0=None, C=64):
    q, k, v, a = _d(q), _d(k), _d(v), _d(a)
    T, dk = q.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if h0 is None else _d(h0).copy()
    o = np.zeros((T, dv))
    for u0 in range(0, T, C):
        sl = slice(u0, min(u0 + C, T))
        Q, K, V, A = q[sl], k[sl], v[sl], a[sl]
        n = Q.shape[0]
        G = np.cumsum(A, axis=0)                      # Gamma_i, inclusive
        causal = np.tril(np.ones((n, n), dtype=bool))
        # lambda_{i,j} = exp(Gamma_i - Gamma_j) for i >= j; entries above the
        # diagonal are not part of D and are set to exp(-inf) = 0.
        diff = np.where(causal[:, :, None], G[:, None, :] - G[None, :, :], -np.inf)
        lam = np.exp(diff)                            # [n, n, dk]
        M = np.einsum("id,jd,ijd->ij", Q, K, lam)
        o_intra = M @ V
        o_inter = (Q * np.exp(G)) @ S
        o[sl] = o_intra + o_inter
        GC = G[-1]
        S = np.exp(GC)[:, None] * S + (K * np.exp(GC[None, :] - G)).T @ V
    return scale * o, S


def causal_linear_attention(q, k, v, scale, h0=None):
    q, k, v = _d(q), _d(k), _d(v)
    o = np.tril(q @ k.T) @ v
    if h0 is not None:
        o = o + q @ _d(h0)
    S = k.T @ v + (0.0 if h0 is None else _d(h0))
    return scale * o, S


def retention(q, k, v, gamma, scale, h0=None):
    q, k, v = _d(q), _d(k), _d(v)
    T = q.shape[0]
    t = np.arange(T)
    expo = t[:, None] - t[None, :]
    D = np.where(expo >= 0, np.power(float(gamma), np.maximum(expo, 0)), 0.0)
    o = ((q @ k.T) * D) @ v
    S = (k * np.power(float(gamma), (T - 1 - t))[:, None]).T @ v
    if h0 is not None:
        # S_t carries gamma^t h0 after t tokens (1-based t).
        o = o + (np.power(float(gamma), t + 1)[:, None] * (q @ _d(h0)))
        S = S + gamma ** T * _d(h0)
    return scale * o, S


def rel_err(x, ref):
    x, ref = _d(x), _d(ref)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / (den if den > 0 else 1.0))
