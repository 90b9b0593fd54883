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

* ``chunk_form_backward``: the same chunk equations differentiated, in the
  form the backward kernels evaluate (in-chunk products, state terms against
  the chunk-start states and state gradients, the log-gate carry); pinned
  against the oracle's reverse-mode backward.

* ``gdn_chunk_form``: the gated delta rule's four-step chunk algorithm
  (KK^T-based lower-triangular inverse, W and U, the chunk recurrence, the
  output), derived from the token recurrence; pins the GDN oracle.

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


def chunk_form_backward(q, k, v, a, scale, do, h0=None, dhT=None, C=64):
    """Gradients of sum <do, o> + <dhT, hT> in chunk form (the equations the
    backward kernels evaluate).  Per chunk u of C tokens, Gamma the in-chunk
    inclusive prefix sums, S_u the state entering the chunk and R_u the
    gradient of the state leaving it:
        A  = tril(dO V^T),  lam_ij = exp(Gamma_i - Gamma_j) (i >= j)
        dQ = scale [ e^Gamma (dO S_u^T) + sum_j A_ij K_j lam_ij ]
        dK = e^(Gamma_C - Gamma) (V R_u^T) + scale sum_i A_ij Q_i lam_ij
        dV = (K e^(Gamma_C - Gamma)) R_u + scale M^T dO,  M_ij = sum_d Q K lam
        dlog_alpha_t = rowsum(R_u * S_(u+1)) + sum_(tau >= t in chunk) (q dq - k dk)
        R_(u-1) = e^Gamma_C R_u + scale (Q e^Gamma)^T dO,  R_last = dhT,  dh0 = R_(-1)
    Returns (dq, dk, dv, dlog_alpha, dh0)."""
    q, k, v, a, do = _d(q), _d(k), _d(v), _d(a), _d(do)
    T, dk = q.shape
    dv = v.shape[1]
    starts = list(range(0, T, C))
    # forward: the state entering every chunk, and the one leaving the last
    S = [np.zeros((dk, dv)) if h0 is None else _d(h0).copy()]
    for u0 in starts:
        sl = slice(u0, min(u0 + C, T))
        G = np.cumsum(a[sl], axis=0)
        S.append(np.exp(G[-1])[:, None] * S[-1] + (k[sl] * np.exp(G[-1][None, :] - G)).T @ v[sl])
    dq, dkk, dvv, da = (np.zeros_like(x) for x in (q, k, v, a))
    R = np.zeros((dk, dv)) if dhT is None else _d(dhT).copy()
    for u in reversed(range(len(starts))):
        sl = slice(starts[u], min(starts[u] + C, T))
        Q, K, V, DO = q[sl], k[sl], v[sl], do[sl]
        n = Q.shape[0]
        G = np.cumsum(a[sl], axis=0)
        causal = np.tril(np.ones((n, n), dtype=bool))
        lam = np.exp(np.where(causal[:, :, None], G[:, None, :] - G[None, :, :], -np.inf))
        A = np.where(causal, DO @ V.T, 0.0)
        M = np.einsum("id,jd,ijd->ij", Q, K, lam)
        dQ = scale * (np.exp(G) * (DO @ S[u].T) + np.einsum("ij,jd,ijd->id", A, K, lam))
        dK = np.exp(G[-1][None, :] - G) * (V @ R.T) + scale * np.einsum("ij,id,ijd->jd", A, Q, lam)
        dV = (K * np.exp(G[-1][None, :] - G)) @ R + scale * M.T @ DO
        carry = np.sum(R * S[u + 1], axis=1)
        P = Q * dQ - K * dK
        da[sl] = carry[None, :] + np.flip(np.cumsum(np.flip(P, axis=0), axis=0), axis=0)
        dq[sl], dkk[sl], dvv[sl] = dQ, dK, dV
        R = np.exp(G[-1])[:, None] * R + scale * (Q * np.exp(G)).T @ DO
    return dq, dkk, dvv, da, R


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


def gdn_chunk_form(q, k, v, g, beta, scale, h0=None, C=64):
    """The gated delta rule by its chunk algorithm ("Qwen Team Releases FlashQLA
    ...", the four steps of the GDN prefill): per chunk, with gamma_t the
    in-chunk product of the gates and Delta the per-token write errors,
      1. T = (I + L)^-1, L strictly lower, L_ti = beta_t (gamma_t/gamma_i) k_t.k_i;
      2. U = T diag(beta) V,  W = T diag(beta) diag(gamma) K;
      3. S_C = gamma_C S_0 + (diag(gamma_C/gamma) K)^T (U - W S_0);
      4. O = scale [diag(gamma) Q S_0 + tril(Q K^T * gamma_t/gamma_i) (U - W S_0)].
    Returns (o [T, dv], hT [dk, dv])."""
    q, k, v, g, beta = _d(q), _d(k), _d(v), _d(g), _d(beta)
    T, dk = q.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if h0 is None else _d(h0).copy()
    o = np.zeros((T, dv))
    for u0 in range(0, T, C):
        sl = slice(u0, min(u0 + C, T))
        Q, K, V, b = q[sl], k[sl], v[sl], beta[sl]
        n = Q.shape[0]
        G = np.cumsum(g[sl])                                   # log gamma_t
        low = np.tril(np.ones((n, n), dtype=bool))
        ratio = np.exp(np.where(low, G[:, None] - G[None, :], -np.inf))   # gamma_t / gamma_i, i <= t
        L = np.where(np.tril(np.ones((n, n), dtype=bool), -1), b[:, None] * ratio * (K @ K.T), 0.0)
        Tm = np.linalg.inv(np.eye(n) + L)
        U = Tm @ (b[:, None] * V)
        W = Tm @ (b[:, None] * np.exp(G)[:, None] * K)
        D = U - W @ S
        o[sl] = scale * (np.exp(G)[:, None] * (Q @ S) + ((Q @ K.T) * ratio) @ D)
        S = np.exp(G[-1]) * S + (K * np.exp(G[-1] - G)[:, None]).T @ D
    return o, S



def gdn_chunk_transition(k, g, beta, C=64):
    """Per chunk of the gated delta rule, the matrix M with S_C = M S_0 + K~^T U:
    M = gamma_C I - K~^T W, K~ = diag(gamma_C/gamma) K (step 3 of the four-step
    chunk algorithm, regrouped around S_0).  Returns the list over chunks."""
    k, g, beta = _d(k), _d(g), _d(beta)
    T, dk = k.shape
    Ms = []
    for u0 in range(0, T, C):
        sl = slice(u0, min(u0 + C, T))
        K, b = k[sl], beta[sl]
        n = K.shape[0]
        G = np.cumsum(g[sl])
        low = np.tril(np.ones((n, n), dtype=bool))
        ratio = np.exp(np.where(low, G[:, None] - G[None, :], -np.inf))
        L = np.where(np.tril(np.ones((n, n), dtype=bool), -1), b[:, None] * ratio * (K @ K.T), 0.0)
        Tm = np.linalg.inv(np.eye(n) + L)
        W = Tm @ (b[:, None] * np.exp(G)[:, None] * K)
        Kt = K * np.exp(G[-1] - G)[:, None]
        Ms.append(np.exp(G[-1]) * np.eye(dk) - Kt.T @ W)
    return Ms


def gdn_segment_form(q, k, v, g, beta, scale, h0=None, C=64, seg_chunks=2):
    """The gated delta rule with the sequence split into segments of seg_chunks
    chunks ("Qwen Team Releases FlashQLA ...", "Core Technical Principles": the
    error of a state started from a wrong initial value evolves by a dk x dk
    matrix per chunk, and those matrices associate).  Pass 1: every segment
    runs from a zero state to its end state S*_s, and the product M_s of its
    chunks' transition matrices is formed.  Pass 2, serial over segments:
    start_{s+1} = M_s start_s + S*_s from start_0 = h0.  Pass 3: every segment
    runs again from its true start (the state is computed twice, as the page
    says).  Returns (o [T, dv], hT [dk, dv])."""
    q, k, v, g, beta = _d(q), _d(k), _d(v), _d(g), _d(beta)
    T, dk = q.shape
    dv = v.shape[1]
    span = C * seg_chunks
    bounds = [(s0, min(s0 + span, T)) for s0 in range(0, T, span)]
    Ms = gdn_chunk_transition(k, g, beta, C)
    ends, prods = [], []
    for si, (a, b_) in enumerate(bounds):
        _, s_star = gdn_chunk_form(q[a:b_], k[a:b_], v[a:b_], g[a:b_], beta[a:b_], scale, None, C)
        ends.append(s_star)
        P = np.eye(dk)
        for c in range(a // C, (b_ + C - 1) // C):
            P = Ms[c] @ P
        prods.append(P)
    start = np.zeros((dk, dv)) if h0 is None else _d(h0).copy()
    starts = []
    for P, s_star in zip(prods, ends):
        starts.append(start)
        start = P @ start + s_star
    o = np.zeros((T, dv))
    hT = None
    for (a, b_), s0 in zip(bounds, starts):
        o[a:b_], hT = gdn_chunk_form(q[a:b_], k[a:b_], v[a:b_], g[a:b_], beta[a:b_], scale, s0, C)
    return o, hT
