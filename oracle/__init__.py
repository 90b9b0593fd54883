"""fp64 CPU oracle for gated linear attention — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, the package entry's ``smoke()`` check and ``bench.py``'s CPU
baseline leg may import this package.  The CUDA library and its Python binding
never do; the oracle shares no code with them.

What it computes (the definition, "Gated Linear Attention (GLA): Mathematical
Foundations, ..." (llms.blog), section "The Gated Recurrent Update"):

    S_t = diag(alpha_t) S_{t-1} + k_t^T v_t,   o_t = scale * q_t S_t,

token by token, in double precision, from S_0 = h0 (zero when absent), and
``backward``: the gradients of sum_t <do_t, o_t> + <dhT, hT> with respect to
q, k, v, log alpha and h0, by reverse-mode differentiation of the same loop.

Pins (checked by ``tests/test_oracle_pins.py``): the unrolled dual attention
form by brute force, vanilla causal linear attention at alpha = 1, RetNet's
fixed decay at alpha = gamma, the chunkwise equations at every chunk size,
state passing across a split, the T = 1 closed form, the alpha -> 0 limit,
linearity in (v, h0), the contraction bound, a hand-worked example, and
mutants of this file that each of those pins must reject.  The backward is
pinned by ``tests/test_oracle_bwd_pins.py``: central differences of the
forward, autograd through the dual attention form, the log-gate identity and
mutants of the backward.

``gdn_oracle`` (its own C file, ``gdn_oracle.c``) is the fp64 token loop of
the gated delta rule (row F4), pinned by ``tests/test_oracle_gdn_pins.py``.
"""

from .gla_oracle import (  # noqa: F401
    backward,
    build,
    forward,
    forward_torch,
    library_path,
    max_threads,
    step,
)
