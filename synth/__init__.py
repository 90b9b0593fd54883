"""Seeded synthetic inputs for gated linear attention (GLA).

This package holds only the random-number recipes that both the fp64 CPU
oracle (``oracle/``) and the CUDA path are fed with.  It contains none of the
method's arithmetic: it draws q, k, v, the log forget gates, the initial
state and the upstream gradients of a backward call, nothing else.
"""

from .gla_inputs import (  # noqa: F401
    CHUNK_CONFIGS,
    DECODE_CONFIG,
    ChunkConfig,
    DecodeConfig,
    make_backward_grads,
    make_chunk_inputs,
    make_config_inputs,
    make_decode_inputs,
    make_gdn_inputs,
)
