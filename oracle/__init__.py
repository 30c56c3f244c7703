"""fp64 CPU oracle for MLA decode -- TEST INFRASTRUCTURE ONLY.

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
may import this package.  The product path never does; it shares no code with
the CUDA library.  See ``mla_oracle.c`` for what is computed and from which
passages of the pages.
"""
from .oracle import (  # noqa: F401
    build,
    load,
    num_threads,
    rope,
    rope_theta,
    yarn_theta,
    yarn_softmax_scale,
    decode,
    cache_append,
    absorb,
    up_project,
    latent_attention,
    output_project,
    fold_output_weights,
    expand_kv,
    prefill_attention,
)
