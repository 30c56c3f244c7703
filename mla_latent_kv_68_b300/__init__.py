"""B300-native weight-absorbed Multi-head Latent Attention decode.

The compute path is the CUDA library ``libmla.so`` (C ABI in include/mla.h),
reached through :mod:`mla_latent_kv_68_b300.binding`.  :mod:`.inputs` draws
the seeded synthetic workloads.
"""

__all__ = ["binding", "inputs", "build"]
