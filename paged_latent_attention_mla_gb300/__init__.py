"""Paged Multi-Head Latent Attention decode for GB300 (sm_103a).

The compute path is libmla_gb300.so (hand-written CUDA, C ABI in include/mla.h);
``_native`` binds it, ``api`` wraps plan + workspace + decode, ``workloads``
draws seeded synthetic decode batches.
"""

from . import workloads  # noqa: F401
from .api import PagedMlaDecoder, decoder_for, merge_ranks  # noqa: F401
