"""Seeded synthetic inputs for paged-KV attention.

This package only *draws* inputs: random bf16 tensors, request lengths, page
assignments and the slot numbers a serving scheduler would hand to the
attention layer.  It contains none of the attention arithmetic, so both the
CPU oracle and the CUDA path can consume the same bits without sharing any
computation.
"""

from .paged import (  # noqa: F401
    PagedBatch,
    RequestSpec,
    build_paged_batch,
    make_config,
    CONFIG_NAMES,
    random_small_batch,
    make_spec_verify,
    make_shared_prefix_decode,
    make_small_prefill,
)
