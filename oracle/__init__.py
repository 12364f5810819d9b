"""CPU oracle for attention over a paged KV pool (test infrastructure).

This package is the slow, plain, fp64 statement of what the library computes.
It exists to check the CUDA path and nothing else: only the test suite, the
entry point's smoke check and the benchmark's CPU-baseline / reference arm may
import it.  The product path never calls it and has no CPU fallback.

It shares no code with the CUDA path (kernels, headers, helpers or constants);
the only thing both sides consume is the seeded input generator in
``workloads/``, which draws inputs and does none of the arithmetic.

Every function in ``oracle.attention`` is pinned by CPU tests against facts
that do not come from the oracle itself (brute-force dense attention, closed
forms, invariants, hand-derived worked examples and a library routine); no
function here is "parity unpinned".
"""

from .attention import (  # noqa: F401
    as_f64,
    kv_append,
    paged_gather,
    request_kv,
    attend_rows,
    attend_range,
    paged_decode,
    paged_extend,
    merge_states,
    decode_split_reference,
    shared_prefix_attention,
    rope_angles,
    rope,
    rope_kv_append,
    bf16_round_nearest_even,
)
