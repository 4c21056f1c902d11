"""CPU oracle for paged decode attention (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never calls it, and it
imports nothing from the library.
"""

from .paged_decode import (  # noqa: F401
    unpack_codes,
    dequantize,
    gather_pages,
    softmax_weights,
    attend,
    partition_states,
    lse_merge,
    paged_decode_attention,
    paged_decode_attention_partitioned,
    visible_range,
)
