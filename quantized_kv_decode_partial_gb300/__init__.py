"""Paged decode attention over a block-pool KV cache (bf16 or affine 4/8-bit pages)
for GB300 (sm_103a): hand-written CUDA kernels behind a C ABI (libpkvdecode.so),
with a thin ctypes binding."""

from .binding import (  # noqa: F401
    EXPORTS,
    LibraryNotBuilt,
    PkvError,
    DecodeParams,
    Plan,
    PoolLayout,
    load_library,
    make_plan,
    paged_decode_attention,
    paged_decode_passes,
    paged_decode_append_attention,
    HostDecodeStep,
    paged_append,
    paged_gather,
    set_wait_limit_ns,
)
