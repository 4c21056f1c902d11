"""Seeded synthetic workloads for paged decode attention.

This module builds inputs only: block pools, block tables, sequence lengths,
queries and affine scale/bias planes. It holds none of the attention
arithmetic, so both the CPU oracle (``oracle/``) and the CUDA library can be
fed from it without sharing any computation.

Layouts follow the paged KV pool of the mlx-bun pages
("@mlx-bun/inference 0.0.0-stage -> 1.0.0", state/paged/cache.ts, class
``BlockPool``: every plane is ``[numBlocks, H_kv, blockSize, width]``):

* bf16 pages: ``k_pool`` bf16 ``[NB, HK, BS, D]``, ``v_pool`` ``[NB, HK, BS, Dv]``;
* affine pages: packed codes as int32 bit patterns of uint32 words
  ``[NB, HK, BS, D*bits/32]`` plus bf16 ``scales``/``biases``
  ``[NB, HK, BS, D/group]`` for K, and the same with Dv for V.

D is the key (and query) head dim, Dv the value head dim (the pages'
``headDim`` and ``vHeadDim``; equal unless a spec sets ``v_head_dim``).

Uniform codes packed 8 (4-bit) or 4 (8-bit) per word are exactly uniform
random 32-bit words, so the generator draws words directly and never packs.

Stale storage is poisoned with NaN so that any read of it shows up: blocks
that no table references, and the rows at or past ``len`` in each sequence's
last page (the cache's trim leaves old bytes there and reads stop at the
sequence length, cache.ts ``trim``).
For affine pages the scales of those rows are NaN.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import torch

BF16_NAN = float("nan")


@dataclass(frozen=True)
class DecodeSpec:
    """One decode workload: shapes, page format, length mix and pool rule."""

    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    n_query: int
    block_size: int
    bits: int  # 16 = bf16 pages; 4 or 8 = affine codes
    group_size: int = 64
    lengths: Optional[tuple] = None  # fixed per-sequence lengths
    length_range: Optional[tuple] = None  # (lo, hi) inclusive, drawn uniformly
    pool_factor: float = 2.0  # pool blocks = ceil(factor * blocks needed)
    partition_tokens: int = 0  # 0 = library choice; -1 = one partition
    window: int = 0  # sliding window in rows (0 = none)
    seed: int = 0
    description: str = ""
    v_head_dim: int = 0  # value head dim; 0 = head_dim

    @property
    def rep(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def dv(self) -> int:
        return self.v_head_dim or self.head_dim


@dataclass
class DecodeCase:
    """Tensors of one workload instance (all on one device)."""

    spec: DecodeSpec
    q: torch.Tensor
    k_pool: torch.Tensor
    v_pool: torch.Tensor
    block_tables: torch.Tensor  # int32 [B, max_blocks]; unused entries = -1
    seq_lens: torch.Tensor  # int32 [B]
    scale: float
    num_blocks: int
    k_scales: Optional[torch.Tensor] = None
    k_biases: Optional[torch.Tensor] = None
    v_scales: Optional[torch.Tensor] = None
    v_biases: Optional[torch.Tensor] = None
    lens_host: list = field(default_factory=list)
    tables_host: list = field(default_factory=list)

    @property
    def partition_tokens(self) -> int:
        p = self.spec.partition_tokens
        if p < 0:  # one partition covering the longest sequence
            return self.block_tables.shape[1] * self.spec.block_size
        return p

    def to(self, device) -> "DecodeCase":
        mv = lambda t: None if t is None else t.to(device)
        return replace(
            self,
            q=mv(self.q), k_pool=mv(self.k_pool), v_pool=mv(self.v_pool),
            block_tables=mv(self.block_tables), seq_lens=mv(self.seq_lens),
            k_scales=mv(self.k_scales), k_biases=mv(self.k_biases),
            v_scales=mv(self.v_scales), v_biases=mv(self.v_biases),
        )


# ---------------------------------------------------------------------------
# The five workloads of this library's measurement plan.
# ---------------------------------------------------------------------------

WORKLOADS = {
    "bf16_1x1024_hq2_d256": DecodeSpec(
        name="bf16_1x1024_hq2_d256", num_seqs=1, num_q_heads=2, num_kv_heads=1, head_dim=256,
        n_query=1, block_size=16, bits=16, lengths=(1024,), pool_factor=2.0,
        partition_tokens=-1, seed=1001,
        description="bf16 paged decode, 1 sequence x 1 query, HQ=2 HK=1 D=256, len 1024, "
                    "BS=16, 64 pages from a 128-block pool, one partition"),
    "affine4_g64_1x8192_hq16_d256": DecodeSpec(
        name="affine4_g64_1x8192_hq16_d256", num_seqs=1, num_q_heads=16, num_kv_heads=4,
        head_dim=256, n_query=1, block_size=32, bits=4, lengths=(8192,), pool_factor=2.0,
        partition_tokens=512, seed=1002,
        description="4-bit affine group-64 paged decode, 1 sequence x 1 query, HQ=16 HK=4 D=256, "
                    "len 8192, BS=32, 512-token partitions then merge"),
    "bf16_batch32_hq32_d128": DecodeSpec(
        name="bf16_batch32_hq32_d128", num_seqs=32, num_q_heads=32, num_kv_heads=8, head_dim=128,
        n_query=1, block_size=16, bits=16, length_range=(512, 16384), pool_factor=1.1,
        partition_tokens=0, seed=1003,
        description="bf16 paged decode batch, 32 sequences x 1 query, lengths U[512,16384], "
                    "HQ=32 HK=8 D=128, BS=16, shared pool +10% free blocks"),
    "affine4_batch64_hq32_d256": DecodeSpec(
        name="affine4_batch64_hq32_d256", num_seqs=64, num_q_heads=32, num_kv_heads=8, head_dim=256,
        n_query=1, block_size=32, bits=4, length_range=(1024, 32768), pool_factor=1.1,
        partition_tokens=0, seed=1004,
        description="affine paged decode batch, 4-bit layer: 64 sequences x 1 query, lengths "
                    "U[1024,32768], HQ=32 HK=8 D=256, BS=32, group 64"),
    "affine8_batch64_hq32_d256": DecodeSpec(
        name="affine8_batch64_hq32_d256", num_seqs=64, num_q_heads=32, num_kv_heads=8, head_dim=256,
        n_query=1, block_size=32, bits=8, length_range=(1024, 32768), pool_factor=1.1,
        partition_tokens=0, seed=1004,
        description="affine paged decode batch, 8-bit layer (same lengths and tables as the "
                    "4-bit layer)"),
    "bf16_8x131072_n4_hq32_d128": DecodeSpec(
        name="bf16_8x131072_n4_hq32_d128", num_seqs=8, num_q_heads=32, num_kv_heads=8, head_dim=128,
        n_query=4, block_size=16, bits=16, lengths=(131072,) * 8, pool_factor=2.0,
        partition_tokens=0, seed=1005,
        description="long-context few-query paged decode, 8 sequences x 4 queries, len 131072, "
                    "HQ=32 HK=8 D=128, BS=16, fragmented 2x pool"),
    "bf16_8x131072_n4_w8192_hq32_d128": DecodeSpec(
        name="bf16_8x131072_n4_w8192_hq32_d128", num_seqs=8, num_q_heads=32, num_kv_heads=8, head_dim=128,
        n_query=4, block_size=16, bits=16, lengths=(131072,) * 8, pool_factor=2.0, window=8192,
        partition_tokens=0, seed=1006,
        description="sliding-window few-query paged decode: the long-context workload with an 8192-row "
                    "window (each query sees its 8192 most recent rows)"),
    "bf16_batch32_hq32_dk192_dv128": DecodeSpec(
        name="bf16_batch32_hq32_dk192_dv128", num_seqs=32, num_q_heads=32, num_kv_heads=8, head_dim=192,
        v_head_dim=128, n_query=1, block_size=16, bits=16, length_range=(512, 16384), pool_factor=1.1,
        partition_tokens=0, seed=1007,
        description="bf16 paged decode batch with key head dim 192 and value head dim 128: 32 sequences x "
                    "1 query, lengths U[512,16384], HQ=32 HK=8, BS=16, shared pool +10% free blocks"),
}

# The two layers of the affine batch workload form one decode step.
LAYER_GROUPS = {
    "affine_batch64_hq32_d256": ("affine4_batch64_hq32_d256", "affine8_batch64_hq32_d256"),
}


def _draw_lengths(spec: DecodeSpec, gen: torch.Generator) -> list:
    if spec.lengths is not None:
        assert len(spec.lengths) == spec.num_seqs
        return [int(x) for x in spec.lengths]
    lo, hi = spec.length_range
    return [int(x) for x in torch.randint(lo, hi + 1, (spec.num_seqs,), generator=gen)]


def draw_lengths(spec: DecodeSpec, seed: Optional[int] = None) -> list:
    """The seeded per-sequence lengths ``make_case`` uses for ``spec``."""
    seed = spec.seed if seed is None else seed
    return _draw_lengths(spec, torch.Generator(device="cpu").manual_seed(seed))


def make_case(spec: DecodeSpec, device="cpu", seed: Optional[int] = None, poison: bool = True,
              lengths: Optional[list] = None) -> DecodeCase:
    """Draw one seeded instance of ``spec`` on ``device``.

    Lengths and block tables come from a CPU generator (so they do not depend
    on the device); values are drawn on ``device`` with a generator seeded
    from the same seed.
    """
    seed = spec.seed if seed is None else seed
    device = torch.device(device)
    cpu = torch.Generator(device="cpu").manual_seed(seed)
    lens = list(lengths) if lengths is not None else _draw_lengths(spec, cpu)
    B, HQ, HK, D, N, BS = (spec.num_seqs, spec.num_q_heads, spec.num_kv_heads, spec.head_dim,
                           spec.n_query, spec.block_size)
    assert len(lens) == B and all(l >= 0 for l in lens)
    pages = [math.ceil(l / BS) for l in lens]
    needed = sum(pages)
    num_blocks = max(1, math.ceil(spec.pool_factor * needed - 1e-9))
    num_blocks = max(num_blocks, needed)
    perm = torch.randperm(num_blocks, generator=cpu)
    max_blocks = max(1, max(pages))
    tables = torch.full((B, max_blocks), -1, dtype=torch.int32)
    tables_host, pos = [], 0
    for b in range(B):
        row = perm[pos:pos + pages[b]].to(torch.int32)
        tables[b, :pages[b]] = row
        tables_host.append([int(x) for x in row])
        pos += pages[b]
    used = perm[:needed]

    gen = torch.Generator(device=device).manual_seed(seed)
    DV = spec.dv
    q = torch.randn((B, HQ, N, D), generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)
    ks = kb = vs = vb = None
    if spec.bits == 16:
        k_pool = torch.randn((num_blocks, HK, BS, D), generator=gen, device=device, dtype=torch.bfloat16)
        v_pool = torch.randn((num_blocks, HK, BS, DV), generator=gen, device=device, dtype=torch.bfloat16)
    else:
        assert spec.bits in (4, 8) and D % spec.group_size == 0 and DV % spec.group_size == 0

        def codes(dim):
            w = torch.randint(0, 1 << 32, (num_blocks, HK, BS, dim * spec.bits // 32), generator=gen,
                              device=device, dtype=torch.int64)
            return w.to(torch.int32)

        def scales(dim):
            s = torch.randn((num_blocks, HK, BS, dim // spec.group_size), generator=gen, device=device,
                            dtype=torch.float32)
            return (s.abs_() * 0.05 + 0.01).to(torch.bfloat16)

        def biases(dim):
            s = torch.randn((num_blocks, HK, BS, dim // spec.group_size), generator=gen, device=device,
                            dtype=torch.float32)
            return (s * 0.2).to(torch.bfloat16)

        k_pool, ks, kb = codes(D), scales(D), biases(D)
        v_pool, vs, vb = codes(DV), scales(DV), biases(DV)

    if poison:
        value_planes = [k_pool, v_pool] if spec.bits == 16 else [ks, kb, vs, vb]
        mask = torch.ones(num_blocks, dtype=torch.bool)
        mask[used] = False
        unused = mask.nonzero().flatten().to(device)
        for t in value_planes:
            if unused.numel():
                t.index_fill_(0, unused, BF16_NAN)
        for b in range(B):
            if lens[b] % BS and pages[b]:
                last = tables_host[b][-1]
                for t in value_planes:
                    t[last, :, lens[b] % BS:, :] = BF16_NAN

    return DecodeCase(
        spec=spec, q=q, k_pool=k_pool, v_pool=v_pool,
        block_tables=tables.to(device), seq_lens=torch.tensor(lens, dtype=torch.int32).to(device),
        scale=1.0 / math.sqrt(D), num_blocks=num_blocks,
        k_scales=ks, k_biases=kb, v_scales=vs, v_biases=vb,
        lens_host=lens, tables_host=tables_host,
    )


def row_bytes(spec: DecodeSpec, dim: Optional[int] = None) -> int:
    """Bytes of one stored row of head dim ``dim`` (default the key head dim): a bf16
    row, or codes + bf16 scale and bias."""
    D = spec.head_dim if dim is None else dim
    if spec.bits == 16:
        return 2 * D
    return D * spec.bits // 8 + (D // spec.group_size) * 4


def required_kv_bytes(spec: DecodeSpec, lens) -> int:
    """K/V bytes a decode step must read: every visible cached row once per KV head, K and V.
    With a sliding window W the N queries of a sequence together see its last W + N - 1 rows."""
    rows = sum(min(l, spec.window + spec.n_query - 1) if spec.window > 0 else l for l in lens)
    return int(rows) * spec.num_kv_heads * (row_bytes(spec) + row_bytes(spec, spec.dv))
