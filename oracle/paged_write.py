"""CPU oracle of the paged cache's write side: appending new K/V rows into their
pages, quantising affine pages on the way (test infrastructure only, like the
rest of ``oracle/``).

The pages append a step's rows by splitting them along block boundaries and
writing each piece into its block at the row offset inside it
("@mlx-bun/inference 0.0.0-stage -> 1.0.0", state/paged/cache.ts:
``PagedKVCache.append`` and ``BlockPool.writeBlock``). Affine pages quantise the
rows first with the framework's affine quantiser, per row and per 64-dim group,
into packed codes (lowest bits first) plus a scale and a bias stored in the
cache's dtype. The quantiser's formula is not on the pages; this oracle takes
the plain min/max reading, with every step in float32 as a GPU takes it:

    lo, hi = min and max of the group (bf16 values, exact in float32)
    scale  = bf16((hi - lo) / (2^bits - 1)),  bias = bf16(lo)
    code   = clamp(round_half_even((x - bias) / scale), 0, 2^bits - 1)
             (code 0 everywhere when the stored scale is 0)

so that the stored scale and bias are the ones the codes were chosen for. The
quantiser is pinned by ``tests/test_oracle_write.py`` (exact grids, the error
bound of half a step, extremes, constant groups, packing round trips).
"""

from __future__ import annotations

import numpy as np


def bf16_round(x) -> np.ndarray:
    """float32 values rounded to bf16 (nearest, ties to even), returned as float32."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    nan = np.isnan(a)
    out = r.astype(np.uint32).view(np.float32).copy()
    out[nan] = np.nan
    return out


def bf16_bits(x) -> np.ndarray:
    """uint16 bit patterns of float32 values that are already bf16-exact."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    return (a.view(np.uint32) >> 16).astype(np.uint16)


def quantize_groups(x, bits: int, group_size: int = 64):
    """Affine codes, scales and biases of rows ``x`` [..., D] (bf16 values).

    Returns (codes int64 [..., D], scales float32 [..., D/G], biases float32
    [..., D/G]); scales and biases are bf16-exact.
    """
    x = np.asarray(x, dtype=np.float32)
    D = x.shape[-1]
    g = x.reshape(x.shape[:-1] + (D // group_size, group_size))
    lo = g.min(axis=-1)
    hi = g.max(axis=-1)
    levels = np.float32((1 << bits) - 1)
    scale = bf16_round((hi - lo) / levels)
    bias = bf16_round(lo)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = (g - bias[..., None]) / scale[..., None]
    q = np.where(scale[..., None] == 0, np.float32(0), q)
    codes = np.clip(np.rint(q), 0, levels).astype(np.int64)
    return codes.reshape(x.shape), scale, bias


def pack_codes(codes, bits: int) -> np.ndarray:
    """Codes [..., D] packed into uint32 words [..., D*bits/32], lowest bits first."""
    codes = np.asarray(codes, dtype=np.uint64)
    pack = 32 // bits
    c = codes.reshape(codes.shape[:-1] + (codes.shape[-1] // pack, pack))
    shifts = (np.arange(pack, dtype=np.uint64) * np.uint64(bits))
    return (c << shifts).sum(axis=-1).astype(np.uint32)


def append_rows(k_new, v_new, block_tables, seq_lens, k_pool, v_pool, *, bits: int = 16, group_size: int = 64,
                k_scales=None, k_biases=None, v_scales=None, v_biases=None):
    """Writes rows ``k_new``/``v_new`` [B, HK, n, D] (bf16 values) of every sequence
    at cache positions len_b .. len_b + n - 1 into copies of the pools, and returns
    the updated planes as a dict (bf16 pools / affine planes as uint16 bf16 bits and
    uint32 code words).

    Position t of sequence b goes to block ``block_tables[b][t // BS]``, row
    ``t % BS`` (cache.ts ``append``: bi = pos / blockSize, within = pos % blockSize).
    """
    k_new = np.asarray(k_new, dtype=np.float32)
    v_new = np.asarray(v_new, dtype=np.float32)
    B, HK, n, D = k_new.shape
    out = {"k_pool": np.array(k_pool, copy=True), "v_pool": np.array(v_pool, copy=True)}
    if bits != 16:
        for name, plane in (("k_scales", k_scales), ("k_biases", k_biases), ("v_scales", v_scales),
                            ("v_biases", v_biases)):
            out[name] = np.array(plane, copy=True)
    BS = out["k_pool"].shape[2]
    for b in range(B):
        for j in range(n):
            t = int(seq_lens[b]) + j
            blk = int(block_tables[b][t // BS])
            r = t % BS
            for plane, rows, pre in (("k", k_new, "k"), ("v", v_new, "v")):
                x = rows[b, :, j, :]  # [HK, D]
                if bits == 16:
                    out[f"{plane}_pool"][blk, :, r, :] = bf16_bits(x)
                else:
                    codes, sc, bi = quantize_groups(x, bits, group_size)
                    out[f"{plane}_pool"][blk, :, r, :] = pack_codes(codes, bits).view(np.int32)
                    out[f"{pre}_scales"][blk, :, r, :] = bf16_bits(sc)
                    out[f"{pre}_biases"][blk, :, r, :] = bf16_bits(bi)
    return out
