"""Plain, slow, float64 CPU oracle for paged decode attention.

TEST INFRASTRUCTURE ONLY. The CUDA library never imports or calls this file;
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg use it. It imports only numpy.

What it computes is the plain definition of the decode read described on the
mlx-bun pages ("@mlx-bun/inference 0.0.0-stage -> 1.0.0", diff page 50:
package/src/kernels/attention/paged.ts, the ``paged_attention_partial`` /
``paged_attention_affine_partial`` / ``paged_attention_merge`` kernels and
``pagedAttentionView``; the same text appears on "mlx-bun 0.4.0 -> 0.5.0",
lab/paged-kv/paged-attention.ts). The direct paged read reaches, up to
summation order, the result of the control arm on those pages (gather the
pages, dequantise, then one softmax over the visible keys), so the oracle is
that control arm written out in float64:

For every sequence b, query row i in [0, N) and query head h::

    kv = h // (HQ // HK)                         consecutive query heads share a KV head
    T  = len_b - N + i + 1                       key t is visible iff t <= len_b - N + i
    lo = max(0, T - W) with a sliding window W   ... and t >= lo (the W most recent rows)
    K[t] = k_pool[table_b[t // BS], kv, t % BS]  block-table gather, t < T
    affine pages: K[t][d] = s[t][d // G] * code[t][d] + b[t][d // G]
    score_t = scale * sum_d q[d] * K[t][d]
    p = softmax(score);  out = sum_t p_t * V[t]

``len_b`` counts the N new rows, which are appended before the read
(state/paged/cache.ts, ``PagedKVCache.appendDecode``). The window follows the
causal mask with a window size of kernels/attention/masks.ts
(``createCausalMask``): a query at position pos sees keys in (pos - W, pos].

Every function below is pinned by the CPU tests in ``tests/test_oracle.py``
(closed forms, special cases, brute force against a library routine).
"""

from __future__ import annotations

import math

import numpy as np


def unpack_codes(words, bits: int) -> np.ndarray:
    """Affine codes from packed 32-bit words, lowest bits first.

    Code ``i`` of a row lives in word ``i // PACK`` at bit offset
    ``(i % PACK) * bits`` with ``PACK = 32 // bits`` (paged.ts, affine partial:
    the ``keys[i/PACK] >> ((i%PACK)*BITS) & ((1<<BITS)-1)`` read; kvq4-decode.ts
    reads nibble ``i`` of a word as ``(word >> 4i) & 15``). Widths that would
    straddle a word are not direct-readable (cache.ts, ``directReadable``).

    ``words``: integer array ``[..., W]`` (uint32 words or their int32 bit
    patterns). Returns int64 ``[..., W * PACK]``.
    """
    if bits not in (1, 2, 4, 8, 16):
        raise ValueError(f"codes of {bits} bits straddle a 32-bit word")
    words = np.asarray(words).astype(np.int64) & 0xFFFFFFFF
    pack = 32 // bits
    mask = (1 << bits) - 1
    shifts = np.arange(pack, dtype=np.int64) * bits
    codes = (words[..., None] >> shifts) & mask
    return codes.reshape(words.shape[:-1] + (words.shape[-1] * pack,))


def dequantize(words, scales, biases, bits: int, group_size: int) -> np.ndarray:
    """Affine dequantisation ``value = scale * code + bias``, in float64.

    ``scales``/``biases``: ``[..., D // group_size]`` (the bf16 planes' values);
    dim ``d`` uses group ``d // group_size`` (paged.ts affine partial,
    ``ks[i/GROUP]`` and ``kb[i/GROUP]``; kvq4-decode.ts ``fma(scale, code,
    bias)``). The value is not rounded back to bf16 here.
    """
    codes = unpack_codes(words, bits).astype(np.float64)
    D = codes.shape[-1]
    g = np.arange(D) // group_size
    s = np.asarray(scales, dtype=np.float64)
    b = np.asarray(biases, dtype=np.float64)
    return s[..., g] * codes + b[..., g]


def gather_pages(pool, table, length: int) -> np.ndarray:
    """Logical rows ``[0, length)`` of one sequence, gathered out of the pool.

    ``pool``: ``[NB, HK, BS, W]`` of any dtype; ``table``: the sequence's
    logical-to-physical block list. Row ``t`` is ``pool[table[t // BS], :,
    t % BS, :]`` (paged.ts partial kernel: ``physical = table[token / BS]``,
    row ``token % BS``; cache.ts ``pickBlocks``). Returns ``[HK, length, W]``
    with the pool's dtype, so the gather itself is bit-exact.
    """
    pool = np.asarray(pool)
    table = np.asarray(table, dtype=np.int64)
    BS = pool.shape[2]
    t = np.arange(length)
    rows = pool[table[t // BS], :, t % BS, :]  # [length, HK, W]
    return np.ascontiguousarray(rows.transpose(1, 0, 2))


def softmax_weights(scores) -> np.ndarray:
    """Softmax of a score vector, in float64."""
    s = np.asarray(scores, dtype=np.float64)
    e = np.exp(s - s.max())
    return e / e.sum()


def attend(q, K, V, scale: float) -> np.ndarray:
    """One query vector against visible keys ``K [T, D]`` and values ``V [T, Dv]``."""
    scores = scale * (np.asarray(K, dtype=np.float64) @ np.asarray(q, dtype=np.float64))
    p = softmax_weights(scores)
    return p @ np.asarray(V, dtype=np.float64)


def partition_states(q, K, V, scale: float, bounds):
    """Per-partition online-softmax state ``(m, l, o)`` of one query vector.

    For the key range ``[lo, hi)`` of each partition: ``m`` is the largest
    score, ``l = sum exp(score - m)`` and ``o = sum exp(score - m) * V``
    (paged.ts partial kernel: ``maximum``, ``total``, ``accum``). An empty
    range gives ``(-inf, 0, 0)``.
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    states = []
    for lo, hi in bounds:
        if hi <= lo:
            states.append((-math.inf, 0.0, np.zeros(V.shape[1])))
            continue
        s = scale * (K[lo:hi] @ q)
        m = float(s.max())
        e = np.exp(s - m)
        states.append((m, float(e.sum()), e @ V[lo:hi]))
    return states


def lse_merge(states) -> np.ndarray:
    """Combine partition states by log-sum-exp.

    ``M = max m_p``; ``out = sum_p e^(m_p - M) o_p / sum_p e^(m_p - M) l_p``,
    skipping partitions with ``m_p = -inf`` (kvq4-decode.ts and
    multi-query.ts merge kernels skip them; paged.ts merge weights them by
    ``exp(-inf) = 0``).
    """
    live = [(m, l, o) for (m, l, o) in states if m != -math.inf]
    if not live:
        raise ValueError("every partition is empty")
    M = max(m for m, _, _ in live)
    num = sum(math.exp(m - M) * o for m, _, o in live)
    den = sum(math.exp(m - M) * l for m, l, _ in live)
    return num / den


def kv_head(h: int, num_q_heads: int, num_kv_heads: int) -> int:
    """KV head serving query head ``h``: consecutive groups of ``HQ // HK`` heads
    (paged.ts partial kernel ``hk = hq / (HQ / HK)``; kvq4-decode.ts reads
    query head ``hk * REP + j``)."""
    return h // (num_q_heads // num_kv_heads)


def _sequence_kv(k_pool, v_pool, table, length, kv_heads, bits, group_size, planes):
    """Gathered float64 K and V of the listed KV heads: dict kv -> (K, V)."""
    out = {}
    for kv in kv_heads:
        sl = slice(kv, kv + 1)
        Kw = gather_pages(np.asarray(k_pool)[:, sl], table, length)[0]
        Vw = gather_pages(np.asarray(v_pool)[:, sl], table, length)[0]
        if bits == 16:
            K, V = Kw.astype(np.float64), Vw.astype(np.float64)
        else:
            ks, kb, vs, vb = (gather_pages(np.asarray(p)[:, sl], table, length)[0] for p in planes)
            K = dequantize(Kw, ks, kb, bits, group_size)
            V = dequantize(Vw, vs, vb, bits, group_size)
        out[kv] = (K, V)
    return out


def _rows(B, HQ, rows):
    return [(b, h) for b in range(B) for h in range(HQ)] if rows is None else list(rows)


def visible_range(length: int, n_query: int, i: int, window: int = 0):
    """Keys [lo, hi) visible to query row i of a sequence holding ``length`` rows."""
    hi = length - n_query + i + 1
    lo = max(0, hi - window) if window > 0 else 0
    return lo, hi


def paged_decode_attention(q, k_pool, v_pool, block_tables, seq_lens, scale: float, n_query: int, *,
                           bits: int = 16, group_size: int = 64, k_scales=None, k_biases=None,
                           v_scales=None, v_biases=None, rows=None, window: int = 0) -> np.ndarray:
    """Decode attention over a paged cache, float64 ``[B, HQ, N, Dv]``.

    ``q``: float ``[B, HQ, N, D]``; ``k_pool``/``v_pool``: float values
    ``[NB, HK, BS, D]`` (bits=16) or packed words ``[NB, HK, BS, D*bits/32]``
    with scale/bias planes ``[NB, HK, BS, D/group]``; ``block_tables``
    ``[B, >=ceil(len/BS)]``; ``seq_lens`` ``[B]`` (each ``>= n_query``).
    ``rows``: optional ``(b, h)`` pairs to compute; the others stay NaN.
    """
    q = np.asarray(q, dtype=np.float64)
    B, HQ, N, D = q.shape
    assert N == n_query
    HK = np.asarray(k_pool).shape[1]
    if HQ % HK:
        raise ValueError("query heads must be a multiple of KV heads")
    planes = (k_scales, k_biases, v_scales, v_biases)
    Dv = D if bits == 16 else None
    out = None
    by_seq = {}
    for b, h in _rows(B, HQ, rows):
        by_seq.setdefault(b, set()).add(h)
    for b, heads in sorted(by_seq.items()):
        L = int(np.asarray(seq_lens)[b])
        if L < N:
            raise ValueError("a sequence holds fewer rows than its new queries")
        table = np.asarray(block_tables)[b]
        kv_heads = sorted({kv_head(h, HQ, HK) for h in heads})
        kvs = _sequence_kv(k_pool, v_pool, table, L, kv_heads, bits, group_size, planes)
        for h in sorted(heads):
            K, V = kvs[kv_head(h, HQ, HK)]
            if out is None:
                Dv = V.shape[1]
                out = np.full((B, HQ, N, Dv), np.nan)
            for i in range(N):
                lo, hi = visible_range(L, N, i, window)
                out[b, h, i] = attend(q[b, h, i], K[lo:hi], V[lo:hi], scale)
    if out is None:
        out = np.full((B, HQ, N, Dv if Dv else D), np.nan)
    return out


def paged_decode_attention_partitioned(q, k_pool, v_pool, block_tables, seq_lens, scale: float,
                                       n_query: int, partition_tokens: int, *, bits: int = 16,
                                       group_size: int = 64, k_scales=None, k_biases=None,
                                       v_scales=None, v_biases=None, rows=None, window: int = 0) -> np.ndarray:
    """The split-sequence form: partitions of ``partition_tokens`` cache rows.

    Partition ``p`` of sequence b covers rows ``[p*P, min((p+1)*P, len_b))``;
    query i keeps only its visible rows in it, so late partitions may be empty
    for early queries. Each partition's ``(m, l, o)`` is combined by
    :func:`lse_merge`. Mathematically equal to :func:`paged_decode_attention`.
    """
    q = np.asarray(q, dtype=np.float64)
    B, HQ, N, D = q.shape
    HK = np.asarray(k_pool).shape[1]
    P = int(partition_tokens)
    if P <= 0:
        raise ValueError("partition_tokens must be positive")
    planes = (k_scales, k_biases, v_scales, v_biases)
    out = None
    by_seq = {}
    for b, h in _rows(B, HQ, rows):
        by_seq.setdefault(b, set()).add(h)
    for b, heads in sorted(by_seq.items()):
        L = int(np.asarray(seq_lens)[b])
        if L < N:
            raise ValueError("a sequence holds fewer rows than its new queries")
        table = np.asarray(block_tables)[b]
        kvs = _sequence_kv(k_pool, v_pool, table, L, sorted({kv_head(h, HQ, HK) for h in heads}),
                           bits, group_size, planes)
        nparts = -(-L // P)
        for h in sorted(heads):
            K, V = kvs[kv_head(h, HQ, HK)]
            if out is None:
                out = np.full((B, HQ, N, V.shape[1]), np.nan)
            for i in range(N):
                lo, hi = visible_range(L, N, i, window)
                bounds = [(max(p * P, lo), min((p + 1) * P, hi)) for p in range(nparts)]
                out[b, h, i] = lse_merge(partition_states(q[b, h, i], K, V, scale, bounds))
    return out
