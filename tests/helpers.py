"""Test helpers: run the oracle on a workload instance, cut sampled sub-problems
out of full-size instances, and compare against the parity bound (max-abs 1e-2,
mean-abs 1e-3 on bf16 outputs)."""

from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import oracle
from quantized_kv_decode_partial_gb300 import paged_decode_attention
from quantized_kv_decode_partial_gb300.workloads import DecodeCase, DecodeSpec

MAX_ABS = 1e-2  # on bf16 outputs, against the float64 oracle
MEAN_ABS = 1e-3


def bf16_ulp(x):
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    _, e = np.frexp(np.maximum(np.abs(np.asarray(x, dtype=np.float64)), 2.0 ** -126))
    return np.ldexp(1.0, e - 8)


def f64(t):
    return None if t is None else t.detach().float().double().cpu().numpy()


def oracle_inputs(case: DecodeCase):
    kw = dict(bits=case.spec.bits, group_size=case.spec.group_size)
    if case.spec.bits == 16:
        kp, vp = f64(case.k_pool), f64(case.v_pool)
    else:
        kp, vp = case.k_pool.cpu().numpy(), case.v_pool.cpu().numpy()
        kw.update(k_scales=f64(case.k_scales), k_biases=f64(case.k_biases), v_scales=f64(case.v_scales),
                  v_biases=f64(case.v_biases))
    args = (f64(case.q), kp, vp, case.block_tables.cpu().numpy(), case.seq_lens.cpu().numpy(), case.scale,
            case.spec.n_query)
    return args, kw


def oracle_out(case: DecodeCase, partition_tokens=None, rows=None):
    args, kw = oracle_inputs(case)
    kw["window"] = case.spec.window
    if partition_tokens:
        return oracle.paged_decode_attention_partitioned(*args, partition_tokens, rows=rows, **kw)
    return oracle.paged_decode_attention(*args, rows=rows, **kw)


def run_gpu(case: DecodeCase, partition_tokens=None, error_flag=None, schedule=0):
    pt = case.partition_tokens if partition_tokens is None else partition_tokens
    return paged_decode_attention(case.q, case.k_pool, case.v_pool, case.block_tables, case.seq_lens, case.scale,
                                  bits=case.spec.bits, group_size=case.spec.group_size, k_scales=case.k_scales,
                                  k_biases=case.k_biases, v_scales=case.v_scales, v_biases=case.v_biases,
                                  partition_tokens=pt, window=case.spec.window, error_flag=error_flag,
                                  schedule=schedule)


def assert_close(got, ref, what="", strict=False):
    """The parity bound (max-abs 1e-2, mean-abs 1e-3) on the computation,
    on top of the bf16 output's own representation error: each element may also
    differ by half a bf16 ulp of the exact value (a correctly rounded result
    does), and the mean by a quarter ulp (the mean of a uniform rounding error).
    Only outputs of magnitude >= 2 get more than 0.004 from the added terms.
    With strict=True the plain bound must hold as well, with no allowance (for
    outputs small enough that a correctly rounded bf16 result meets it)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    diff = np.abs(got - ref)
    ulp = bf16_ulp(ref)
    worst = np.max(diff - 0.5 * ulp)
    assert worst <= MAX_ABS, f"{what}: max-abs {diff.max():.3e} (beyond half-ulp {worst:.3e})"
    mean_allow = MEAN_ABS + 0.25 * ulp.mean()
    strict_ok = bool(diff.max() <= MAX_ABS and diff.mean() <= MEAN_ABS)
    log = os.environ.get("PKV_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps({"case": what, "max_abs": float(diff.max()), "mean_abs": float(diff.mean()),
                                "strict_ok": strict_ok, "max_beyond_half_ulp": float(worst),
                                "mean_allow": float(mean_allow), "max_abs_ref": float(np.abs(ref).max()),
                                "mean_abs_ref": float(np.abs(ref).mean())}) + "\n")
    assert diff.mean() <= mean_allow, f"{what}: mean-abs {diff.mean():.3e} > {mean_allow:.3e}"
    if strict:
        assert strict_ok, f"{what}: strict bound missed: max-abs {diff.max():.3e}, mean-abs {diff.mean():.3e}"
    return float(diff.max()), float(diff.mean())


def subcase(case: DecodeCase, b: int, kv: int) -> DecodeCase:
    """The (sequence b, KV head kv) sub-problem of a device-resident instance,
    copied to the CPU: only its own pages (renumbered 0..nb-1), its query heads."""
    s = case.spec
    L = case.lens_host[b]
    nb = math.ceil(L / s.block_size)
    tbl = case.block_tables[b, :nb].long()
    rep = s.rep

    def pick(plane):
        return None if plane is None else plane[tbl][:, kv:kv + 1].contiguous().cpu()

    sub_spec = DecodeSpec(name=s.name + f"_b{b}_kv{kv}", num_seqs=1, num_q_heads=rep, num_kv_heads=1,
                          head_dim=s.head_dim, n_query=s.n_query, block_size=s.block_size, bits=s.bits,
                          group_size=s.group_size, lengths=(L,), window=s.window, v_head_dim=s.v_head_dim)
    return DecodeCase(
        spec=sub_spec, q=case.q[b:b + 1, kv * rep:(kv + 1) * rep].contiguous().cpu(),
        k_pool=pick(case.k_pool), v_pool=pick(case.v_pool),
        block_tables=torch.arange(nb, dtype=torch.int32)[None], seq_lens=torch.tensor([L], dtype=torch.int32),
        scale=case.scale, num_blocks=nb, k_scales=pick(case.k_scales), k_biases=pick(case.k_biases),
        v_scales=pick(case.v_scales), v_biases=pick(case.v_biases), lens_host=[L],
        tables_host=[list(range(nb))])
