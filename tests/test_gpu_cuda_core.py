"""GPU parity of the CUDA-core contraction (pkv_decode_params.contraction =
PKV_CONTRACTION_CUDA_CORE): per-lane f32 FMAs and warp-shuffle reductions, the form
of the pages' direct paged kernel, for bf16 pages with at most 4 query rows per KV
head. Checked against the float64 oracle on ragged lengths (1 row up to several
partitions and a ragged tail, NaN-poisoned stale rows), every head dim, 1..4 query
rows, causal tails, windows and every finishing form (one partition, cluster merge,
workspace + merge kernel), and against the tensor-core contraction on the full-size
workloads it serves."""

import zlib

import numpy as np
import pytest
import torch

from helpers import assert_close, oracle_out, subcase
from quantized_kv_decode_partial_gb300 import binding as B
from quantized_kv_decode_partial_gb300 import paged_decode_append_attention, paged_decode_attention
from quantized_kv_decode_partial_gb300.workloads import WORKLOADS, DecodeSpec, make_case

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
CC = B.PKV_CONTRACTION_CUDA_CORE


def spec(name, **kw):
    base = dict(name=name, num_seqs=3, num_q_heads=4, num_kv_heads=2, head_dim=128, n_query=1, block_size=16,
                bits=16, length_range=(1, 300), pool_factor=2.0, seed=zlib.crc32(name.encode()) % 10000)
    base.update(kw)
    return DecodeSpec(**base)


def run(case, partition_tokens, contraction=CC, error_flag=None):
    return paged_decode_attention(case.q, case.k_pool, case.v_pool, case.block_tables, case.seq_lens, case.scale,
                                  partition_tokens=partition_tokens, window=case.spec.window,
                                  error_flag=error_flag, contraction=contraction)


CASES = [
    (spec("cc_d128_nq2"), [-1, 16, 48, 0]),
    (spec("cc_d128_nq4", num_q_heads=8), [-1, 32, 0]),
    (spec("cc_d128_nq1", num_q_heads=2), [-1, 64]),
    (spec("cc_d128_nq3_n3", num_q_heads=2, num_kv_heads=2, n_query=3, length_range=(3, 400)), [-1, 32]),
    (spec("cc_d256_nq2", head_dim=256, length_range=(1, 600)), [-1, 16, 64, 0]),
    (spec("cc_d256_nq4_n2", head_dim=256, n_query=2, length_range=(2, 400)), [-1, 48]),
    (spec("cc_d64_nq4_n4", num_q_heads=2, num_kv_heads=2, head_dim=64, n_query=4, block_size=32,
          length_range=(4, 500)), [-1, 32, 0]),
    (spec("cc_d64_nq2", num_q_heads=4, head_dim=64, block_size=64), [-1, 64]),
    (spec("cc_window", num_q_heads=8, length_range=(20, 900), window=100), [-1, 64, 0]),
    (spec("cc_window_n4", num_q_heads=1, num_kv_heads=1, n_query=4, length_range=(4, 700), window=37), [-1, 32]),
]


@pytest.mark.parametrize("sp,parts", CASES, ids=[s.name for s, _ in CASES])
def test_cuda_core_contraction_matches_oracle(sp, parts):
    case = make_case(sp)
    ref = oracle_out(case)
    d = case.to(DEV)
    for pt in parts:
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        ptok = (max(case.lens_host) + 64) if pt == -1 else pt
        out = run(d, ptok, error_flag=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(out.double().cpu().numpy(), ref, f"{sp.name} partition={pt}", strict=True)


@pytest.mark.parametrize("parts,head_dim", [(16, 128), (9, 256), (4, 64)])
def test_cuda_core_cluster_merge(parts, head_dim):
    sp = spec(f"cc_cluster_{parts}_{head_dim}", num_seqs=1, head_dim=head_dim, block_size=32,
              lengths=(parts * 64 - 5,), length_range=None)
    case = make_case(sp)
    plan = B.make_plan(B.layout_for(case.k_pool, head_dim, 16),
                       B.DecodeParams(1, sp.num_q_heads, 1, case.block_tables.shape[1], 64, 0, CC))
    assert plan.merge_in_cluster == 1 and plan.contraction == CC
    out = run(case.to(DEV), 64)
    assert_close(out.double().cpu().numpy(), oracle_out(case), sp.name, strict=True)


def test_cuda_core_grids_of_several_ctas_per_sm():
    sp = spec("cc_big_grid", num_seqs=60, num_q_heads=16, num_kv_heads=4, length_range=(1, 260))
    case = make_case(sp)
    ref = oracle_out(case)
    d = case.to(DEV)
    for pt in (max(case.lens_host) + 64, 32):
        plan = B.make_plan(B.layout_for(case.k_pool, 128, 16),
                           B.DecodeParams(sp.num_seqs, 16, 1, case.block_tables.shape[1], pt, 0, CC))
        assert plan.threads_per_cta == 128 and plan.contraction == CC
        out = run(d, pt)
        assert_close(out.double().cpu().numpy(), ref, f"{sp.name} partition={pt}", strict=True)


def test_cuda_core_fused_append_matches_append_then_decode():
    sp = spec("cc_fused", num_q_heads=4, num_kv_heads=2, n_query=2, length_range=(3, 300))
    case = make_case(sp, poison=False)
    g = torch.Generator().manual_seed(11)
    k_new = torch.randn((3, 2, 2, 128), generator=g).to(torch.bfloat16).to(DEV)
    v_new = torch.randn((3, 2, 2, 128), generator=g).to(torch.bfloat16).to(DEV)
    a, b = case.to(DEV), case.to(DEV)
    B.paged_append(k_new, v_new, a.block_tables, a.seq_lens - 2, a.k_pool, a.v_pool)
    ref = run(a, 32)
    out = paged_decode_append_attention(b.q, k_new, v_new, b.k_pool, b.v_pool, b.block_tables, b.seq_lens,
                                        case.scale, partition_tokens=32, contraction=CC)
    torch.cuda.synchronize()
    assert torch.equal(a.k_pool.view(torch.int16), b.k_pool.view(torch.int16))
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("name", ["bf16_1x1024_hq2_d256", "bf16_batch32_hq32_d128"])
def test_cuda_core_full_size_workloads(name):
    sp = WORKLOADS[name]
    case = make_case(sp, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run(case, case.partition_tokens, error_flag=err)
    tensor = run(case, case.partition_tokens, contraction=B.PKV_CONTRACTION_TENSOR)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rng = np.random.default_rng(5)
    picks = {(0, 0), (sp.num_seqs - 1, sp.num_kv_heads - 1)}
    while len(picks) < min(4, sp.num_seqs * sp.num_kv_heads):
        picks.add((int(rng.integers(sp.num_seqs)), int(rng.integers(sp.num_kv_heads))))
    for b, kv in sorted(picks):
        ref = oracle_out(subcase(case, b, kv))
        assert_close(out[b:b + 1, kv * sp.rep:(kv + 1) * sp.rep].double().cpu().numpy(), ref,
                     f"{name} cuda cores b={b} kv={kv}", strict=True)
    # the two contractions agree within the bound on the whole output
    diff = (out.double() - tensor.double()).abs()
    assert float(diff.max()) <= 1e-2 and float(diff.mean()) <= 1e-3
