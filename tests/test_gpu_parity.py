"""GPU parity: the CUDA path through the C ABI against the float64 CPU oracle.

Tolerance (bf16 outputs vs the oracle): max-abs <= 1e-2 and mean-abs <= 1e-3.
Gathers and layout changes are checked bit for bit.
"""

import math
import zlib

import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, oracle_out, run_gpu, subcase
from quantized_kv_decode_partial_gb300 import PkvError, paged_decode_attention, paged_gather
from quantized_kv_decode_partial_gb300 import binding as B
from quantized_kv_decode_partial_gb300.workloads import WORKLOADS, DecodeSpec, make_case

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def spec(name, **kw):
    base = dict(name=name, num_seqs=3, num_q_heads=8, num_kv_heads=2, head_dim=128, n_query=1, block_size=16,
                bits=16, length_range=(1, 300), pool_factor=2.0, seed=zlib.crc32(name.encode()) % 10000)
    base.update(kw)
    return DecodeSpec(**base)


# Every kernel instantiation, ragged lengths (1 row up to several partitions and
# a ragged tail), GQA factors 1..32, n_query 1..4, page sizes 16..128.
SMALL = [
    (spec("bf16_d128_nq4"), [-1, 16, 48, 0]),
    (spec("bf16_d128_nq16_n2", num_q_heads=16, n_query=2, block_size=32, length_range=(2, 500)), [-1, 64, 0]),
    (spec("bf16_d64_nq32", num_q_heads=32, num_kv_heads=1, head_dim=64, lengths=(1, 17, 33, 250),
          length_range=None, num_seqs=4), [-1, 32]),
    (spec("bf16_d64_rep1_n3", num_q_heads=4, num_kv_heads=4, head_dim=64, n_query=3, block_size=64,
          length_range=(3, 400)), [-1, 80]),
    (spec("bf16_d64_nq16", num_q_heads=8, num_kv_heads=1, head_dim=64, n_query=2, block_size=16), [-1, 64]),
    (spec("bf16_d256_nq8_n2", head_dim=256, n_query=2, length_range=(2, 400)), [-1, 64, 0]),
    (spec("u4_d256_nq4", head_dim=256, bits=4, block_size=32, length_range=(1, 600)), [-1, 32, 64, 0]),
    (spec("u4_d128_nq16_n2", num_q_heads=16, head_dim=128, bits=4, n_query=2, block_size=64,
          length_range=(2, 500)), [-1, 96]),
    (spec("u4_d128_nq4", head_dim=128, bits=4, block_size=32), [-1, 64]),
    (spec("u8_d256_nq4", head_dim=256, bits=8, block_size=32, length_range=(1, 600)), [-1, 32, 0]),
    (spec("u8_d128_nq16_n2", num_q_heads=8, num_kv_heads=1, head_dim=128, bits=8, n_query=2, block_size=32,
          length_range=(2, 500)), [-1, 64]),
    (spec("u8_d128_nq4", head_dim=128, bits=8, block_size=64), [-1, 128]),
    (spec("u4_d256_nq8_n4", num_q_heads=4, num_kv_heads=2, head_dim=256, bits=4, n_query=4, block_size=32,
          length_range=(4, 300)), [-1, 32]),
    # more query rows per KV head than one warp holds: warps share chunks, each with its own rows
    (spec("bf16_d128_nq32", num_q_heads=32, num_kv_heads=1, length_range=(1, 400)), [-1, 48, 0]),
    (spec("bf16_d128_nq64_n4", num_q_heads=16, num_kv_heads=1, n_query=4, length_range=(4, 400)), [-1, 64]),
    (spec("bf16_d64_nq64_n2", num_q_heads=64, num_kv_heads=2, head_dim=64, n_query=2, length_range=(2, 300)), [-1, 32]),
    (spec("bf16_d256_nq32_n4", num_q_heads=8, num_kv_heads=1, head_dim=256, n_query=4, length_range=(4, 300)), [-1, 64]),
    (spec("bf16_d256_nq16", num_q_heads=16, num_kv_heads=1, head_dim=256, length_range=(1, 300)), [-1, 48]),
    (spec("u4_d256_nq16", num_q_heads=16, num_kv_heads=1, head_dim=256, bits=4, block_size=32,
          length_range=(1, 400)), [-1, 64]),
    (spec("u4_d128_nq64_n2", num_q_heads=32, num_kv_heads=1, head_dim=128, bits=4, n_query=2, block_size=32,
          length_range=(2, 400)), [-1, 96]),
    (spec("u8_d256_nq32_n2", num_q_heads=16, num_kv_heads=1, head_dim=256, bits=8, n_query=2, block_size=32,
          length_range=(2, 400)), [-1, 64]),
    (spec("u8_d128_nq32", num_q_heads=32, num_kv_heads=1, head_dim=128, bits=8, block_size=32,
          length_range=(1, 400)), [-1, 32]),
    # 4-bit pages with at most 4 query rows: the paired-value-group form (query columns 4-7
    # repeat rows 0-3), with causal tails of 2 and 3 new rows and a padding column
    (spec("u4_pv_rep2_n2", num_q_heads=4, num_kv_heads=2, head_dim=256, bits=4, n_query=2, block_size=32,
          length_range=(2, 500)), [-1, 32, 0]),
    (spec("u4_pv_rep1_n3", num_q_heads=2, num_kv_heads=2, head_dim=128, bits=4, n_query=3, block_size=32,
          length_range=(3, 500)), [-1, 64]),
    (spec("u4_pv_nq1", num_q_heads=2, num_kv_heads=2, head_dim=256, bits=4, block_size=64,
          length_range=(1, 500)), [-1, 96]),
    (spec("u4_pv_nq2_d128", num_q_heads=4, num_kv_heads=2, head_dim=128, bits=4, block_size=32,
          length_range=(1, 400)), [-1, 32]),
    # key and value head dims that differ (the pages' vHeadDim)
    (spec("bf16_dk192_dv128_nq4", head_dim=192, v_head_dim=128), [-1, 32, 0]),
    (spec("bf16_dk192_dv128_nq16_n2", num_q_heads=16, head_dim=192, v_head_dim=128, n_query=2,
          length_range=(2, 400)), [-1, 64]),
    (spec("bf16_dk192_dv128_nq32", num_q_heads=32, num_kv_heads=1, head_dim=192, v_head_dim=128,
          length_range=(1, 400)), [-1, 48]),
    (spec("bf16_dk256_dv128", head_dim=256, v_head_dim=128, length_range=(1, 400)), [-1, 64]),
    (spec("bf16_dk128_dv256_n2", num_q_heads=4, head_dim=128, v_head_dim=256, n_query=2,
          length_range=(2, 400)), [-1, 64]),
    (spec("u4_dk256_dv128", head_dim=256, v_head_dim=128, bits=4, block_size=32, length_range=(1, 500)), [-1, 64]),
    (spec("u4_dk128_dv256", head_dim=128, v_head_dim=256, bits=4, block_size=32, length_range=(1, 500)), [-1, 96]),
    (spec("u8_dk256_dv128", head_dim=256, v_head_dim=128, bits=8, block_size=32, length_range=(1, 500)), [-1, 32]),
    (spec("u8_dk128_dv256_n2", num_q_heads=4, head_dim=128, v_head_dim=256, bits=8, n_query=2, block_size=32,
          length_range=(2, 500)), [-1, 64]),
    # 33..64 query rows per KV head at 256-dim heads: one query group of 8 warps
    (spec("bf16_d256_nq64_n2", num_q_heads=32, num_kv_heads=1, head_dim=256, n_query=2, length_range=(2, 300)),
     [-1, 48, 0]),
    (spec("bf16_d256_nq40", num_q_heads=40, num_kv_heads=1, head_dim=256, length_range=(1, 300)), [-1, 64]),
    (spec("u4_d256_nq64", num_q_heads=64, num_kv_heads=1, head_dim=256, bits=4, block_size=32,
          length_range=(1, 400)), [-1, 64, 0]),
    (spec("u8_d256_nq48_n4", num_q_heads=12, num_kv_heads=1, head_dim=256, bits=8, n_query=4, block_size=32,
          length_range=(4, 400)), [-1, 32]),
    # key/value head dims that differ, with more than 8 query rows per KV head
    (spec("bf16_dk256_dv128_nq16", num_q_heads=16, num_kv_heads=1, head_dim=256, v_head_dim=128,
          length_range=(1, 400)), [-1, 64]),
    (spec("bf16_dk128_dv256_nq32_n2", num_q_heads=16, num_kv_heads=1, head_dim=128, v_head_dim=256, n_query=2,
          length_range=(2, 400)), [-1, 48]),
    (spec("bf16_dk192_dv128_nq64", num_q_heads=64, num_kv_heads=1, head_dim=192, v_head_dim=128,
          length_range=(1, 300)), [-1, 32]),
    (spec("bf16_dk256_dv128_nq64_n4", num_q_heads=16, num_kv_heads=1, head_dim=256, v_head_dim=128, n_query=4,
          length_range=(4, 300)), [-1, 64]),
    (spec("u4_dk256_dv128_nq32", num_q_heads=32, num_kv_heads=1, head_dim=256, v_head_dim=128, bits=4,
          block_size=32, length_range=(1, 500)), [-1, 64]),
    (spec("u4_dk128_dv256_nq64", num_q_heads=64, num_kv_heads=1, head_dim=128, v_head_dim=256, bits=4,
          block_size=32, length_range=(1, 400)), [-1, 96]),
    (spec("u8_dk256_dv128_nq24_n3", num_q_heads=8, num_kv_heads=1, head_dim=256, v_head_dim=128, bits=8, n_query=3,
          block_size=32, length_range=(3, 500)), [-1, 32]),
    (spec("u8_dk128_dv256_nq64", num_q_heads=64, num_kv_heads=1, head_dim=128, v_head_dim=256, bits=8,
          block_size=32, length_range=(1, 400)), [-1, 64]),
]


@pytest.mark.parametrize("sp,parts", SMALL, ids=[s.name for s, _ in SMALL])
def test_small_cases_match_oracle(sp, parts):
    case = make_case(sp)
    ref = oracle_out(case)
    dcase = case.to(DEV)
    for pt in parts:
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        ptok = (max(case.lens_host) + 64) if pt == -1 else pt
        out = run_gpu(dcase, partition_tokens=ptok, error_flag=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(out.double().cpu().numpy(), ref, f"{sp.name} partition={pt}")


# The small cases above launch at most one CTA per SM for up to 8 query rows per KV head,
# which takes the eight-warp variant (seven for bf16 D=256); these grids of more than one
# CTA per SM take the four-warp one for the same shapes (seven warps for bf16 D=256, whose
# CTAs hold their SM alone).
BIG_GRID = [(16, 64, 0), (16, 128, 0), (16, 256, 0), (4, 128, 0), (4, 256, 0), (8, 128, 0), (8, 256, 0),
            (16, 192, 128), (16, 256, 128), (4, 128, 256)]


# bf16 D=256 CTAs hold their SM alone (16 KB stages) and take 7, 6 or 8 warps for query
# groups of one, two or four warps: several waves of them through the workspace, the
# balanced schedule, and blocks smaller than a chunk.
LONE = [(8, 1), (8, 2), (16, 2)]  # (query heads per KV head, query rows): 8, 16 and 32 rows


@pytest.mark.parametrize("rep,n_query", LONE, ids=[f"rows{r * n}" for r, n in LONE])
@pytest.mark.parametrize("block_size", [16, 8])
def test_lone_bf16_d256_ctas_on_grids_of_several_waves(rep, n_query, block_size):
    sp = spec(f"lone_d256_{rep}_{n_query}_{block_size}", num_seqs=40, num_q_heads=rep, num_kv_heads=1, head_dim=256,
              n_query=n_query, block_size=block_size, length_range=(n_query, 2000))
    case = make_case(sp)
    ref = oracle_out(case)
    d = case.to(DEV)
    plan = B.make_plan(B.layout_for(d.k_pool, 256, 16), B.DecodeParams(sp.num_seqs, rep, n_query,
                                                                      d.block_tables.shape[1], 64, 0))
    assert plan.threads_per_cta == {1: 224, 2: 192, 4: 256}[rep * n_query // 8] and plan.workspace_bytes > 0
    for pt, schedule in ((64, 0), (0, B.PKV_SCHEDULE_BALANCED)):
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        out = run_gpu(d, partition_tokens=pt, error_flag=err, schedule=schedule)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(out.double().cpu().numpy(), ref, f"{sp.name} partition={pt} schedule={schedule}")


@pytest.mark.parametrize("bits,D,DV", BIG_GRID, ids=[f"b{b}_d{d}_{v}" for b, d, v in BIG_GRID])
def test_grids_of_several_ctas_per_sm_match_oracle(bits, D, DV):
    sp = spec(f"big_grid_{bits}_{D}_{DV}", num_seqs=44, num_q_heads=16, num_kv_heads=4, head_dim=D, v_head_dim=DV,
              bits=bits, block_size=16 if bits == 16 else 32, length_range=(1, 260))
    case = make_case(sp)
    ref = oracle_out(case)
    dcase = case.to(DEV)
    for pt in (max(case.lens_host) + 64, 32):
        plan = B.make_plan(B.layout_for(case.k_pool, D, bits, v_pool=case.v_pool),
                           B.DecodeParams(sp.num_seqs, 16, 1, case.block_tables.shape[1], pt))
        # bf16 D=256 CTAs hold their SM alone anyway (16 KB stages) and take seven warps
        assert plan.threads_per_cta == (224 if (bits, D, DV or D) == (16, 256, 256) else 128)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        out = run_gpu(dcase, partition_tokens=pt, error_flag=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(out.double().cpu().numpy(), ref, f"{sp.name} partition={pt}")


@pytest.mark.parametrize("bits,parts,head_dim,rep", [(16, 16, 128, 4), (4, 16, 256, 4), (8, 2, 128, 4),
                                                      (16, 9, 128, 4), (16, 12, 256, 4), (16, 5, 64, 4),
                                                      (16, 8, 256, 64), (4, 6, 256, 48)])
def test_cluster_merge_matches_oracle(bits, parts, head_dim, rep):
    # one sequence: the partitions of each KV head merge inside a thread-block cluster (CTAs alone on
    # their SMs: 8 warps, or 7 for bf16 D=256; 8 warps in one query group for 33..64 rows)
    sp = spec(f"cluster_{bits}_{parts}_{head_dim}_{rep}", num_seqs=1, head_dim=head_dim, bits=bits, block_size=32,
              lengths=(parts * 64 - 5,), length_range=None, num_q_heads=2 * rep)
    case = make_case(sp)
    plan = B.make_plan(B.layout_for(case.k_pool, sp.head_dim, bits),
                       B.DecodeParams(1, sp.num_q_heads, 1, case.block_tables.shape[1], 64))
    assert plan.merge_in_cluster == 1 and plan.max_partitions == parts
    out = run_gpu(case.to(DEV), partition_tokens=64)
    assert_close(out.double().cpu().numpy(), oracle_out(case), f"cluster {bits} {parts} {head_dim}")


# Affine pages on grids of several waves of two CTAs per SM, with 1..8 query rows, windows
# and partitions of one or a few chunks.
MANY_CTAS = [
    (spec("many_u4_d256_nq4", num_seqs=120, head_dim=256, bits=4, block_size=32, length_range=(1, 700)), [32, 96]),
    (spec("many_u4_d128_nq8_n2", num_seqs=120, num_q_heads=8, head_dim=128, bits=4, n_query=2, block_size=32,
          length_range=(2, 600)), [32, 64]),
    (spec("many_u8_d256_nq1", num_seqs=120, num_q_heads=2, head_dim=256, bits=8, block_size=32,
          length_range=(1, 700)), [32, 64]),
    (spec("many_u8_d128_nq4_n4", num_seqs=160, num_q_heads=2, num_kv_heads=2, head_dim=128, bits=8, n_query=4,
          block_size=64, length_range=(4, 500)), [32]),
    (spec("many_u4_window", num_seqs=120, head_dim=256, bits=4, block_size=32, length_range=(50, 900), window=300),
     [32, 64]),
]


@pytest.mark.parametrize("sp,parts", MANY_CTAS, ids=[s.name for s, _ in MANY_CTAS])
def test_affine_grids_of_several_waves_match_oracle(sp, parts):
    case = make_case(sp)
    ref = oracle_out(case)
    dcase = case.to(DEV)
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    for pt in parts:
        plan = B.make_plan(B.layout_for(case.k_pool, sp.head_dim, sp.bits),
                           B.DecodeParams(sp.num_seqs, sp.num_q_heads, sp.n_query, case.block_tables.shape[1], pt,
                                          sp.window))
        assert sp.num_seqs * sp.num_kv_heads * plan.max_partitions > 2 * sms and plan.threads_per_cta == 128
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        out = run_gpu(dcase, partition_tokens=pt, error_flag=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        # 8-bit outputs reach |40|, where a bf16 output's own rounding passes 1e-2
        assert_close(out.double().cpu().numpy(), ref, f"{sp.name} partition={pt}", strict=sp.bits != 8)


def test_affine_grid_of_several_waves_flags_a_bad_block():
    sp = spec("many_badblock", num_seqs=120, head_dim=256, bits=4, block_size=32, length_range=(100, 300))
    case = make_case(sp).to(DEV)
    good = run_gpu(case, partition_tokens=32)
    tb = case.block_tables.clone()
    tb[7, 2] = case.num_blocks + 3
    case.block_tables = tb
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_gpu(case, partition_tokens=32, error_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & B.PKV_DEVERR_BAD_BLOCK
    keep = [i for i in range(sp.num_seqs) if i != 7]
    assert torch.equal(out[keep].view(torch.int16), good[keep].view(torch.int16))


WINDOWED = [
    (spec("win_bf16_n1", length_range=(20, 900), window=100), [-1, 64, 0]),
    (spec("win_bf16_n4", num_q_heads=4, num_kv_heads=1, n_query=4, length_range=(4, 700), window=37), [-1, 32, 96]),
    (spec("win_u4", head_dim=256, bits=4, block_size=32, length_range=(50, 900), window=300), [-1, 64, 0]),
    (spec("win_u4_pv_n2", num_q_heads=2, num_kv_heads=1, head_dim=256, bits=4, n_query=2, block_size=32,
          length_range=(20, 700), window=90), [-1, 32]),
    (spec("win_u8_n2", head_dim=128, bits=8, block_size=32, n_query=2, length_range=(2, 600), window=1), [-1, 96]),
    (spec("win_bf16_one_seq", num_seqs=1, lengths=(2000,), length_range=None, window=700), [128, 256]),
]


@pytest.mark.parametrize("sp,parts", WINDOWED, ids=[s.name for s, _ in WINDOWED])
def test_sliding_window_matches_oracle(sp, parts):
    case = make_case(sp)
    ref = oracle_out(case)
    dcase = case.to(DEV)
    for pt in parts:
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        ptok = (max(case.lens_host) + 64) if pt == -1 else pt
        out = run_gpu(dcase, partition_tokens=ptok, error_flag=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(out.double().cpu().numpy(), ref, f"{sp.name} partition={pt}")


def test_partitioned_oracle_agrees_with_gpu_partitions():
    sp = spec("u4_partitions", head_dim=256, bits=4, block_size=32, num_seqs=2, length_range=(300, 700))
    case = make_case(sp)
    for pt in (32, 96):
        ref = oracle_out(case, partition_tokens=pt)
        out = run_gpu(case.to(DEV), partition_tokens=pt)
        assert_close(out.double().cpu().numpy(), ref, f"partition {pt}")


# ---------------------------------------------------------------------------
# the measured workloads at full size: sampled (sequence, KV head) sub-problems
# ---------------------------------------------------------------------------

FULL = ["bf16_1x1024_hq2_d256", "affine4_g64_1x8192_hq16_d256", "bf16_batch32_hq32_d128",
        "affine4_batch64_hq32_d256", "affine8_batch64_hq32_d256", "bf16_8x131072_n4_hq32_d128",
        "bf16_8x131072_n4_w8192_hq32_d128", "bf16_batch32_hq32_dk192_dv128"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workloads_sampled(name):
    sp = WORKLOADS[name]
    case = make_case(sp, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_gpu(case, error_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.isfinite(out.float()).all()
    rng = np.random.default_rng(99)
    picks = {(0, 0), (sp.num_seqs - 1, sp.num_kv_heads - 1)}
    while len(picks) < min(4, sp.num_seqs * sp.num_kv_heads):
        picks.add((int(rng.integers(sp.num_seqs)), int(rng.integers(sp.num_kv_heads))))
    for b, kv in sorted(picks):
        sub = subcase(case, b, kv)
        ref = oracle_out(sub)
        got = out[b:b + 1, kv * sp.rep:(kv + 1) * sp.rep].double().cpu().numpy()
        # bf16 and 4-bit outputs stay below 2 in magnitude here, where the plain bound
        # needs no allowance for the output's own rounding; 8-bit outputs reach 40
        assert_close(got, ref, f"{name} b={b} kv={kv}", strict=sp.bits != 8)


# ---------------------------------------------------------------------------
# bit-exact properties
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("bits", [16, 4])
def test_gather_is_bit_exact(bits):
    sp = spec(f"gather_{bits}", head_dim=128, bits=bits, block_size=32, length_range=(1, 200))
    case = make_case(sp)
    d = case.to(DEV)
    max_len = max(case.lens_host) + 7
    planes = [("k", case.k_pool, d.k_pool), ("v", case.v_pool, d.v_pool)]
    if bits != 16:
        planes += [("ks", case.k_scales, d.k_scales), ("vb", case.v_biases, d.v_biases)]
    for name, host, dev in planes:
        got = paged_gather(dev, d.block_tables, d.seq_lens, max_len).cpu()
        raw = host.view(torch.int16) if host.dtype == torch.bfloat16 else host
        got_raw = got.view(torch.int16) if got.dtype == torch.bfloat16 else got
        for b in range(sp.num_seqs):
            L = case.lens_host[b]
            ref = oracle.gather_pages(raw.numpy(), case.tables_host[b], L)
            assert np.array_equal(got_raw[b, :, :L].numpy(), ref), name
            assert not got_raw[b, :, L:].any(), name  # untouched rows stay zero


@pytest.mark.parametrize("bits", [16, 8])
def test_physical_block_permutation_is_bitwise_invariant(bits):
    sp = spec(f"perm_{bits}", head_dim=128 if bits == 16 else 256, bits=bits, block_size=32,
              length_range=(50, 600))
    case = make_case(sp)
    base = run_gpu(case.to(DEV), partition_tokens=64)
    g = torch.Generator().manual_seed(3)
    perm = torch.randperm(case.num_blocks, generator=g)
    inv = torch.argsort(perm)
    moved = case.to("cpu")
    for f in ("k_pool", "v_pool", "k_scales", "k_biases", "v_scales", "v_biases"):
        t = getattr(moved, f)
        if t is not None:
            setattr(moved, f, t[inv].contiguous())
    tb = moved.block_tables.clone()
    tb[tb >= 0] = perm[tb[tb >= 0].long()].to(torch.int32)
    moved.block_tables = tb
    out = run_gpu(moved.to(DEV), partition_tokens=64)
    assert torch.equal(out.view(torch.int16), base.view(torch.int16))


def test_cuda_graph_replay_matches_eager():
    sp = spec("graph", head_dim=128, num_q_heads=32, num_kv_heads=8, length_range=(100, 3000), num_seqs=4)
    case = make_case(sp, device=DEV)
    eager = run_gpu(case, partition_tokens=256)
    out = torch.empty_like(eager)
    plan = B.make_plan(B.layout_for(case.k_pool, 128, 16), B.DecodeParams(4, 32, 1, case.block_tables.shape[1], 256))
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        paged_decode_attention(case.q, case.k_pool, case.v_pool, case.block_tables, case.seq_lens, case.scale,
                               partition_tokens=256, out=out, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        paged_decode_attention(case.q, case.k_pool, case.v_pool, case.block_tables, case.seq_lens, case.scale,
                               partition_tokens=256, out=out, workspace=ws)
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))


# ---------------------------------------------------------------------------
# invalid inputs: flagged on the device, never a fault
# ---------------------------------------------------------------------------

def test_bad_block_id_is_flagged_and_isolated():
    sp = spec("badblock", num_seqs=3, length_range=(100, 300))
    case = make_case(sp).to(DEV)
    good = run_gpu(case, partition_tokens=64)
    tb = case.block_tables.clone()
    tb[1, 2] = case.num_blocks + 5
    case.block_tables = tb
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_gpu(case, partition_tokens=64, error_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & B.PKV_DEVERR_BAD_BLOCK
    assert torch.isfinite(out.float()).all()
    assert torch.equal(out[[0, 2]].view(torch.int16), good[[0, 2]].view(torch.int16))


@pytest.mark.parametrize("bad_len", ["short", "long"])
def test_bad_seq_len_is_flagged_and_zeroed(bad_len):
    sp = spec("badlen", num_seqs=3, n_query=2, length_range=(100, 300))
    case = make_case(sp).to(DEV)
    for pt in (64, 4096):
        good = run_gpu(case, partition_tokens=pt)
        lens = case.seq_lens.clone()
        lens[1] = 1 if bad_len == "short" else case.block_tables.shape[1] * sp.block_size + 1
        bad = case.to(DEV)
        bad.seq_lens = lens
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        out = run_gpu(bad, partition_tokens=pt, error_flag=err)
        torch.cuda.synchronize()
        assert int(err.item()) & B.PKV_DEVERR_BAD_SEQ_LEN
        assert not out[1].float().any()
        assert torch.equal(out[[0, 2]].view(torch.int16), good[[0, 2]].view(torch.int16))


def test_host_side_errors_return_codes():
    sp = spec("hosterr")
    case = make_case(sp).to(DEV)
    flat = case.k_pool.view(-1)
    shifted = torch.as_strided(flat, (case.k_pool.shape[0] - 1,) + tuple(case.k_pool.shape[1:]),
                               case.k_pool.stride(), storage_offset=1)  # 2 bytes off a 16-byte boundary
    with pytest.raises(PkvError) as e:
        paged_decode_attention(case.q, shifted, case.v_pool, case.block_tables, case.seq_lens, case.scale)
    assert e.value.code == B.PKV_ERR_MISALIGNED
    with pytest.raises(PkvError) as e:
        paged_decode_attention(case.q, case.k_pool, case.v_pool, case.block_tables, case.seq_lens, case.scale,
                               partition_tokens=16, workspace=torch.empty(16, dtype=torch.uint8, device=DEV))
    assert e.value.code == B.PKV_ERR_WORKSPACE_TOO_SMALL


def test_minimum_lengths_and_exact_fill():
    # len == n_query (only the new rows), and len filling every block of the table exactly
    sp = spec("edges", num_seqs=2, n_query=3, num_q_heads=4, num_kv_heads=2, lengths=(3, 64), length_range=None,
              block_size=16)
    case = make_case(sp)
    ref = oracle_out(case)
    for pt in (16, 4096):
        out = run_gpu(case.to(DEV), partition_tokens=pt)
        assert_close(out.double().cpu().numpy(), ref, f"edges pt={pt}")


def test_host_driven_step_matches_device_entry():
    # pkv_paged_decode_attention_host: one packed input copy, decode, output copy, on one stream
    from quantized_kv_decode_partial_gb300 import HostDecodeStep
    sp = spec("host_io", head_dim=256, bits=4, block_size=32, length_range=(1, 600))
    case = make_case(sp)
    d = case.to(DEV)
    ref = run_gpu(d, partition_tokens=64)
    stream = torch.cuda.Stream(device=DEV)
    kw = dict(bits=4, k_scales=d.k_scales, k_biases=d.k_biases, v_scales=d.v_scales, v_biases=d.v_biases,
              partition_tokens=64, stream=stream)
    step = HostDecodeStep(case.q, case.block_tables, case.seq_lens, d.k_pool, d.v_pool, case.scale, **kw)
    for _ in range(2):
        step.out_host.fill_(float("nan"))
        step()
        stream.synchronize()
        assert torch.equal(step.out_host.view(torch.int16), ref.cpu().view(torch.int16))
    # new per-step values written into the host block reach the device: the second
    # sequence's query rows are zeroed, and only they change (to the mean of their V rows)
    step.host["q"][1].zero_()
    step()
    stream.synchronize()
    d.q[1].zero_()
    ref2 = run_gpu(d, partition_tokens=64)
    assert torch.equal(step.out_host.view(torch.int16), ref2.cpu().view(torch.int16))
    assert not torch.equal(ref2[1], ref[1]) and torch.equal(ref2[0], ref[0])
    # tables left out of the per-step copy stay as first copied
    step2 = HostDecodeStep(case.q, case.block_tables, case.seq_lens, d.k_pool, d.v_pool, case.scale,
                           copy_tables=False, **kw)
    assert step2.in_bytes < step.in_bytes
    step2.host["block_tables"].fill_(-7)  # would be flagged as bad blocks if copied
    step2()
    stream.synchronize()
    assert torch.equal(step2.out_host.view(torch.int16), ref.cpu().view(torch.int16))


def test_back_to_back_host_driven_steps():
    # Host-driven steps of two instances enqueued back to back, with no synchronisation: the
    # second step's kernel may start (and read its host-memory inputs) while the first is still
    # running; each output must still be its own instance's.
    from quantized_kv_decode_partial_gb300 import HostDecodeStep
    stream = torch.cuda.Stream(device=DEV)
    steps, refs = [], []
    for k in range(3):
        sp = spec(f"host_b2b_{k}", head_dim=256, bits=4, block_size=32, length_range=(200, 600))
        case = make_case(sp)
        d = case.to(DEV)
        refs.append(run_gpu(d, partition_tokens=64).cpu())
        steps.append(HostDecodeStep(case.q, case.block_tables, case.seq_lens, d.k_pool, d.v_pool, case.scale, bits=4,
                                    k_scales=d.k_scales, k_biases=d.k_biases, v_scales=d.v_scales,
                                    v_biases=d.v_biases, partition_tokens=64, stream=stream))
    torch.cuda.synchronize()
    for _ in range(2):
        for st in steps:
            st.out_host.fill_(float("nan"))
        for st in steps:
            st()
        stream.synchronize()
        for st, ref in zip(steps, refs):
            assert torch.equal(st.out_host.view(torch.int16), ref.view(torch.int16))


def test_back_to_back_host_steps_of_a_windowed_cluster_grid():
    # A window gives every unit the same span, so the plan is one wave of clusters of
    # several CTAs per SM; host-driven steps launch that grid as a programmatic dependent
    # of the previous step. Steps of two instances enqueued back to back with no
    # synchronisation must each equal the device entry bit for bit.
    import ctypes

    from quantized_kv_decode_partial_gb300 import HostDecodeStep
    stream = torch.cuda.Stream(device=DEV)
    steps, refs = [], []
    for k in range(2):
        # 12 sequences: 96 units, too many for a wave of one CTA per SM with two partitions
        sp = spec(f"host_win_{k}", num_seqs=12, num_q_heads=32, num_kv_heads=8, n_query=4, window=4096,
                  lengths=(5000, 4200, 6000, 4100, 5500, 4500, 4800, 5200, 4300, 5900, 4700, 5100), length_range=None)
        case = make_case(sp)
        d = case.to(DEV)
        if k == 0:
            lay = B.layout_for(d.k_pool, 128, 16)
            par = B.DecodeParams(sp.num_seqs, 32, 4, d.block_tables.shape[1], 0, 4096)
            plan = B.Plan()
            assert B.load_library().pkv_plan_for_current_device(ctypes.byref(lay), ctypes.byref(par),
                                                                ctypes.byref(plan)) == 0
            assert plan.merge_in_cluster == 1 and plan.threads_per_cta == 128 and plan.max_partitions >= 2
            b, kv = 2, 5
            ref_sub = oracle_out(subcase(d, b, kv))
        refs.append(run_gpu(d, partition_tokens=0).cpu())
        if k == 0:
            got = refs[0][b, kv * 4:(kv + 1) * 4][None].double().numpy()
            assert_close(got, ref_sub, "windowed cluster grid, one (sequence, KV head)")
        steps.append(HostDecodeStep(case.q, case.block_tables, case.seq_lens, d.k_pool, d.v_pool, case.scale,
                                    window=4096, stream=stream))
    torch.cuda.synchronize()
    for _ in range(3):
        for st in steps:
            st.out_host.fill_(float("nan"))
        for st in steps:
            st()
        stream.synchronize()
        for st, ref in zip(steps, refs):
            assert torch.equal(st.out_host.view(torch.int16), ref.view(torch.int16))


def test_host_driven_fused_step_matches_device_fused_step():
    from quantized_kv_decode_partial_gb300 import HostDecodeStep
    sp = spec("host_fused", num_q_heads=8, num_kv_heads=2, n_query=2, length_range=(3, 300))
    case = make_case(sp, poison=False)
    g = torch.Generator().manual_seed(5)
    k_new = torch.randn((3, 2, 2, 128), generator=g).to(torch.bfloat16)
    v_new = torch.randn((3, 2, 2, 128), generator=g).to(torch.bfloat16)
    a, b = case.to(DEV), case.to(DEV)
    ref = B.paged_decode_append_attention(a.q, k_new.to(DEV), v_new.to(DEV), a.k_pool, a.v_pool, a.block_tables,
                                          a.seq_lens, case.scale, partition_tokens=32)
    stream = torch.cuda.Stream(device=DEV)
    step = HostDecodeStep(case.q, case.block_tables, case.seq_lens, b.k_pool, b.v_pool, case.scale, k_new=k_new,
                          v_new=v_new, partition_tokens=32, stream=stream)
    step()
    stream.synchronize()
    assert torch.equal(step.out_host.view(torch.int16), ref.cpu().view(torch.int16))
    assert torch.equal(a.k_pool.view(torch.int16), b.k_pool.view(torch.int16))
    assert torch.equal(a.v_pool.view(torch.int16), b.v_pool.view(torch.int16))


@pytest.mark.parametrize("bits,D,DV", [(16, 128, 128), (16, 192, 128), (16, 128, 256), (4, 128, 256), (8, 256, 128)])
def test_workspace_writes_stay_inside_the_planned_bytes(bits, D, DV):
    # a grid of more than one wave with several partitions: states go through the workspace
    sp = spec(f"ws_bounds_{bits}_{D}_{DV}", num_seqs=40, num_q_heads=8, num_kv_heads=4, head_dim=D, v_head_dim=DV,
              bits=bits, block_size=16 if bits == 16 else 32, length_range=(100, 400))
    case = make_case(sp)
    d = case.to(DEV)
    pt = 64
    plan = B.make_plan(B.layout_for(d.k_pool, D, bits, v_pool=d.v_pool),
                       B.DecodeParams(sp.num_seqs, sp.num_q_heads, 1, d.block_tables.shape[1], pt))
    assert plan.merge_in_cluster == 0 and plan.max_partitions > 1 and plan.workspace_bytes > 0
    guard = 1 << 16
    buf = torch.full((plan.workspace_bytes + guard,), 0x5A, dtype=torch.uint8, device=DEV)
    ws = buf[:plan.workspace_bytes]
    out = paged_decode_attention(d.q, d.k_pool, d.v_pool, d.block_tables, d.seq_lens, case.scale, bits=bits,
                                 k_scales=d.k_scales, k_biases=d.k_biases, v_scales=d.v_scales, v_biases=d.v_biases,
                                 partition_tokens=pt, workspace=ws)
    torch.cuda.synchronize()
    assert bool((buf[plan.workspace_bytes:] == 0x5A).all()), "write past the planned workspace"
    assert_close(out.double().cpu().numpy(), oracle_out(case), f"{sp.name}")


def merge_groups(dv, parts):
    """Partition groups per output row the merge pass takes: the fewest g (a power of
    two) with 4 g >= the partition count, at most 256 / (dv / 4)."""
    g = 1
    while g < 256 // (dv // 4) and 4 * g < parts:
        g *= 2
    return g


# (bits, key dim, value dim, partitions, groups per merged row): 61 sequences of 9 query
# heads on 3 KV heads give 549 output rows, a ragged last merge CTA for every row packing
# (16, 8, 4, 2 or 1 rows per CTA), and a grid of several waves, so the states go through
# the workspace and the merge kernel.
MERGE_PACK = [(16, 64, 0, 3, 1), (16, 128, 0, 4, 1), (16, 256, 0, 2, 1), (16, 256, 0, 7, 2), (16, 64, 0, 13, 4),
              (16, 192, 128, 6, 2), (4, 256, 0, 4, 1), (8, 128, 0, 20, 8), (16, 64, 0, 40, 16), (4, 128, 256, 9, 4)]


@pytest.mark.parametrize("bits,D,DV,parts,groups", MERGE_PACK,
                         ids=[f"b{b}_d{d}_{v}_p{p}" for b, d, v, p, _ in MERGE_PACK])
def test_merge_packs_rows_and_zeroes_a_bad_length(bits, D, DV, parts, groups):
    pt = 32
    rng = np.random.default_rng(zlib.crc32(f"pack{bits}{D}{DV}{parts}".encode()))
    lens = rng.integers(1, parts * pt + 1, 61)
    lens[7] = parts * pt  # the table is exactly parts partitions wide
    sp = spec(f"merge_pack_{bits}_{D}_{DV}_{parts}", num_seqs=61, num_q_heads=9, num_kv_heads=3, head_dim=D,
              v_head_dim=DV, bits=bits, block_size=16 if bits == 16 else 32, lengths=tuple(int(x) for x in lens),
              length_range=None)
    case = make_case(sp)
    d = case.to(DEV)
    plan = B.make_plan(B.layout_for(d.k_pool, D, bits, v_pool=d.v_pool),
                       B.DecodeParams(sp.num_seqs, sp.num_q_heads, 1, d.block_tables.shape[1], pt))
    assert plan.merge_in_cluster == 0 and plan.max_partitions == parts
    assert merge_groups(DV or D, parts) == groups
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    good = run_gpu(d, partition_tokens=pt, error_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_close(good.double().cpu().numpy(), oracle_out(case), sp.name)
    # a length below n_query in the middle of a packed merge CTA: that sequence's rows
    # are zero, every other row is unchanged bit for bit
    bad = case.to(DEV)
    bad.seq_lens = d.seq_lens.clone()
    bad.seq_lens[30] = 0
    out = run_gpu(bad, partition_tokens=pt, error_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & B.PKV_DEVERR_BAD_SEQ_LEN
    assert not out[30].float().any()
    keep = [i for i in range(sp.num_seqs) if i != 30]
    assert torch.equal(out[keep].view(torch.int16), good[keep].view(torch.int16))


@pytest.mark.parametrize("pinned", [True, False], ids=["mapped_pinned", "pageable"])
def test_one_shot_host_entry_with_pinned_and_pageable_memory(pinned):
    # mapped page-locked memory is copied by the SMs, pageable memory by the copy engine
    import ctypes
    lib = B.load_library()
    sp = spec(f"host_one_shot_{pinned}", length_range=(1, 300))
    case = make_case(sp)
    d = case.to(DEV)
    ref = run_gpu(d, partition_tokens=48)
    qb = case.q.numel() * 2
    blk_host = torch.empty(qb, dtype=torch.uint8)
    blk_host = blk_host.pin_memory() if pinned else blk_host
    blk_host.copy_(case.q.view(torch.uint8).reshape(-1))
    q_dev = torch.zeros_like(d.q)
    out_host = torch.full(ref.shape, float("nan"), dtype=torch.bfloat16)
    out_host = out_host.pin_memory() if pinned else out_host
    out_dev = torch.empty_like(ref)
    layout = B.layout_for(d.k_pool, sp.head_dim, 16, v_pool=d.v_pool)
    params = B.DecodeParams(sp.num_seqs, sp.num_q_heads, 1, d.block_tables.shape[1], 48)
    plan = B.make_plan(layout, params)
    ws = torch.empty(max(1, plan.workspace_bytes), dtype=torch.uint8, device=DEV)
    rc = lib.pkv_paged_decode_attention_host(
        ctypes.byref(layout), ctypes.byref(params), blk_host.data_ptr(), q_dev.data_ptr(), qb, out_host.data_ptr(),
        q_dev.data_ptr(), None, None, d.k_pool.data_ptr(), d.v_pool.data_ptr(), None, None, None, None,
        d.block_tables.data_ptr(), d.seq_lens.data_ptr(), float(case.scale), out_dev.data_ptr(), ws.data_ptr(),
        ws.numel(), None, torch.cuda.current_stream(DEV).cuda_stream)
    assert rc == B.PKV_OK
    torch.cuda.synchronize()
    assert torch.equal(out_host.view(torch.int16), ref.cpu().view(torch.int16))


@pytest.mark.parametrize("bits", [16, 4])
def test_table_entries_past_the_length_are_never_used(bits):
    # The partial pass issues a partition's first chunks before the length is known.
    # Table entries past each sequence's length (here valid block ids of other data, or
    # ids far out of range) must change neither the output nor the error word.
    sp = spec(f"stale_tables_{bits}", num_seqs=4, head_dim=256 if bits == 4 else 128, bits=bits,
              block_size=32 if bits == 4 else 16, length_range=(1, 200))
    case = make_case(sp)
    # leave room past every length: a wider table
    wide = torch.full((sp.num_seqs, case.block_tables.shape[1] + 16), -1, dtype=torch.int32)
    wide[:, :case.block_tables.shape[1]] = case.block_tables
    ref = None
    for fill in ("valid", "out_of_range"):
        tb = wide.clone()
        g = torch.Generator().manual_seed(3)
        for b in range(sp.num_seqs):
            used = -(-case.lens_host[b] // sp.block_size)
            n = tb.shape[1] - used
            tb[b, used:] = (torch.randint(0, case.num_blocks, (n,), generator=g) if fill == "valid"
                            else torch.full((n,), case.num_blocks + 1000, dtype=torch.int64)).to(torch.int32)
        d = case.to(DEV)
        d.block_tables = tb.to(DEV)
        for pt in (16 if bits == 16 else 32, 64, 1 << 12):
            err = torch.zeros(1, dtype=torch.int32, device=DEV)
            out = run_gpu(d, partition_tokens=pt, error_flag=err)
            torch.cuda.synchronize()
            assert int(err.item()) == 0, (fill, pt)
            if ref is None:
                ref = oracle_out(case)
            assert_close(out.double().cpu().numpy(), ref, f"{sp.name} {fill} partition={pt}")
