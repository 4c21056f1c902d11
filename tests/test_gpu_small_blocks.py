"""Blocks smaller than a chunk, against the float64 oracle.

The partial kernel stages 16 rows (bf16 pages) or 32 / 16 rows (affine pages) per
chunk. With blocks of 8 or 16 rows a chunk spans 2 or 4 blocks: it is copied block
by block (one TMA copy per block piece and 128-byte segment, plus the scale/bias rows
of each piece), each piece landing at its place in the chunk, by instantiations of
the grids of several CTAs per SM made for such pools. These cases run every finishing
form (one partition, cluster merge, workspace merge), windows, several query rows and
bad block ids on such pools; a request for the balanced schedule runs partitions, and
the CUDA-core contraction and the fused append-and-attend call (which writes a
chunk's new rows into one block) are refused.
"""

import ctypes
import zlib

import pytest
import torch

from helpers import assert_close, oracle_out, run_gpu
from quantized_kv_decode_partial_gb300 import PkvError, paged_decode_append_attention, paged_decode_attention
from quantized_kv_decode_partial_gb300 import binding as B
from quantized_kv_decode_partial_gb300.workloads import DecodeSpec, make_case

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def spec(name, **kw):
    base = dict(name=name, num_seqs=3, num_q_heads=8, num_kv_heads=2, head_dim=128, n_query=1, block_size=8,
                bits=16, length_range=(1, 400), pool_factor=2.0, seed=zlib.crc32(name.encode()) % 10000)
    base.update(kw)
    return DecodeSpec(**base)


# (spec, partition sizes: -1 one partition, 0 the library's plan, else rows)
CASES = [
    (spec("sb_bf16_d128_bs8"), [-1, 16, 48, 0]),
    (spec("sb_bf16_d64_bs8_nq32", num_q_heads=32, num_kv_heads=1, head_dim=64), [-1, 32]),
    (spec("sb_bf16_d256_bs8_n2", head_dim=256, n_query=2, length_range=(2, 400)), [-1, 64, 0]),
    (spec("sb_bf16_d128_bs8_nq64_n4", num_q_heads=16, num_kv_heads=1, n_query=4, length_range=(4, 300)), [-1, 48]),
    (spec("sb_bf16_dk192_dv128_bs8", head_dim=192, v_head_dim=128), [-1, 32]),
    (spec("sb_u4_d256_bs16", head_dim=256, bits=4, block_size=16, length_range=(1, 600)), [-1, 32, 64, 0]),
    (spec("sb_u4_d256_bs8_nq2", num_q_heads=4, head_dim=256, bits=4, length_range=(1, 600)), [-1, 64]),
    (spec("sb_u4_d128_bs8_nq16_n2", num_q_heads=16, head_dim=128, bits=4, n_query=2, length_range=(2, 500)),
     [-1, 96]),
    (spec("sb_u4_d256_bs16_nq64", num_q_heads=64, num_kv_heads=1, head_dim=256, bits=4, block_size=16,
          length_range=(1, 300)), [-1, 64]),
    (spec("sb_u8_d128_bs8", bits=8, length_range=(1, 500)), [-1, 32]),
    (spec("sb_u8_d256_bs8_n2", head_dim=256, bits=8, n_query=2, length_range=(2, 500)), [-1, 64]),
    (spec("sb_u8_d256_bs16", head_dim=256, bits=8, block_size=16, length_range=(1, 500)), [-1, 32]),
    (spec("sb_u4_dk256_dv128_bs16", head_dim=256, v_head_dim=128, bits=4, block_size=16, length_range=(1, 500)),
     [-1, 64]),
    (spec("sb_win_bf16_bs8_n2", n_query=2, window=50, length_range=(2, 400)), [-1, 32, 0]),
    (spec("sb_win_u4_bs16", num_q_heads=4, head_dim=256, bits=4, block_size=16, window=100,
          length_range=(1, 600)), [-1, 64]),
]


@pytest.mark.parametrize("sp,parts", CASES, ids=[s.name for s, _ in CASES])
def test_blocks_smaller_than_a_chunk_match_oracle(sp, parts):
    case = make_case(sp)
    ref = oracle_out(case)
    d = case.to(DEV)
    for pt in parts:
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        ptok = (max(case.lens_host) + 64) if pt == -1 else pt
        out = run_gpu(d, partition_tokens=ptok, error_flag=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(out.double().cpu().numpy(), ref, f"{sp.name} partition={pt}")


@pytest.mark.parametrize("bits,D", [(16, 128), (4, 256), (8, 128)])
def test_grids_of_many_ctas_on_small_blocks(bits, D):
    # several waves of partitions through the workspace, fixed and the library's (asked for
    # the balanced schedule, which such pools do not take)
    sp = spec(f"sb_many_{bits}_{D}", num_seqs=40, num_q_heads=16, num_kv_heads=4, head_dim=D, bits=bits,
              block_size=8 if bits == 16 else 16, length_range=(1, 2000))
    case = make_case(sp)
    ref = oracle_out(case)
    d = case.to(DEV)
    kw = dict(bits=bits, k_scales=d.k_scales, k_biases=d.k_biases, v_scales=d.v_scales, v_biases=d.v_biases)
    asked = B.make_plan(B.layout_for(d.k_pool, D, bits),
                        B.DecodeParams(sp.num_seqs, 16, 1, d.block_tables.shape[1], 0, 0, 0, B.PKV_SCHEDULE_BALANCED))
    assert asked.balanced == 0 and asked.workspace_bytes > 0
    for partition, schedule in ((64, 0), (0, B.PKV_SCHEDULE_BALANCED)):
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        out = paged_decode_attention(d.q, d.k_pool, d.v_pool, d.block_tables, d.seq_lens, case.scale,
                                     partition_tokens=partition, schedule=schedule, error_flag=err, **kw)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(out.double().cpu().numpy(), ref, f"{sp.name} partition={partition} schedule={schedule}")


def test_single_cta_grids_take_the_several_per_sm_instantiation_on_small_blocks():
    # one sequence: a grid of at most one CTA per SM, which on such pools runs the
    # instantiation for several CTAs per SM (the CUDA-core contraction is refused)
    sp = spec("sb_one_seq_u4", num_seqs=1, num_q_heads=16, num_kv_heads=4, head_dim=256, bits=4, block_size=16,
              lengths=(3000,), length_range=None)
    case = make_case(sp)
    d = case.to(DEV)
    plan = B.make_plan(B.layout_for(d.k_pool, 256, 4), B.DecodeParams(1, 16, 1, d.block_tables.shape[1], 512, 0))
    assert plan.threads_per_cta == 128 and plan.merge_in_cluster == 1
    assert_close(run_gpu(d, partition_tokens=512).double().cpu().numpy(), oracle_out(case), sp.name)
    bf16 = B.PoolLayout(1000, 4, 8, 128, 16, 64)
    refused = B.Plan()
    par = B.DecodeParams(1, 4, 1, 64, 0, 0, B.PKV_CONTRACTION_CUDA_CORE)
    assert B.load_library().pkv_make_plan(ctypes.byref(bf16), ctypes.byref(par), 152, ctypes.byref(refused)) == \
        B.PKV_ERR_UNSUPPORTED_SHAPE


def test_bad_block_in_a_chunk_of_small_blocks_is_flagged_and_isolated():
    sp = spec("sb_badblock", head_dim=256, bits=4, block_size=8, length_range=(200, 400))
    d = make_case(sp).to(DEV)
    kw = dict(partition_tokens=64)
    good = run_gpu(d, **kw)
    tb = d.block_tables.clone()
    tb[1, 5] = d.num_blocks + 3  # the second piece of a chunk of the second sequence
    d.block_tables = tb
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_gpu(d, error_flag=err, **kw)
    torch.cuda.synchronize()
    assert int(err.item()) & B.PKV_DEVERR_BAD_BLOCK
    assert torch.isfinite(out.float()).all()
    assert torch.equal(out[[0, 2]].view(torch.int16), good[[0, 2]].view(torch.int16))


def test_fused_call_refuses_blocks_smaller_than_a_chunk():
    sp = spec("sb_fused", length_range=(20, 100))
    d = make_case(sp).to(DEV)
    k_new = torch.zeros((sp.num_seqs, sp.num_kv_heads, 1, sp.head_dim), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(PkvError) as e:
        paged_decode_append_attention(d.q, k_new, k_new, d.k_pool, d.v_pool, d.block_tables, d.seq_lens, d.scale,
                                      partition_tokens=64)
    assert e.value.code == B.PKV_ERR_UNSUPPORTED_SHAPE


def test_host_driven_step_and_two_passes_on_small_blocks():
    # the host-driven step (inputs read from pinned host memory) and the two-pass entry
    # points run the same instantiation as the one-call entry, bit for bit
    from quantized_kv_decode_partial_gb300 import HostDecodeStep, paged_decode_passes
    sp = spec("sb_host", num_seqs=12, num_q_heads=16, num_kv_heads=4, head_dim=256, bits=4, block_size=16,
              length_range=(1, 1500))
    case = make_case(sp)
    d = case.to(DEV)
    kw = dict(bits=4, k_scales=d.k_scales, k_biases=d.k_biases, v_scales=d.v_scales, v_biases=d.v_biases,
              partition_tokens=64)
    ref = paged_decode_attention(d.q, d.k_pool, d.v_pool, d.block_tables, d.seq_lens, case.scale, **kw)
    torch.cuda.synchronize()
    assert_close(ref.double().cpu().numpy(), oracle_out(case), sp.name)
    stream = torch.cuda.Stream(device=DEV)
    step = HostDecodeStep(case.q, case.block_tables, case.seq_lens, d.k_pool, d.v_pool, case.scale, stream=stream,
                          **kw)
    step()
    stream.synchronize()
    assert torch.equal(step.out_host.view(torch.int16), ref.cpu().view(torch.int16))
    plan = B.make_plan(B.layout_for(d.k_pool, 256, 4), B.DecodeParams(sp.num_seqs, 16, 1, d.block_tables.shape[1],
                                                                      64, 0))
    ws = torch.empty(max(1, plan.workspace_bytes), dtype=torch.uint8, device=DEV)
    out = torch.full_like(ref, float("nan"))
    for passes in ("partial", "merge"):
        paged_decode_passes(d.q, d.k_pool, d.v_pool, d.block_tables, d.seq_lens, case.scale, passes=passes, out=out,
                            workspace=ws, **kw)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
