"""The entry point that allocates nothing, against the main entry point.

pkv_paged_decode_attention_no_alloc serves callers that cannot allocate device
memory (their allocator owns every byte, or they only hold one call's tensors):
its partition states live in the library's static device scratch instead of a
caller workspace. Called here through the C ABI, twice in a row on the same
scratch, its output must match pkv_paged_decode_attention's within the parity
tolerance of the other GPU tests. This file is collected last on purpose.
"""

import ctypes
import zlib

import pytest
import torch

from helpers import assert_close, run_gpu
from quantized_kv_decode_partial_gb300 import binding as B
from quantized_kv_decode_partial_gb300.workloads import DecodeCase, DecodeSpec, make_case

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def spec(name, **kw):
    base = dict(name=name, num_seqs=3, num_q_heads=8, num_kv_heads=2, head_dim=128, n_query=1, block_size=16,
                bits=16, length_range=(100, 3000), pool_factor=2.0, seed=zlib.crc32(name.encode()) % 10000)
    base.update(kw)
    return DecodeSpec(**base)


def no_alloc_call(lib, case, partition_tokens, out, err=None):
    sp = case.spec
    layout = B.layout_for(case.k_pool, sp.head_dim, sp.bits, sp.group_size)
    params = B.DecodeParams(sp.num_seqs, sp.num_q_heads, sp.n_query, case.block_tables.shape[1], partition_tokens)
    p = lambda t: None if t is None else t.data_ptr()
    return lib.pkv_paged_decode_attention_no_alloc(
        ctypes.byref(layout), ctypes.byref(params), p(case.q), p(case.k_pool), p(case.v_pool), p(case.k_scales),
        p(case.k_biases), p(case.v_scales), p(case.v_biases), p(case.block_tables), p(case.seq_lens),
        float(case.scale), p(out), p(err), torch.cuda.current_stream(DEV).cuda_stream)


@pytest.mark.parametrize("sp,partition", [
    (spec("na_bf16_auto"), 0),
    (spec("na_bf16_p64", n_query=2, num_q_heads=16), 64),
    (spec("na_u4_auto", head_dim=256, bits=4, block_size=32), 0),
    (spec("na_u8_p96", head_dim=128, bits=8, block_size=32, num_q_heads=4, num_kv_heads=1), 96),
], ids=lambda x: x.name if hasattr(x, "name") else str(x))
def test_no_alloc_matches_main_entry_twice(sp, partition):
    lib = B.load_library()
    case = make_case(sp).to(DEV)
    ref = run_gpu(case, partition_tokens=partition).double().cpu().numpy()
    for _ in range(2):  # the second call reuses the scratch the first one left behind
        out = torch.full_like(case.q, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        assert no_alloc_call(lib, case, partition, out, err) == B.PKV_OK
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(out.double().cpu().numpy(), ref, f"{sp.name} no-alloc")


def test_no_alloc_coarsens_library_partitions_and_rejects_oversized_ones():
    lib = B.load_library()
    # One sequence, 8 query heads on 1 KV head, 8 queries (64 query rows), a 262144-row
    # table: the library's own plan (512-row partitions, 512 of them) needs about 17 MB of
    # partition states, more than the 16 MiB scratch, so the no-alloc entry doubles the
    # partition size. A caller-fixed 16-row partition cannot fit at all.
    sp = spec("na_big", num_seqs=1, num_q_heads=8, num_kv_heads=1, head_dim=128, n_query=8,
              lengths=(262144,), length_range=None, pool_factor=1.0)
    case = make_case(sp, device=DEV, poison=False)
    plan = B.make_plan(B.layout_for(case.k_pool, 128, 16),
                       B.DecodeParams(1, 8, 8, case.block_tables.shape[1], 0))
    assert plan.workspace_bytes > B.PKV_STATIC_SCRATCH_BYTES
    out = torch.empty_like(case.q)
    assert no_alloc_call(lib, case, 16, out) == B.PKV_ERR_SCRATCH_TOO_SMALL
    ref = run_gpu(case, partition_tokens=0).double().cpu().numpy()
    for _ in range(2):
        out.fill_(float("nan"))
        assert no_alloc_call(lib, case, 0, out) == B.PKV_OK
        torch.cuda.synchronize()
        assert_close(out.double().cpu().numpy(), ref, "na_big auto")


def test_no_alloc_coarsening_stops_at_one_partition_for_tables_past_2_pow_30():
    # Tables longer than 2^30 rows (16385 blocks of 65536 rows) with 64 query rows for each of
    # 256 sequences: the library's plan needs two partitions even at 2^30 rows each, whose
    # states (17 MB) still exceed the 16 MiB scratch. Coarsening must go on to a single
    # partition (no scratch at all) and return, not loop. Every sequence reads the first
    # rows of block 0; table entries past the lengths are never used.
    lib = B.load_library()
    seqs, rep, d, bs, max_blocks = 256, 64, 128, 65536, 16385
    g = torch.Generator().manual_seed(7)
    lens = torch.randint(50, 300, (seqs,), generator=g, dtype=torch.int32)
    k_pool = torch.randn((1, 1, bs, d), generator=g).to(torch.bfloat16)
    v_pool = torch.randn((1, 1, bs, d), generator=g).to(torch.bfloat16)
    q = torch.randn((seqs, rep, 1, d), generator=g).to(torch.bfloat16)
    tables = torch.zeros((seqs, max_blocks), dtype=torch.int32)
    sp = DecodeSpec(name="na_2p30", num_seqs=seqs, num_q_heads=rep, num_kv_heads=1, head_dim=d, n_query=1,
                    block_size=bs, bits=16, lengths=tuple(int(x) for x in lens))
    case = DecodeCase(spec=sp, q=q, k_pool=k_pool, v_pool=v_pool, block_tables=tables, seq_lens=lens,
                      scale=d ** -0.5, num_blocks=1, lens_host=[int(x) for x in lens]).to(DEV)
    layout = B.layout_for(case.k_pool, d, 16)
    auto = B.make_plan(layout, B.DecodeParams(seqs, rep, 1, max_blocks, 0))
    assert auto.workspace_bytes > B.PKV_STATIC_SCRATCH_BYTES
    two = B.make_plan(layout, B.DecodeParams(seqs, rep, 1, max_blocks, 1 << 30))
    assert two.max_partitions == 2 and two.workspace_bytes > B.PKV_STATIC_SCRATCH_BYTES
    ref = run_gpu(case, partition_tokens=max_blocks * bs)  # one partition
    for _ in range(2):
        out = torch.full_like(case.q, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        assert no_alloc_call(lib, case, 0, out, err) == B.PKV_OK
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
