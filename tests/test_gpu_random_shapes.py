"""A seeded sweep of random shapes through the C ABI against the float64 oracle:
page formats, key/value head-dim pairs, GQA factors, query counts, page sizes,
ragged lengths, partition sizes (single, cluster, workspace) and sliding windows,
drawn from what the library supports, so that combinations the hand-written cases
miss still get checked."""

import random

import pytest
import torch

from helpers import assert_close, oracle_out, run_gpu
from quantized_kv_decode_partial_gb300 import binding as B
from quantized_kv_decode_partial_gb300.workloads import DecodeSpec, make_case

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")

# (bits, key head dim, value head dim, most query rows per KV head)
SHAPES = [(16, 64, 64, 64), (16, 128, 128, 64), (16, 256, 256, 32), (16, 192, 128, 32), (16, 256, 128, 8),
          (16, 128, 256, 8), (4, 128, 128, 64), (4, 256, 256, 32), (4, 256, 128, 8), (4, 128, 256, 8),
          (8, 128, 128, 64), (8, 256, 256, 32), (8, 256, 128, 8), (8, 128, 256, 8)]


def draw(i):
    rnd = random.Random(9000 + i)
    bits, dk, dv, max_rows = rnd.choice(SHAPES)
    n_query = rnd.choice([1, 1, 2, 3, 4])
    rep = rnd.choice([r for r in (1, 2, 4, 8, 16) if r * n_query <= max_rows] or [1])
    hk = rnd.choice([1, 2, 3])
    bs = rnd.choice([16, 32, 64] if bits == 16 else [32, 64])
    num_seqs = rnd.choice([1, 2, 5, 9])
    hi = rnd.choice([40, 300, 900])
    window = rnd.choice([0, 0, 0, 1, 7, 100])
    part = rnd.choice([-1, 0, 16 if bits == 16 else 32, 64, 96, 160])
    spec = DecodeSpec(name=f"rand{i}", num_seqs=num_seqs, num_q_heads=rep * hk, num_kv_heads=hk, head_dim=dk,
                      v_head_dim=dv, n_query=n_query, block_size=bs, bits=bits, length_range=(n_query, hi),
                      pool_factor=1.5, partition_tokens=part, window=window, seed=9000 + i)
    return spec


@pytest.mark.parametrize("i", range(40))
def test_random_shape_matches_oracle(i):
    spec = draw(i)
    case = make_case(spec)
    ref = oracle_out(case)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_gpu(case.to(DEV), error_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_close(out.double().cpu().numpy(), ref, f"{spec}")


def draw_more(i):
    # the same space with blocks smaller than the staged chunk (8 or 16 rows) and the
    # schedule drawn too (the balanced schedule applies where partition_tokens is 0 and
    # the blocks hold whole chunks; elsewhere the call runs partitions)
    rnd = random.Random(19000 + i)
    spec = draw(10000 + i)
    bs = rnd.choice([8, 16, 32] if spec.bits == 16 else [8, 16, 32, 64])
    part = rnd.choice([-1, 0, 0, 64, 160])
    schedule = rnd.choice([B.PKV_SCHEDULE_AUTO, B.PKV_SCHEDULE_PARTITIONS, B.PKV_SCHEDULE_BALANCED])
    return DecodeSpec(**{**spec.__dict__, "name": f"rand_more{i}", "block_size": bs, "partition_tokens": part,
                         "seed": 19000 + i}), schedule


@pytest.mark.parametrize("i", range(40))
def test_random_shape_with_small_blocks_and_schedules_matches_oracle(i):
    spec, schedule = draw_more(i)
    case = make_case(spec)
    ref = oracle_out(case)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_gpu(case.to(DEV), error_flag=err, schedule=schedule)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_close(out.double().cpu().numpy(), ref, f"{spec} schedule={schedule}")
