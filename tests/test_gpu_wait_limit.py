"""The bounded pipeline waits of the partial kernel give up cleanly.

Every wait of the partial kernel's main loop for a stage's data is bounded. A
wait that runs out sets PKV_DEVERR_TIMEOUT, stops the CTA's reading, lets every
copy the CTA has issued land, and returns through the normal epilogue (cluster
barriers included), so nothing faults or hangs. With a bound of one nanosecond
(pkv_set_wait_limit_ns) a wait runs out on ordinary inputs, because a stage
takes microseconds to arrive from HBM (the inputs are evicted from L2 first);
the copies themselves are real and complete. Afterwards the default bound is restored, and the next call on the same
stream must be correct: bit-identical to the call made before.
"""

import zlib

import pytest
import torch

from helpers import run_gpu
from quantized_kv_decode_partial_gb300 import binding as B
from quantized_kv_decode_partial_gb300.workloads import DecodeSpec, draw_lengths, make_case

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def spec(name, **kw):
    base = dict(name=name, num_seqs=16, num_q_heads=32, num_kv_heads=8, head_dim=128, n_query=1, block_size=16,
                bits=16, length_range=(4000, 12000), pool_factor=1.1, seed=zlib.crc32(name.encode()) % 10000)
    base.update(kw)
    return DecodeSpec(**base)


# The finishing forms of the partial pass: partition states through the workspace and
# the merge kernel (many CTAs per SM; bf16 and 8-bit pages), a thread-block cluster merge
# (one CTA per SM), query rows shared by several warps, a single partition writing the
# output, and the balanced schedule (asked for on a bf16 batch; a page group that gives
# up marks the rest of its run as empty). Every case streams enough K/V per SM that its
# warps wait on HBM (the 4-bit kernels compute long enough per chunk that their stages
# have landed before they are waited for).
BAL = B.PKV_SCHEDULE_BALANCED
CASES = [  # (spec, partition rows, schedule)
    (spec("wait_bf16_workspace"), 256, 0),
    (spec("wait_u8_workspace", head_dim=256, bits=8, block_size=32), 512, 0),
    (spec("wait_bf16_cluster", num_seqs=1, lengths=(131072,), length_range=None, pool_factor=1.0), 8192, 0),
    (spec("wait_bf16_query_groups", num_seqs=32, num_kv_heads=1), 1024, 0),
    (spec("wait_bf16_single", num_seqs=32, length_range=(2000, 4000)), 8192, 0),
    (spec("wait_bf16_balanced", num_seqs=32), 0, BAL),
]


def test_cases_take_the_finishing_forms_they_name():
    forms = []
    for sp, partition, schedule in CASES:
        max_blocks = -(-max(draw_lengths(sp)) // sp.block_size)
        layout = B.PoolLayout(1 << 16, sp.num_kv_heads, sp.block_size, sp.head_dim, sp.bits, 64)
        plan = B.make_plan(layout, B.DecodeParams(sp.num_seqs, sp.num_q_heads, 1, max_blocks, partition, 0, 0,
                                                  schedule),
                           sm_count=torch.cuda.get_device_properties(DEV).multi_processor_count)
        forms.append("balanced" if plan.balanced else "single" if plan.max_partitions == 1
                     else "cluster" if plan.merge_in_cluster else "workspace")
    assert forms == ["workspace", "workspace", "cluster", "workspace", "single", "balanced"]


@pytest.mark.parametrize("sp,partition,schedule", CASES, ids=[s.name for s, _, _ in CASES])
def test_short_wait_bound_gives_up_without_a_fault(sp, partition, schedule):
    case = make_case(sp, poison=False).to(DEV)
    ref = run_gpu(case, partition_tokens=partition, schedule=schedule)
    torch.cuda.synchronize()
    # Evict the inputs from L2 (129 MB on a GB300) by writing a larger buffer, so that the
    # stages come from HBM and take microseconds to arrive.
    torch.empty(512 << 20, dtype=torch.uint8, device=DEV).fill_(1)
    torch.cuda.synchronize()
    previous = B.set_wait_limit_ns(1)
    try:
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        out = run_gpu(case, partition_tokens=partition, error_flag=err, schedule=schedule)
        torch.cuda.synchronize()  # the kernel returned: no hang, no fault
    finally:
        B.set_wait_limit_ns(previous)
    assert int(err.item()) == B.PKV_DEVERR_TIMEOUT, int(err.item())
    assert out.shape == ref.shape
    # the stream and the context are still good: the next call is the one from before
    err2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    again = run_gpu(case, partition_tokens=partition, error_flag=err2, schedule=schedule)
    torch.cuda.synchronize()
    assert int(err2.item()) == 0
    assert torch.equal(again.view(torch.int16), ref.view(torch.int16))
