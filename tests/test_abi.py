"""CPU checks of the C ABI: the library loads without a GPU, exports every entry
point the header declares, plans partitions, and rejects bad arguments with
its error codes before touching CUDA."""

import ctypes
import os
import re

import pytest

from quantized_kv_decode_partial_gb300 import binding as B
from quantized_kv_decode_partial_gb300 import build as pkv_build
from quantized_kv_decode_partial_gb300.workloads import WORKLOADS

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "pkv_decode.h")


@pytest.fixture(scope="module")
def lib():
    pkv_build.build()
    return B.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(pkv_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(B.EXPORTS)


def test_binding_constants_match_the_header():
    # every integer #define of the header that the binding mirrors has the header's value
    text = open(HEADER).read()
    defines = {m.group(1): int(m.group(2), 0) for m in re.finditer(r"^#define (PKV_\w+) \(?(-?\w+)\)?", text, re.M)
               if re.fullmatch(r"-?(0x[0-9a-fA-F]+|\d+)", m.group(2))}
    mirrored = {name: value for name, value in defines.items() if hasattr(B, name)}
    assert {"PKV_SCHEDULE_BALANCED", "PKV_CONTRACTION_CUDA_CORE", "PKV_ERR_UNSUPPORTED_SHAPE",
            "PKV_DEVERR_TIMEOUT"} <= set(mirrored)
    for name, value in mirrored.items():
        assert getattr(B, name) == value, name


def test_struct_layouts_match_the_header():
    # the binding's ctypes structures list the header's fields in order
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    for cname, cls in (("pkv_pool_layout", B.PoolLayout), ("pkv_decode_params", B.DecodeParams), ("pkv_plan", B.Plan)):
        body = re.search(r"typedef struct %s \{(.*?)\} %s;" % (cname, cname), text, re.S).group(1)
        names = []
        for decl in body.split(";"):
            decl = decl.strip()
            if decl:
                names += [n.strip() for n in decl.split(None, 1)[1].split(",")]
        assert names == [f for f, _ in cls._fields_], cname


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


def test_version_and_messages(lib):
    assert lib.pkv_version() >= 100
    for code in range(0, -9, -1):
        msg = lib.pkv_strerror(code).decode()
        assert msg and msg != "unknown error code"
    assert lib.pkv_strerror(-99).decode() == "unknown error code"


def _layout(spec, num_blocks=1000):
    return B.PoolLayout(num_blocks, spec.num_kv_heads, spec.block_size, spec.head_dim, spec.bits, spec.group_size,
                        spec.v_head_dim)


def _params(spec, max_blocks, partition=None):
    pt = spec.partition_tokens if partition is None else partition
    if pt < 0:
        pt = max_blocks * spec.block_size
    return B.DecodeParams(spec.num_seqs, spec.num_q_heads, spec.n_query, max_blocks, pt, spec.window)


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_plan_for_workloads(lib, name):
    sp = WORKLOADS[name]
    lmax = max(sp.lengths) if sp.lengths else sp.length_range[1]
    max_blocks = -(-lmax // sp.block_size)
    plan = B.make_plan(_layout(sp), _params(sp, max_blocks), sm_count=152)
    ch = 16 if sp.bits == 16 else 32  # partitions are whole multiples of this
    assert plan.chunk_rows in (16, 32) and plan.partition_tokens % ch == 0 and ch % plan.chunk_rows == 0
    table_parts = -(-max_blocks * sp.block_size // plan.partition_tokens)
    if sp.window:  # only the partitions that tile the window's span from its 32-row aligned base
        rows = min(max_blocks * sp.block_size, sp.window + sp.n_query - 1 + 31)
        assert plan.max_partitions == -(-rows // plan.partition_tokens)
    else:
        assert plan.max_partitions == table_parts
    if sp.partition_tokens > 0:
        assert plan.partition_tokens == sp.partition_tokens
    # grids of at most one CTA per SM take the variant with more warps and stages (4 query-row
    # tiles of 8 at most); one wave of CTAs with 2..16 partitions merges inside a thread-block cluster
    ctas = sp.num_seqs * sp.num_kv_heads * plan.max_partitions
    rows = sp.rep * sp.n_query
    solo = ctas <= 152 and (rows <= 8 or (sp.bits == 16 and sp.head_dim == sp.dv == 128 and rows <= 16))
    assert (plan.smem_bytes > 114 * 1024) if solo else plan.threads_per_cta == 128
    two_per_sm = not solo and plan.smem_bytes <= 114 * 1024
    assert plan.merge_in_cluster == (2 <= plan.max_partitions <= (16 if two_per_sm or solo else 8)
                                     and ctas <= (2 if two_per_sm else 1) * 152)
    if plan.max_partitions == 1 or plan.merge_in_cluster:
        assert plan.workspace_bytes == 0
    else:
        slots = sp.num_seqs * sp.num_q_heads * sp.n_query * plan.max_partitions
        assert plan.workspace_bytes >= slots * (sp.dv + 2) * 4
        # auto plans: never below 256 rows; either about four waves of 2 CTAs per SM, or at least one
        # wave of CTAs that each still get 512 KB of K/V, or the 256-row floor
        if sp.partition_tokens == 0:
            assert plan.partition_tokens >= 256
            ctas = sp.num_seqs * sp.num_kv_heads * plan.max_partitions
            kv_row = sum(2 * d if sp.bits == 16 else d * sp.bits // 8 + d // 16 for d in (sp.head_dim, sp.dv))
            assert (ctas >= 8 * 152 or plan.partition_tokens == 256
                    or (ctas >= 2 * 152 and plan.partition_tokens // 2 < (512 << 10) // kv_row))
            # and no CTA above 3 MB of K/V unless halving would go below the 512 KB floor
            assert (plan.partition_tokens * kv_row <= 3 << 20
                    or plan.partition_tokens // 2 < max(256, (512 << 10) // kv_row))
    assert plan.threads_per_cta in (128, 192, 224, 256) and 0 < plan.smem_bytes <= 227 * 1024
    if not solo and not (sp.bits == 16 and sp.head_dim == 256):  # 16 KB stages of bf16 D=256: one CTA per SM
        assert plan.smem_bytes <= 114 * 1024  # two CTAs per SM


@pytest.mark.parametrize("bits,head_dim,threads", [(16, 64, 256), (16, 128, 256), (16, 256, 224), (4, 128, 256),
                                                   (4, 256, 256), (8, 128, 256), (8, 256, 256)])
def test_small_grids_take_the_one_cta_per_sm_variant(lib, bits, head_dim, threads):
    lay = B.PoolLayout(4096, 4, 32, head_dim, bits, 64)
    small = B.make_plan(lay, B.DecodeParams(1, 16, 1, 256, 512, 0), sm_count=152)  # 4 heads x 16 parts
    assert small.threads_per_cta == threads and 114 * 1024 < small.smem_bytes <= 227 * 1024
    assert small.merge_in_cluster == 1 and small.workspace_bytes == 0
    big = B.make_plan(lay, B.DecodeParams(3, 16, 1, 256, 512, 0), sm_count=152)  # 192 CTAs: more than one per SM
    # bf16 D=256: four warps' 16 KB stages would fill more than half the SM, so those CTAs
    # hold it alone and take seven warps as well
    assert big.threads_per_cta == (224 if (bits, head_dim) == (16, 256) else 128)
    assert big.smem_bytes < small.smem_bytes
    wide_q = B.make_plan(lay, B.DecodeParams(1, 16, 4, 256, 512, 0), sm_count=152)  # 16 query rows per KV head
    # 16 rows: bf16 D=128 has a variant for one CTA per SM; bf16 D=256 CTAs hold their SM
    # alone anyway and take three page groups of two warps
    assert wide_q.threads_per_cta == {(16, 128): 256, (16, 256): 192}.get((bits, head_dim), 128)


def test_single_sequence_plans_merge_in_a_cluster(lib):
    sp = WORKLOADS["affine4_g64_1x8192_hq16_d256"]  # 16 partitions x 4 KV heads = 64 CTAs
    plan = B.make_plan(_layout(sp), _params(sp, 256), sm_count=152)
    assert plan.max_partitions == 16 and plan.merge_in_cluster == 1 and plan.workspace_bytes == 0
    # 17 partitions do not fit a cluster; a grid of more than one wave does not use one either
    assert B.make_plan(_layout(sp), _params(sp, 256, 480), sm_count=152).merge_in_cluster == 0
    assert B.make_plan(_layout(sp), _params(sp, 256), sm_count=16).merge_in_cluster == 0


@pytest.mark.parametrize("bits,head_dim,max_rows", [(16, 64, 64), (16, 128, 64), (16, 256, 64), (4, 128, 64),
                                                     (4, 256, 64), (8, 128, 64), (8, 256, 64)])
def test_query_rows_per_kv_head_limits(lib, bits, head_dim, max_rows):
    for nq in (1, 8, 9, 16, 17, 32, 33, 64, 65):
        lay = B.PoolLayout(100, 1, 32, head_dim, bits, 64)
        par = B.DecodeParams(1, nq, 1, 4, 0, 0)  # REP = nq, N = 1
        plan = B.Plan()
        rc = lib.pkv_make_plan(ctypes.byref(lay), ctypes.byref(par), 152, ctypes.byref(plan))
        assert rc == (B.PKV_OK if nq <= max_rows else B.PKV_ERR_UNSUPPORTED_SHAPE), (nq, rc)


@pytest.mark.parametrize("bits,dk,dv,max_rows", [(16, 192, 128, 64), (16, 256, 128, 64), (16, 128, 256, 64),
                                                  (4, 256, 128, 64), (4, 128, 256, 64), (8, 256, 128, 64),
                                                  (8, 128, 256, 64)])
def test_key_and_value_head_dims_may_differ(lib, bits, dk, dv, max_rows):
    for nq in (1, 8, 9, 32, 33, 64, 65):
        lay = B.PoolLayout(100, 2, 32, dk, bits, 64, dv)
        par = B.DecodeParams(1, 2 * nq, 1, 4, 64, 0)
        plan = B.Plan()
        rc = lib.pkv_make_plan(ctypes.byref(lay), ctypes.byref(par), 1, ctypes.byref(plan))  # 1 SM: no cluster
        assert rc == (B.PKV_OK if nq <= max_rows else B.PKV_ERR_UNSUPPORTED_SHAPE), (nq, rc)
        if rc == B.PKV_OK:  # 33..64 rows: one query group of 8 warps (256 threads)
            assert plan.threads_per_cta == (256 if nq > 32 else 128)
        if rc == B.PKV_OK:  # partition states hold value-dim rows: 2 partitions x 2 nq query heads
            slots = 2 * 2 * nq
            assert plan.max_partitions == 2 and plan.merge_in_cluster == 0
            assert plan.workspace_bytes == -(-slots * dv * 4 // 256) * 256 + slots * 2 * 4


@pytest.mark.parametrize("bits,dk,dv,code", [(16, 64, 128, B.PKV_ERR_UNSUPPORTED_SHAPE),
                                             (16, 192, 192, B.PKV_ERR_BAD_LAYOUT),
                                             (16, 128, 96, B.PKV_ERR_BAD_LAYOUT),
                                             (4, 192, 128, B.PKV_ERR_BAD_LAYOUT),
                                             (8, 256, 64, B.PKV_ERR_BAD_LAYOUT)])
def test_head_dim_pairs_without_a_kernel_are_rejected(lib, bits, dk, dv, code):
    lay = B.PoolLayout(100, 1, 32, dk, bits, 64, dv)
    plan = B.Plan()
    assert lib.pkv_make_plan(ctypes.byref(lay), ctypes.byref(B.DecodeParams(1, 4, 1, 4, 0, 0)), 152,
                             ctypes.byref(plan)) == code


def test_plan_auto_is_monotone_in_sm_count(lib):
    sp = WORKLOADS["bf16_8x131072_n4_hq32_d128"]
    parts = [B.make_plan(_layout(sp), _params(sp, 8192, 0), sm_count=s).partition_tokens for s in (8, 76, 152, 304)]
    assert parts == sorted(parts, reverse=True)


@pytest.mark.parametrize("field,value,code", [
    ("bits", 3, B.PKV_ERR_BAD_LAYOUT), ("bits", 2, B.PKV_ERR_BAD_LAYOUT), ("group_size", 32, B.PKV_ERR_BAD_LAYOUT),
    ("head_dim", 96, B.PKV_ERR_BAD_LAYOUT), ("block_size", 4, B.PKV_ERR_BAD_LAYOUT),
    ("block_size", 24, B.PKV_ERR_BAD_LAYOUT), ("block_size", 48, B.PKV_ERR_BAD_LAYOUT),
    ("num_blocks", 0, B.PKV_ERR_BAD_LAYOUT), ("num_blocks", 1 << 28, B.PKV_ERR_BAD_LAYOUT),
])
def test_plan_rejects_bad_layouts(lib, field, value, code):
    sp = WORKLOADS["affine4_g64_1x8192_hq16_d256"]
    lay = _layout(sp)
    setattr(lay, field, value)
    plan = B.Plan()
    assert lib.pkv_make_plan(ctypes.byref(lay), ctypes.byref(_params(sp, 256)), 152, ctypes.byref(plan)) == code


@pytest.mark.parametrize("field,value,code", [
    ("num_q_heads", 6, B.PKV_ERR_BAD_PARAMS), ("n_query", 0, B.PKV_ERR_BAD_PARAMS),
    ("num_seqs", 0, B.PKV_ERR_BAD_PARAMS), ("max_blocks_per_seq", 0, B.PKV_ERR_BAD_PARAMS),
    ("partition_tokens", -1, B.PKV_ERR_BAD_PARAMS), ("n_query", 17, B.PKV_ERR_UNSUPPORTED_SHAPE),
    ("window", -1, B.PKV_ERR_BAD_PARAMS),
])
def test_plan_rejects_bad_params(lib, field, value, code):
    sp = WORKLOADS["affine4_g64_1x8192_hq16_d256"]  # HQ 16 / HK 4: REP 4, so n_query 17 asks for 68 > 64 rows
    par = _params(sp, 256)
    setattr(par, field, value)
    plan = B.Plan()
    assert lib.pkv_make_plan(ctypes.byref(_layout(sp)), ctypes.byref(par), 152, ctypes.byref(plan)) == code


def test_decode_call_validates_before_cuda(lib):
    sp = WORKLOADS["affine4_g64_1x8192_hq16_d256"]
    lay, par = _layout(sp), _params(sp, 256)
    fake = 1 << 20  # aligned, never dereferenced: validation fails first
    args = [fake] * 9
    call = lambda a, lay=lay: lib.pkv_paged_decode_attention(
        ctypes.byref(lay), ctypes.byref(par), *a[:9], 0.0625, fake, fake, 1 << 30, None, None)
    null_q = list(args)
    null_q[0] = None
    assert call(null_q) == B.PKV_ERR_NULL_POINTER
    no_scales = list(args)
    no_scales[3] = None  # affine pages need their scale planes
    assert call(no_scales) == B.PKV_ERR_NULL_POINTER
    mis = list(args)
    mis[1] = fake + 8
    assert call(mis) == B.PKV_ERR_MISALIGNED
    bad = B.PoolLayout(lay.num_blocks, lay.num_kv_heads, lay.block_size, lay.head_dim, 5, 64)
    assert call(args, bad) == B.PKV_ERR_BAD_LAYOUT


def test_decode_without_gpu_fails_loudly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    sp = WORKLOADS["bf16_1x1024_hq2_d256"]
    lay, par = _layout(sp, 128), _params(sp, 64)
    fake = 1 << 20
    rc = lib.pkv_paged_decode_attention(ctypes.byref(lay), ctypes.byref(par), fake, fake, fake, None, None, None,
                                        None, fake, fake, 0.0625, fake, None, 0, None, None)
    assert rc == B.PKV_ERR_CUDA
    assert lib.pkv_last_cuda_error().decode()


def test_step_handle_validates_before_cuda(lib):
    sp = WORKLOADS["bf16_1x1024_hq2_d256"]
    lay, par = _layout(sp, 128), _params(sp, 64)
    fake = 1 << 20
    h = ctypes.c_void_p(123)

    def create(layout, in_bytes=0, in_host=None, out=fake, handle=True):
        return lib.pkv_step_create(ctypes.byref(layout), ctypes.byref(par), in_host, fake, in_bytes, None, fake,
                                   None, None, fake, fake, None, None, None, None, fake, fake, 0.0625, out, None, 0,
                                   None, None, ctypes.byref(h) if handle else None)

    assert create(lay, handle=False) == B.PKV_ERR_NULL_POINTER
    assert create(B.PoolLayout(128, 1, 16, 96, 16, 64)) == B.PKV_ERR_BAD_LAYOUT and not h.value
    assert create(lay, in_bytes=64) == B.PKV_ERR_NULL_POINTER  # bytes to copy but no host block
    assert create(lay, out=None) == B.PKV_ERR_NULL_POINTER
    lib.pkv_step_destroy(None)  # allowed
    assert lib.pkv_step_run(None) == B.PKV_ERR_NULL_POINTER
    import torch
    if not torch.cuda.is_available():  # valid arguments reach CUDA, which fails loudly here
        assert create(lay) == B.PKV_ERR_CUDA and not h.value


def test_gather_validates(lib):
    fake = 1 << 20
    assert lib.pkv_paged_gather(fake, 10, 2, 16, 6, fake, fake, 1, 4, 64, fake, None, None) == B.PKV_ERR_BAD_PARAMS
    assert lib.pkv_paged_gather(None, 10, 2, 16, 8, fake, fake, 1, 4, 64, fake, None, None) == B.PKV_ERR_NULL_POINTER
    assert lib.pkv_paged_gather(fake + 4, 10, 2, 16, 8, fake, fake, 1, 4, 64, fake, None, None) == B.PKV_ERR_MISALIGNED


def test_missing_library_raises(tmp_path):
    with pytest.raises(B.LibraryNotBuilt):
        B.load_library(str(tmp_path / "nope.so"))


@pytest.mark.parametrize("bits,block_size", [(16, 16), (4, 32)])
def test_partition_tokens_past_the_table_give_one_partition(lib, bits, block_size):
    # A caller's partition size of INT_MAX (or anything past the table) means one
    # partition, never a size that wraps around int32.
    lay = B.PoolLayout(1000, 2, block_size, 128, bits, 64)
    for max_blocks in (4, 1 << 20):
        max_len = max_blocks * block_size
        for pt in (max_len, max_len + 1, 2**31 - 1, 2**31 - block_size + 1):
            plan = B.Plan()
            rc = lib.pkv_make_plan(ctypes.byref(lay), ctypes.byref(B.DecodeParams(3, 8, 1, max_blocks, pt, 0)), 152,
                                   ctypes.byref(plan))
            assert rc == B.PKV_OK
            assert plan.max_partitions == 1 and plan.partition_tokens == max_len and plan.workspace_bytes == 0


def test_wait_limit_setter_round_trip(lib):
    # 0 restores the default bound of one second; the previous bound comes back.
    first = lib.pkv_set_wait_limit_ns(0)
    assert lib.pkv_set_wait_limit_ns(123) == 10**9
    assert lib.pkv_set_wait_limit_ns(0) == 123
    assert lib.pkv_set_wait_limit_ns(first) == 10**9
    assert lib.pkv_set_wait_limit_ns(0) == first


@pytest.mark.parametrize("bits,dk,dv,nq,ok", [(16, 128, 128, 4, True), (16, 256, 256, 2, True), (16, 64, 64, 1, True),
                                             (16, 128, 128, 5, False), (16, 192, 128, 2, False),
                                             (4, 256, 256, 4, False), (8, 128, 128, 2, False)])
def test_cuda_core_contraction_shapes(lib, bits, dk, dv, nq, ok):
    lay = B.PoolLayout(100, 1, 32, dk, bits, 64, 0 if dv == dk else dv)
    plan = B.Plan()
    par = B.DecodeParams(1, nq, 1, 4, 64, 0, B.PKV_CONTRACTION_CUDA_CORE)
    rc = lib.pkv_make_plan(ctypes.byref(lay), ctypes.byref(par), 152, ctypes.byref(plan))
    assert rc == (B.PKV_OK if ok else B.PKV_ERR_UNSUPPORTED_SHAPE)
    if ok:
        assert plan.contraction == B.PKV_CONTRACTION_CUDA_CORE
    tc = B.DecodeParams(1, nq, 1, 4, 64, 0, B.PKV_CONTRACTION_TENSOR)
    if lib.pkv_make_plan(ctypes.byref(lay), ctypes.byref(tc), 152, ctypes.byref(plan)) == B.PKV_OK:
        assert plan.contraction == B.PKV_CONTRACTION_TENSOR


def test_contraction_field_is_validated(lib):
    lay = B.PoolLayout(100, 1, 32, 128, 16, 64)
    plan = B.Plan()
    for bad in (-1, 3):
        par = B.DecodeParams(1, 2, 1, 4, 64, 0, bad)
        assert lib.pkv_make_plan(ctypes.byref(lay), ctypes.byref(par), 152, ctypes.byref(plan)) == B.PKV_ERR_BAD_PARAMS


def test_output_rows_past_int32_are_rejected(lib):
    lay = B.PoolLayout(100, 65535, 16, 64, 16, 64)
    plan = B.Plan()
    # 65535 sequences x 65535 query heads: 4.3e9 output rows
    par = B.DecodeParams(65535, 65535, 1, 4, 64, 0)
    assert lib.pkv_make_plan(ctypes.byref(lay), ctypes.byref(par), 152, ctypes.byref(plan)) == B.PKV_ERR_BAD_PARAMS


@pytest.mark.parametrize("bits,block_size", [(16, 8), (4, 8), (4, 16), (8, 8), (8, 16), (16, 48), (4, 96)])
def test_blocks_of_8_rows_or_more_that_divide_a_chunk_are_accepted(lib, bits, block_size):
    # a chunk (16 rows for bf16 pages, 32 for affine) spans several such blocks; or blocks
    # of whole chunks. Pools of smaller blocks take the instantiations of grids of several
    # CTAs per SM (128 threads, even for one CTA per SM), neither the balanced schedule nor
    # the CUDA-core contraction.
    lay = B.PoolLayout(1000, 2, block_size, 128, bits, 64)
    plan = B.Plan()
    par = B.DecodeParams(2, 8, 1, 4096 // block_size, 0, 0, 0, B.PKV_SCHEDULE_BALANCED)
    assert lib.pkv_make_plan(ctypes.byref(lay), ctypes.byref(par), 152, ctypes.byref(plan)) == B.PKV_OK
    assert plan.partition_tokens % (16 if bits == 16 else 32) == 0
    small = block_size < plan.chunk_rows
    assert plan.balanced == int(not small)
    if small:
        assert plan.threads_per_cta == 128
        if bits == 16:
            cc = B.DecodeParams(2, 4, 1, 4096 // block_size, 0, 0, B.PKV_CONTRACTION_CUDA_CORE)
            assert lib.pkv_make_plan(ctypes.byref(lay), ctypes.byref(cc), 152, ctypes.byref(plan)) == \
                B.PKV_ERR_UNSUPPORTED_SHAPE


def test_schedule_field_is_validated(lib):
    lay = B.PoolLayout(100, 1, 32, 128, 16, 64)
    plan = B.Plan()
    for bad in (-1, 3):
        par = B.DecodeParams(1, 2, 1, 4, 64, 0, 0, bad)
        assert lib.pkv_make_plan(ctypes.byref(lay), ctypes.byref(par), 152, ctypes.byref(plan)) == B.PKV_ERR_BAD_PARAMS


def _balanced_bytes(runs, units, nq, dv):
    slots = (runs + units) * nq
    return -(-slots * dv * 4 // 256) * 256 + slots * 2 * 4


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_balanced_schedule_where_partitions_would_use_the_workspace(lib, name):
    # The library's split (partition_tokens = 0) of a 4-bit workload whose partitions would
    # go through the workspace and the merge kernel takes the balanced schedule; its
    # workspace then holds a state slot per (run, unit) pair for the largest grid the
    # shared memory allows (runs = SMs x CTAs per SM x page groups), and the partitions'
    # states as well (the fused call runs those).
    sp = WORKLOADS[name]
    lmax = max(sp.lengths) if sp.lengths else sp.length_range[1]
    max_blocks = -(-lmax // sp.block_size)
    auto = B.make_plan(_layout(sp), _params(sp, max_blocks, 0), sm_count=152)
    parts = B.make_plan(_layout(sp), B.DecodeParams(sp.num_seqs, sp.num_q_heads, sp.n_query, max_blocks, 0,
                                                    sp.window, 0, B.PKV_SCHEDULE_PARTITIONS), sm_count=152)
    assert parts.balanced == 0
    workspace_partitions = parts.max_partitions > 1 and not parts.merge_in_cluster
    assert auto.balanced == int(workspace_partitions and sp.bits == 4)
    assert (auto.partition_tokens, auto.max_partitions, auto.merge_in_cluster) == \
        (parts.partition_tokens, parts.max_partitions, parts.merge_in_cluster)
    if auto.balanced:
        per_sm = max(1, min(228 * 1024 // (auto.smem_bytes + 1024), 2048 // auto.threads_per_cta, 32))
        nq = sp.rep * sp.n_query
        wq = 8 if auto.threads_per_cta == 256 and nq > 32 else 1  # a query group of 8 warps is its CTA
        page_groups = auto.threads_per_cta // 32 // wq
        need = _balanced_bytes(152 * per_sm * page_groups, sp.num_seqs * sp.num_kv_heads, nq, sp.dv)
        assert auto.workspace_bytes >= max(need, parts.workspace_bytes)
    else:
        assert auto.workspace_bytes == parts.workspace_bytes


def test_balanced_schedule_conditions(lib):
    # 4-bit pages, one KV head of 4 query heads, tables of 8192 rows: 64 to 257 units, so
    # the library's split makes several partitions per unit, several waves of CTAs
    lay = B.PoolLayout(4096, 1, 32, 128, 4, 64)

    def plan(num_seqs, partition=0, schedule=0, contraction=0):
        return B.make_plan(lay, B.DecodeParams(num_seqs, 4, 1, 256, partition, 0, contraction, schedule),
                           sm_count=152)

    assert plan(64).balanced == 1 and plan(64).max_partitions > 1
    assert plan(64, partition=1024).balanced == 0        # a caller's partition size is kept
    assert plan(64, schedule=B.PKV_SCHEDULE_PARTITIONS).balanced == 0
    assert plan(256).balanced == 1
    assert plan(257).balanced == 0                       # more sequences than the prefix holds
    # bf16 pages stream at the memory's pace: partitions, unless asked for; never with the
    # CUDA-core contraction
    bf16 = B.PoolLayout(4096, 1, 16, 128, 16, 64)
    assert B.make_plan(bf16, B.DecodeParams(64, 4, 1, 512, 0, 0), sm_count=152).balanced == 0
    assert B.make_plan(bf16, B.DecodeParams(64, 4, 1, 512, 0, 0, 0, B.PKV_SCHEDULE_BALANCED),
                       sm_count=152).balanced == 1
    assert B.make_plan(bf16, B.DecodeParams(64, 4, 1, 512, 0, 0, B.PKV_CONTRACTION_CUDA_CORE,
                                            B.PKV_SCHEDULE_BALANCED), sm_count=152).balanced == 0
    # one sequence of 8 KV heads and 4096 rows: 16 partitions per head merge in a cluster
    lay8 = B.PoolLayout(4096, 8, 16, 128, 16, 64)
    one = B.make_plan(lay8, B.DecodeParams(1, 8, 1, 256, 0, 0), sm_count=152)
    assert one.merge_in_cluster == 1 and one.balanced == 0 and one.workspace_bytes == 0
    forced = B.make_plan(lay8, B.DecodeParams(1, 8, 1, 256, 0, 0, 0, B.PKV_SCHEDULE_BALANCED), sm_count=152)
    assert forced.balanced == 1 and forced.merge_in_cluster == 1 and forced.workspace_bytes > 0
