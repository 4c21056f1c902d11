"""GPU parity of the write side: pkv_paged_append against the write oracle, bit
for bit (codes, scales, biases and bf16 rows), then a decode over the appended
cache against the attention oracle."""

import zlib
from dataclasses import replace

import numpy as np
import pytest
import torch

from helpers import assert_close, oracle_out, run_gpu
from oracle import paged_write as pw
from quantized_kv_decode_partial_gb300 import binding as B
from quantized_kv_decode_partial_gb300 import paged_append
from quantized_kv_decode_partial_gb300.workloads import DecodeSpec, make_case

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def bits_of(t):
    if t is None:
        return None
    if t.dtype == torch.bfloat16:
        return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)
    return t.detach().cpu().numpy()


def setup(bits, D, n_new, num_seqs=3, seed_name="", dv=0, bs=0):
    name = f"app_{bits}_{D}_{n_new}_{seed_name}" + (f"_dv{dv}" if dv else "") + (f"_bs{bs}" if bs else "")
    seed = zlib.crc32(name.encode()) % 10000
    bs = bs or (16 if bits == 16 else 32)
    DV = dv or D
    sp = DecodeSpec(name=name, num_seqs=num_seqs, num_q_heads=4, num_kv_heads=2, head_dim=D, n_query=1,
                    block_size=bs, bits=bits, length_range=(1, 150), pool_factor=2.0, seed=seed, v_head_dim=dv)
    g = torch.Generator().manual_seed(seed + 1)
    lens = [int(x) for x in torch.randint(0, 150, (num_seqs,), generator=g)]
    lens[0] = bs - 1  # the new rows of sequence 0 cross a page boundary
    case = make_case(sp, lengths=[l + n_new for l in lens], poison=False)  # tables hold the new rows' pages
    # new rows with very different ranges per group (including a constant group)
    k_new = torch.randn((num_seqs, 2, n_new, D), generator=g) * torch.rand((num_seqs, 2, n_new, D // 16), generator=g).repeat_interleave(16, -1) * 8
    v_new = torch.randn((num_seqs, 2, n_new, DV), generator=g)
    k_new[..., :64] = k_new[..., :1]
    return sp, case, lens, k_new.to(torch.bfloat16), v_new.to(torch.bfloat16)


# (bits, D, new rows, value head dim, block size; 0: a chunk's rows)
CASES = [(16, 128, 1, 0, 0), (16, 64, 3, 0, 0), (16, 256, 2, 0, 0), (4, 256, 1, 0, 0), (4, 128, 3, 0, 0),
         (8, 256, 2, 0, 0), (8, 128, 1, 0, 0), (16, 192, 2, 128, 0), (4, 128, 2, 256, 0), (8, 256, 1, 128, 0),
         (16, 128, 3, 0, 8), (4, 256, 2, 0, 16), (4, 128, 3, 0, 8), (8, 256, 2, 0, 8)]


@pytest.mark.parametrize("bits,D,n_new,dv,bs", CASES)
def test_append_is_bit_exact(bits, D, n_new, dv, bs):
    sp, case, lens, k_new, v_new = setup(bits, D, n_new, dv=dv, bs=bs)
    ref = pw.append_rows(k_new.float().numpy(), v_new.float().numpy(), case.block_tables.numpy(), lens,
                         bits_of(case.k_pool), bits_of(case.v_pool), bits=bits,
                         k_scales=bits_of(case.k_scales), k_biases=bits_of(case.k_biases),
                         v_scales=bits_of(case.v_scales), v_biases=bits_of(case.v_biases))
    d = case.to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    paged_append(k_new.to(DEV), v_new.to(DEV), d.block_tables, torch.tensor(lens, dtype=torch.int32, device=DEV),
                 d.k_pool, d.v_pool, bits=bits, k_scales=d.k_scales, k_biases=d.k_biases, v_scales=d.v_scales,
                 v_biases=d.v_biases, error_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = {"k_pool": d.k_pool, "v_pool": d.v_pool}
    if bits != 16:
        got.update(k_scales=d.k_scales, k_biases=d.k_biases, v_scales=d.v_scales, v_biases=d.v_biases)
    for name, t in got.items():
        assert np.array_equal(bits_of(t), ref[name]), name


@pytest.mark.parametrize("bits", [16, 4, 8])
def test_decode_after_append_matches_oracle(bits):
    D = 256 if bits == 4 else 128
    sp, case, lens, k_new, v_new = setup(bits, D, 2, seed_name="decode")
    d = case.to(DEV)
    lens_d = torch.tensor(lens, dtype=torch.int32, device=DEV)
    paged_append(k_new.to(DEV), v_new.to(DEV), d.block_tables, lens_d, d.k_pool, d.v_pool, bits=bits,
                 k_scales=d.k_scales, k_biases=d.k_biases, v_scales=d.v_scales, v_biases=d.v_biases)
    d.seq_lens = lens_d + 2
    host = d.to("cpu")  # the appended cache, read back for the oracle
    out = run_gpu(d, partition_tokens=32)
    assert_close(out.double().cpu().numpy(), oracle_out(host), f"decode after append {bits}")


def test_append_flags_bad_blocks_and_lengths():
    sp, case, lens, k_new, v_new = setup(4, 256, 1, seed_name="bad")
    d = case.to(DEV)
    tb = d.block_tables.clone()
    tb[1, lens[1] // sp.block_size] = case.num_blocks + 3
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    paged_append(k_new.to(DEV), v_new.to(DEV), tb, torch.tensor(lens, dtype=torch.int32, device=DEV), d.k_pool,
                 d.v_pool, bits=4, k_scales=d.k_scales, k_biases=d.k_biases, v_scales=d.v_scales,
                 v_biases=d.v_biases, error_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & B.PKV_DEVERR_BAD_BLOCK
    err.zero_()
    too_long = torch.tensor([tb.shape[1] * sp.block_size] * 3, dtype=torch.int32, device=DEV)
    snapshot = d.k_pool.clone()
    paged_append(k_new.to(DEV), v_new.to(DEV), d.block_tables, too_long, d.k_pool, d.v_pool, bits=4,
                 k_scales=d.k_scales, k_biases=d.k_biases, v_scales=d.v_scales, v_biases=d.v_biases, error_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & B.PKV_DEVERR_BAD_SEQ_LEN
    assert torch.equal(d.k_pool, snapshot)  # nothing written


# ---------------------------------------------------------------- fused append + attend

def setup_fused(bits, D, N, hq, hk, seed_name, num_seqs=3, length_range=(1, 300), window=0, dv=0):
    name = f"fused_{bits}_{D}_{N}_{hq}_{seed_name}" + (f"_dv{dv}" if dv else "")
    seed = zlib.crc32(name.encode()) % 10000
    bs = 16 if bits == 16 else 32
    g = torch.Generator().manual_seed(seed + 1)
    lens = [int(x) for x in torch.randint(*length_range, (num_seqs,), generator=g)]
    lens[0] = bs - 1  # the new rows of sequence 0 cross a page boundary
    sp = DecodeSpec(name=name, num_seqs=num_seqs, num_q_heads=hq, num_kv_heads=hk, head_dim=D, n_query=N,
                    block_size=bs, bits=bits, length_range=length_range, pool_factor=2.0, seed=seed, window=window,
                    v_head_dim=dv)
    case = make_case(sp, lengths=[l + N for l in lens], poison=False)  # seq_lens count the new rows
    k_new = (torch.randn((num_seqs, hk, N, D), generator=g) * 3).to(torch.bfloat16)
    v_new = torch.randn((num_seqs, hk, N, dv or D), generator=g).to(torch.bfloat16)
    return sp, case, lens, k_new, v_new


FUSED = [
    # bits, D, N, HQ, HK, partition_tokens (-1 single, 0 auto), window, value head dim (0: D), sequences
    (16, 128, 1, 8, 2, -1, 0, 0, 3),
    (16, 128, 4, 8, 2, 32, 0, 0, 3),
    (16, 256, 2, 4, 2, 64, 0, 0, 3),
    (16, 64, 3, 8, 1, 48, 0, 0, 3),
    (4, 256, 2, 8, 2, 64, 0, 0, 3),
    (4, 128, 1, 4, 1, 0, 0, 0, 3),
    (8, 128, 3, 8, 2, 32, 0, 0, 3),
    (8, 256, 1, 8, 2, -1, 0, 0, 3),
    (16, 128, 4, 8, 2, 32, 40, 0, 3),
    (16, 192, 2, 8, 2, 32, 0, 128, 3),
    (4, 256, 1, 8, 2, 64, 0, 128, 3),
    # one query group of 8 warps (33..64 query rows at 256-dim heads)
    (16, 256, 2, 64, 2, 64, 0, 0, 3),
    (4, 256, 4, 24, 2, 64, 0, 128, 3),
    # affine, 8 query rows, grids of several waves
    (4, 256, 2, 8, 2, 32, 0, 0, 120),
    (8, 128, 1, 8, 2, 32, 0, 0, 120),
]


@pytest.mark.parametrize("bits,D,N,hq,hk,part,window,dv,seqs", FUSED,
                         ids=[f"b{c[0]}_d{c[1]}_n{c[2]}_p{c[5]}_w{c[6]}_v{c[7]}_s{c[8]}" for c in FUSED])
def test_fused_append_attend_matches_append_then_decode(bits, D, N, hq, hk, part, window, dv, seqs):
    sp, case, lens, k_new, v_new = setup_fused(bits, D, N, hq, hk, f"p{part}w{window}", window=window, dv=dv,
                                               num_seqs=seqs)
    part = 1 << 20 if part < 0 else part  # one partition: any size past the table
    # the write oracle's pools, then the attention oracle over them
    ref = pw.append_rows(k_new.float().numpy(), v_new.float().numpy(), case.block_tables.numpy(), lens,
                         bits_of(case.k_pool), bits_of(case.v_pool), bits=bits,
                         k_scales=bits_of(case.k_scales), k_biases=bits_of(case.k_biases),
                         v_scales=bits_of(case.v_scales), v_biases=bits_of(case.v_biases))
    planes = ("k_pool", "v_pool") + (() if bits == 16 else ("k_scales", "k_biases", "v_scales", "v_biases"))

    # two-call path: pkv_paged_append, then pkv_paged_decode_attention
    two = case.to(DEV)
    paged_append(k_new.to(DEV), v_new.to(DEV), two.block_tables, two.seq_lens - N, two.k_pool, two.v_pool,
                 bits=bits, k_scales=two.k_scales, k_biases=two.k_biases, v_scales=two.v_scales,
                 v_biases=two.v_biases)
    out_two = run_gpu(two, partition_tokens=part)

    # fused path
    one = case.to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out_one = B.paged_decode_append_attention(
        one.q, k_new.to(DEV), v_new.to(DEV), one.k_pool, one.v_pool, one.block_tables, one.seq_lens, case.scale,
        bits=bits, k_scales=one.k_scales, k_biases=one.k_biases, v_scales=one.v_scales, v_biases=one.v_biases,
        partition_tokens=part, window=window, error_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for name in planes:  # the rows written are the write oracle's, bit for bit
        assert np.array_equal(bits_of(getattr(one, name)), ref[name]), name
    assert torch.equal(out_one.view(torch.int16), out_two.view(torch.int16))  # same plan, same bits
    host = one.to("cpu")
    assert_close(out_one.double().cpu().numpy(), oracle_out(host), f"fused {bits} {D} {N}")


def test_fused_append_skips_and_flags_a_bad_block():
    sp, case, lens, k_new, v_new = setup_fused(16, 128, 2, 4, 2, "bad")
    d = case.to(DEV)
    tb = d.block_tables.clone()
    t_new = lens[1]  # first new row of sequence 1
    tb[1, t_new // sp.block_size] = case.num_blocks + 5
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    snapshot = d.k_pool.clone()
    B.paged_decode_append_attention(d.q, k_new.to(DEV), v_new.to(DEV), d.k_pool, d.v_pool, tb, d.seq_lens,
                                    case.scale, partition_tokens=32, error_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & B.PKV_DEVERR_BAD_BLOCK
    # sequence 1's rows in the bad block were not written anywhere else
    changed = (d.k_pool.view(torch.int16) != snapshot.view(torch.int16)).any(dim=-1).nonzero().tolist()
    good_rows = set()
    for b in range(3):
        for j in range(2):
            t = lens[b] + j
            blk = int(tb[b, t // sp.block_size])
            if blk < case.num_blocks:
                for h in range(2):
                    good_rows.add((blk, h, t % sp.block_size))
    assert {tuple(r) for r in changed} <= good_rows


def test_fused_append_rejects_a_missing_new_row():
    sp, case, lens, k_new, v_new = setup_fused(16, 128, 1, 4, 2, "null")
    d = case.to(DEV)
    with pytest.raises(B.PkvError) as e:
        B.paged_decode_append_attention(d.q, None, v_new.to(DEV), d.k_pool, d.v_pool, d.block_tables, d.seq_lens,
                                        case.scale)
    assert e.value.code == B.PKV_ERR_NULL_POINTER


def _as_tensor(arr, like):
    """A numpy plane from the write oracle as a CPU tensor of `like`'s dtype."""
    if like.dtype == torch.bfloat16:
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(arr).view(np.int32))


@pytest.mark.parametrize("bits,D", [(4, 256), (16, 256), (16, 128)])
def test_back_to_back_fused_steps_read_each_others_rows(bits, D):
    # A decode loop: S fused steps on one stream with no synchronisation between them. Step s
    # appends row L0 + s and attends over L0 + s + 1 rows, the rows earlier steps wrote included.
    # One sequence on a small grid: the partial kernels launch as programmatic dependents of the
    # step before, so this checks that nothing is read before that step has finished.
    S, L0, hq, hk = 4, 700, 8, 2
    name = f"loop_{bits}_{D}"
    seed = zlib.crc32(name.encode()) % 10000
    bs = 16 if bits == 16 else 32
    sp = DecodeSpec(name=name, num_seqs=1, num_q_heads=hq, num_kv_heads=hk, head_dim=D, n_query=1, block_size=bs,
                    bits=bits, length_range=None, lengths=(L0 + S,), pool_factor=2.0, seed=seed)
    case = make_case(sp, lengths=[L0 + S], poison=False)
    g = torch.Generator().manual_seed(seed + 1)
    qs = [torch.randn((1, hq, 1, D), generator=g).to(torch.bfloat16) for _ in range(S)]
    kn = [(torch.randn((1, hk, 1, D), generator=g) * 2).to(torch.bfloat16) for _ in range(S)]
    vn = [torch.randn((1, hk, 1, D), generator=g).to(torch.bfloat16) for _ in range(S)]
    d = case.to(DEV)
    lens = [torch.tensor([L0 + s + 1], dtype=torch.int32, device=DEV) for s in range(S)]
    plan = B.make_plan(B.layout_for(d.k_pool, D, bits), B.DecodeParams(1, hq, 1, d.block_tables.shape[1], 128))
    assert plan.merge_in_cluster == 1 and plan.max_partitions >= 2  # one CTA per SM, cluster merge
    outs = []
    for s in range(S):
        outs.append(B.paged_decode_append_attention(
            qs[s].to(DEV), kn[s].to(DEV), vn[s].to(DEV), d.k_pool, d.v_pool, d.block_tables, lens[s], case.scale,
            bits=bits, k_scales=d.k_scales, k_biases=d.k_biases, v_scales=d.v_scales, v_biases=d.v_biases,
            partition_tokens=128))
    torch.cuda.synchronize()
    planes = ("k_pool", "v_pool") + (() if bits == 16 else ("k_scales", "k_biases", "v_scales", "v_biases"))
    state = {name: bits_of(getattr(case, name)) for name in planes}
    for s in range(S):
        state = pw.append_rows(kn[s].float().numpy(), vn[s].float().numpy(), case.block_tables.numpy(), [L0 + s],
                               state["k_pool"], state["v_pool"], bits=bits, k_scales=state.get("k_scales"),
                               k_biases=state.get("k_biases"), v_scales=state.get("v_scales"),
                               v_biases=state.get("v_biases"))
        host = replace(case, q=qs[s], seq_lens=torch.tensor([L0 + s + 1], dtype=torch.int32), lens_host=[L0 + s + 1],
                       **{name: _as_tensor(state[name], getattr(case, name)) for name in planes})
        assert_close(outs[s].double().cpu().numpy(), oracle_out(host), f"loop step {s} {bits} {D}")
    for name in planes:  # after the loop the pools hold every step's row, bit for bit
        assert np.array_equal(bits_of(getattr(d, name)), state[name]), name
