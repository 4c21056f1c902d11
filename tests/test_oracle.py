"""Pins of the CPU oracle against facts the pages and the mathematics fix.

Each test checks the oracle against something other than itself: hand-worked
values of the code layout (tests/golden), closed forms, special cases and an
independent dense formulation run through a library routine
(``torch.nn.functional.scaled_dot_product_attention`` in float64). The
mutation tests at the end plant a plausible mistake in the oracle and check
that one of these pins catches it.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import paged_decode as opd
from quantized_kv_decode_partial_gb300.workloads import DecodeSpec, make_case

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "affine_dequant_pins.json")


# ---------------------------------------------------------------------------
# helpers: case -> numpy inputs, and an independent dense formulation
# ---------------------------------------------------------------------------

def np_inputs(case):
    f64 = lambda t: None if t is None else t.float().double().numpy()
    kw = dict(bits=case.spec.bits, group_size=case.spec.group_size)
    if case.spec.bits == 16:
        kp, vp = f64(case.k_pool), f64(case.v_pool)
    else:
        kp, vp = case.k_pool.numpy(), case.v_pool.numpy()
        kw.update(k_scales=f64(case.k_scales), k_biases=f64(case.k_biases),
                  v_scales=f64(case.v_scales), v_biases=f64(case.v_biases))
    return (f64(case.q), kp, vp, case.block_tables.numpy(), case.seq_lens.numpy(), case.scale,
            case.spec.n_query), kw


def codes_by_bits(words, bits):
    """Codes through numpy.unpackbits: a route that uses no shifts or masks."""
    w = np.ascontiguousarray(np.asarray(words).astype(np.int64) & 0xFFFFFFFF).astype("<u4")
    by = w.view(np.uint8).reshape(w.shape + (4,))
    b = np.unpackbits(by, axis=-1, bitorder="little").reshape(w.shape[:-1] + (w.shape[-1] * 32,))
    b = b.reshape(b.shape[:-1] + (b.shape[-1] // bits, bits)).astype(np.int64)
    return b @ (1 << np.arange(bits, dtype=np.int64))


def dense_reference(case):
    """Dense float64 attention: whole pages picked per block, heads expanded by
    repeat_interleave, an explicit boolean causal-tail mask, and torch's SDPA."""
    s = case.spec
    B, HQ, HK, N, BS, D = s.num_seqs, s.num_q_heads, s.num_kv_heads, s.n_query, s.block_size, s.head_dim
    q = case.q.double()
    outs = []
    for b in range(B):
        L = case.lens_host[b]
        nb = -(-L // BS)
        tbl = case.block_tables[b, :nb].long()

        def pick(plane):
            x = plane[tbl]  # [nb, HK, BS, W]
            return x.permute(1, 0, 2, 3).reshape(HK, nb * BS, x.shape[-1])[:, :L]

        if s.bits == 16:
            K, V = pick(case.k_pool).double(), pick(case.v_pool).double()
        else:
            def deq(words, sc, bi):
                c = torch.from_numpy(codes_by_bits(pick(words).numpy(), s.bits)).double()
                rep = lambda p: pick(p).double().repeat_interleave(s.group_size, dim=-1)
                return c * rep(sc) + rep(bi)
            K = deq(case.k_pool, case.k_scales, case.k_biases)
            V = deq(case.v_pool, case.v_scales, case.v_biases)
        Ke = K.repeat_interleave(HQ // HK, dim=0)
        Ve = V.repeat_interleave(HQ // HK, dim=0)
        i = torch.arange(N)[:, None]
        t = torch.arange(L)[None, :]
        mask = t <= (L - N + i)
        if s.window > 0:  # the W most recent positions of each query, its own included
            mask &= t > (L - N + i - s.window)
        outs.append(torch.nn.functional.scaled_dot_product_attention(
            q[b], Ke, Ve, attn_mask=mask, scale=case.scale).numpy())
    return np.stack(outs)


def tiny(name, **kw):
    base = dict(name=name, num_seqs=2, num_q_heads=4, num_kv_heads=2, head_dim=16, n_query=1,
                block_size=4, bits=16, group_size=8, length_range=(1, 40), pool_factor=2.0, seed=7)
    base.update(kw)
    return DecodeSpec(**base)


TINY = [
    tiny("bf16_bs4"),
    tiny("bf16_bs1_n3", block_size=1, n_query=3, length_range=(3, 20), seed=11),
    tiny("bf16_bs16_rep4", num_q_heads=4, num_kv_heads=1, block_size=16, length_range=(16, 40), seed=12),
    tiny("u4_bs4", bits=4, seed=13),
    tiny("u8_bs4_n2", bits=8, n_query=2, length_range=(2, 33), seed=14),
    tiny("u4_bs16_g16", bits=4, head_dim=32, group_size=16, block_size=16, length_range=(5, 40), seed=15),
    tiny("bf16_window7_n3", n_query=3, window=7, length_range=(3, 40), seed=16),
    tiny("u8_window1_n2", bits=8, n_query=2, window=1, length_range=(2, 30), seed=17),
    # value head dim different from the key head dim (the pages' vHeadDim)
    tiny("bf16_dk16_dv8_n2", v_head_dim=8, n_query=2, length_range=(2, 40), seed=18),
    tiny("u4_dk16_dv32", bits=4, v_head_dim=32, seed=19),
    tiny("u8_dk32_dv16_window5", bits=8, head_dim=32, v_head_dim=16, group_size=16, window=5, seed=20),
]


# ---------------------------------------------------------------------------
# dequantisation and the packed layout
# ---------------------------------------------------------------------------

def test_dequant_golden_values():
    g = json.load(open(GOLDEN))
    for c in g["cases"]:
        words = np.array([[int(w, 16) for w in c["words"]]], dtype=np.int64)
        codes = oracle.unpack_codes(words, c["bits"])[0]
        assert codes.tolist() == c["codes"], c
        n = len(c["codes"])
        vals = oracle.dequantize(words, np.full((1, 1), c["scale"]), np.full((1, 1), c["bias"]),
                                 c["bits"], group_size=n)[0]
        assert vals.tolist() == c["values"], c


def test_dequant_group_index():
    gc = json.load(open(GOLDEN))["group_case"]
    words = np.full((1, gc["n_words"]), int(gc["word"], 16), dtype=np.int64)
    vals = oracle.dequantize(words, np.array([gc["scales"]]), np.array([gc["biases"]]), gc["bits"],
                             gc["group_size"])[0]
    assert vals.shape == (128,)
    assert np.all(vals[:64] == gc["values_group0"]) and np.all(vals[64:] == gc["values_group1"])


@pytest.mark.parametrize("bits", [4, 8])
def test_unpack_matches_bitwise_route(bits):
    rng = np.random.default_rng(3)
    words = rng.integers(0, 1 << 32, size=(5, 3, 16), dtype=np.int64)
    assert np.array_equal(oracle.unpack_codes(words, bits), codes_by_bits(words, bits))
    # int32 bit patterns (how torch stores the words) read the same
    as_i32 = words.astype(np.uint32).view(np.int32)
    assert np.array_equal(oracle.unpack_codes(as_i32, bits), codes_by_bits(words, bits))


def test_straddling_width_rejected():
    with pytest.raises(ValueError):
        oracle.unpack_codes(np.zeros((1, 3), dtype=np.int64), 3)


# ---------------------------------------------------------------------------
# gather
# ---------------------------------------------------------------------------

def test_gather_hand_example():
    NB, HK, BS, W = 3, 2, 2, 3
    pool = np.zeros((NB, HK, BS, W), dtype=np.int64)
    for blk in range(NB):
        for h in range(HK):
            for r in range(BS):
                for c in range(W):
                    pool[blk, h, r, c] = 1000 * blk + 100 * h + 10 * r + c
    got = oracle.gather_pages(pool, [2, 0], 3)
    assert got.shape == (HK, 3, W)
    expect_h1 = [[2100, 2101, 2102], [2110, 2111, 2112], [100, 101, 102]]
    assert got[1].tolist() == expect_h1
    assert got[0, 2].tolist() == [0, 1, 2]


def test_gather_is_bit_exact_for_nan_payloads():
    pool = np.arange(2 * 1 * 4 * 2, dtype=np.uint16).reshape(2, 1, 4, 2)
    pool[1, 0, 3, 1] = 0x7FC1  # a NaN payload survives untouched
    got = oracle.gather_pages(pool, [1, 0], 6)
    assert got.dtype == np.uint16 and got[0, 3, 1] == 0x7FC1 and got[0, 4].tolist() == [0, 1]


# ---------------------------------------------------------------------------
# softmax, closed forms and special cases
# ---------------------------------------------------------------------------

def test_softmax_weights_sum_to_one_and_shift_invariant():
    rng = np.random.default_rng(0)
    for s in [rng.normal(size=50), rng.normal(size=7) * 1e3, np.array([-1e300, 0.0, 5.0])]:
        p = oracle.softmax_weights(s)
        assert abs(p.sum() - 1.0) < 1e-12 and np.all(p >= 0)
        assert np.allclose(p, oracle.softmax_weights(s + 123.0), rtol=0, atol=1e-15)


def test_two_key_closed_form():
    x = 0.7
    q = np.array([1.0, 0.0])
    K = np.array([[0.0, 5.0], [x, -2.0]])
    V = np.array([[4.0, 1.0], [-2.0, 3.0]])
    p1 = math.exp(x) / (1.0 + math.exp(x))
    expect = (1 - p1) * V[0] + p1 * V[1]
    assert np.allclose(oracle.attend(q, K, V, 1.0), expect, rtol=0, atol=1e-15)


@pytest.mark.parametrize("bits,dv", [(16, 0), (4, 0), (16, 24), (8, 8)])
def test_one_token_cache_returns_its_v_row(bits, dv):
    spec = tiny("one", num_seqs=1, lengths=(1,), length_range=None, bits=bits, seed=21, v_head_dim=dv)
    case = make_case(spec)
    args, kw = np_inputs(case)
    out = oracle.paged_decode_attention(*args, **kw)
    phys = case.tables_host[0][0]
    for h in range(spec.num_q_heads):
        kv = h // spec.rep
        if bits == 16:
            row = case.v_pool[phys, kv, 0].double().numpy()
        else:
            row = oracle.dequantize(case.v_pool[phys, kv, 0].numpy(), case.v_scales[phys, kv, 0].double().numpy(),
                                    case.v_biases[phys, kv, 0].double().numpy(), bits, spec.group_size)
        assert np.array_equal(out[0, h, 0], row)


def test_identical_keys_and_zero_scale_give_mean_of_v():
    spec = tiny("ident", num_seqs=1, lengths=(29,), length_range=None, n_query=2, seed=22)
    case = make_case(spec, poison=False)
    case.k_pool[:] = case.k_pool[0, :, :1, :]  # every key row equal
    args, kw = np_inputs(case)
    out = oracle.paged_decode_attention(*args, **kw)
    zero = oracle.paged_decode_attention(*args[:5], 0.0, args[6], **kw)
    V = oracle.gather_pages(case.v_pool.double().numpy(), case.tables_host[0], 29)
    for h in range(spec.num_q_heads):
        for i in range(2):
            T = 29 - 2 + i + 1
            mean = V[h // spec.rep, :T].mean(axis=0)
            assert np.max(np.abs(out[0, h, i] - mean)) < 1e-12
            assert np.max(np.abs(zero[0, h, i] - mean)) < 1e-12


def test_window_of_one_returns_the_own_row_and_a_wide_window_changes_nothing():
    spec = tiny("win", num_seqs=2, n_query=3, length_range=(5, 40), seed=23)
    case = make_case(spec)
    args, kw = np_inputs(case)
    own = oracle.paged_decode_attention(*args, window=1, **kw)
    for b in range(2):
        L = case.lens_host[b]
        V = oracle.gather_pages(case.v_pool.double().numpy(), case.tables_host[b], L)
        for h in range(spec.num_q_heads):
            for i in range(3):
                assert np.array_equal(own[b, h, i], V[h // spec.rep, L - 3 + i])
    full = oracle.paged_decode_attention(*args, **kw)
    wide = oracle.paged_decode_attention(*args, window=max(case.lens_host), **kw)
    assert np.array_equal(full, wide)


# ---------------------------------------------------------------------------
# partitions and the log-sum-exp merge
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("spec", [TINY[1], TINY[4], TINY[6]], ids=lambda s: s.name)
def test_merge_equals_unsplit_for_every_partition_size(spec):
    case = make_case(spec)
    args, kw = np_inputs(case)
    kw["window"] = spec.window
    whole = oracle.paged_decode_attention(*args, **kw)
    Lmax = max(case.lens_host)
    for P in list(range(1, 9)) + [13, Lmax, Lmax + 5]:
        split = oracle.paged_decode_attention_partitioned(*args, P, **kw)
        rel = np.max(np.abs(split - whole) / (np.abs(whole) + 1e-300))
        assert rel < 1e-12, (P, rel)


def test_lse_merge_skips_empty_partitions():
    st = [(-math.inf, 0.0, np.zeros(2)), (0.5, 2.0, np.array([2.0, 4.0])), (-math.inf, 0.0, np.zeros(2))]
    assert np.array_equal(oracle.lse_merge(st), np.array([1.0, 2.0]))
    with pytest.raises(ValueError):
        oracle.lse_merge(st[:1])


# ---------------------------------------------------------------------------
# brute force against a library routine, invariances, stale storage
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("spec", TINY, ids=lambda s: s.name)
def test_matches_dense_sdpa(spec):
    case = make_case(spec)
    args, kw = np_inputs(case)
    got = oracle.paged_decode_attention(*args, window=spec.window, **kw)
    ref = dense_reference(case)
    assert np.isfinite(got).all()  # poisoned stale rows and blocks were never read
    assert np.max(np.abs(got - ref)) < 1e-12


@pytest.mark.parametrize("spec", [TINY[0], TINY[4]], ids=lambda s: s.name)
def test_physical_block_permutation_invariance(spec):
    case = make_case(spec)
    args, kw = np_inputs(case)
    base = oracle.paged_decode_attention(*args, **kw)
    rng = np.random.default_rng(5)
    perm = rng.permutation(case.num_blocks)  # new slot of old block j is perm[j]
    inv = np.argsort(perm)
    planes = [args[1], args[2]] + [kw[k] for k in ("k_scales", "k_biases", "v_scales", "v_biases") if k in kw]
    moved = [p[inv] for p in planes]
    tables = args[3].copy()
    tables[tables >= 0] = perm[tables[tables >= 0]]
    kw2 = dict(kw)
    if case.spec.bits != 16:
        kw2.update(k_scales=moved[2], k_biases=moved[3], v_scales=moved[4], v_biases=moved[5])
    out = oracle.paged_decode_attention(args[0], moved[0], moved[1], tables, *args[4:], **kw2)
    assert np.array_equal(out, base)


def test_rows_subset_matches_full():
    case = make_case(TINY[4])
    args, kw = np_inputs(case)
    full = oracle.paged_decode_attention(*args, **kw)
    sub = oracle.paged_decode_attention(*args, rows=[(1, 3), (0, 0)], **kw)
    assert np.array_equal(sub[1, 3], full[1, 3]) and np.array_equal(sub[0, 0], full[0, 0])
    assert np.isnan(sub[0, 1]).all()


def test_short_sequence_rejected():
    spec = tiny("short", num_seqs=1, lengths=(2,), length_range=None, n_query=3)
    case = make_case(spec, lengths=[2])
    args, kw = np_inputs(case)
    with pytest.raises(ValueError):
        oracle.paged_decode_attention(*args, **kw)


# ---------------------------------------------------------------------------
# mutation tests: a planted mistake must fail a pin
# ---------------------------------------------------------------------------

def _pins_fail(monkeypatch, name, mutant):
    monkeypatch.setattr(opd, name, mutant)
    failures = 0
    for spec in TINY:
        case = make_case(spec)
        args, kw = np_inputs(case)
        try:
            got = opd.paged_decode_attention(*args, window=spec.window, **kw)
        except (ValueError, IndexError):  # e.g. K and V planes of different head dims exchanged
            failures += 1
            continue
        ref = dense_reference(case)
        if got.shape != ref.shape or not (np.isfinite(got).all() and np.max(np.abs(got - ref)) < 1e-12):
            failures += 1
    return failures


def test_mutant_high_nibble_first_is_caught(monkeypatch):
    real = opd.unpack_codes

    def mutant(words, bits):
        c = real(words, bits)
        pack = 32 // bits
        return c.reshape(c.shape[:-1] + (-1, pack))[..., ::-1].reshape(c.shape)

    assert _pins_fail(monkeypatch, "unpack_codes", mutant) > 0
    g = json.load(open(GOLDEN))["cases"][0]
    assert mutant(np.array([[int(g["words"][0], 16)]]), 4)[0].tolist() != g["codes"]


def test_mutant_group_index_modulo_is_caught(monkeypatch):
    def mutant(words, scales, biases, bits, group_size):
        codes = opd.unpack_codes(words, bits).astype(np.float64)
        G = np.asarray(scales).shape[-1]
        g = np.arange(codes.shape[-1]) % G
        return np.asarray(scales)[..., g] * codes + np.asarray(biases)[..., g]

    assert _pins_fail(monkeypatch, "dequantize", mutant) > 0


def test_mutant_softmax_without_max_is_caught():
    def mutant(s):
        e = np.exp(np.asarray(s, dtype=np.float64))
        return e / e.sum()
    s = np.array([1000.0, 999.0])
    with np.errstate(over="ignore", invalid="ignore"):
        bad = mutant(s)
    assert not (np.isfinite(bad).all() and abs(bad.sum() - 1) < 1e-12)


def test_mutant_head_map_and_causal_offset_are_caught(monkeypatch):
    real = opd.attend

    def shifted(q, K, V, scale):  # drops the newest visible key (off-by-one causal end)
        return real(q, K[:-1], V[:-1], scale) if len(K) > 1 else real(q, K, V, scale)

    assert _pins_fail(monkeypatch, "attend", shifted) > 0
    monkeypatch.setattr(opd, "attend", real)

    real_kv = opd._sequence_kv

    def swapped(k_pool, v_pool, *a, **k):  # K and V planes exchanged
        return real_kv(v_pool, k_pool, *a, **k)

    assert _pins_fail(monkeypatch, "_sequence_kv", swapped) > 0
    monkeypatch.setattr(opd, "_sequence_kv", real_kv)

    def interleaved(h, num_q_heads, num_kv_heads):  # head h served by KV head h % HK
        return h % num_kv_heads

    assert _pins_fail(monkeypatch, "kv_head", interleaved) > 0
    monkeypatch.setattr(opd, "kv_head", lambda h, q, k: h // (q // k))

    real_range = opd.visible_range

    def window_too_wide(length, n_query, i, window=0):  # one extra row below the window
        lo, hi = real_range(length, n_query, i, window)
        return (max(0, lo - 1) if window > 0 else lo), hi

    assert _pins_fail(monkeypatch, "visible_range", window_too_wide) > 0
