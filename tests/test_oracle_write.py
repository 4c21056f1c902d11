"""Pins of the write-side oracle (affine quantise-on-append and row placement)."""

import numpy as np
import pytest

import oracle
from oracle import paged_write as pw


def test_bf16_round_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9, 1.0 + 2 ** -9, -3.0 - 2 ** -8, 65504.0], dtype=np.float32)
    got = pw.bf16_round(x)
    # 1 + 2^-8 is half way between 1 and 1 + 2^-7: ties go to the even mantissa (1.0)
    assert got.tolist() == [1.0, 1.0, 1.0 + 2 ** -7, 1.0, -3.0, 65536.0]
    assert np.isnan(pw.bf16_round(np.array([np.nan], dtype=np.float32))).all()


def test_exact_4bit_grid():
    k = np.tile(np.arange(16), 4)
    x = (1.0 + 0.5 * k).astype(np.float32)[None]  # one 64-dim group on an exact grid
    codes, scale, bias = pw.quantize_groups(x, 4)
    assert scale.tolist() == [[0.5]] and bias.tolist() == [[1.0]]
    assert codes[0].tolist() == k.tolist()


def test_exact_8bit_grid():
    c = np.array([4 * j for j in range(63)] + [255])
    x = (0.125 * c).astype(np.float32)[None]
    codes, scale, bias = pw.quantize_groups(x, 8)
    assert scale.tolist() == [[0.125]] and bias.tolist() == [[0.0]]
    assert codes[0].tolist() == c.tolist()


@pytest.mark.parametrize("bits", [4, 8])
def test_error_bound_and_extremes(bits):
    rng = np.random.default_rng(bits)
    x = pw.bf16_round(rng.normal(size=(50, 256)).astype(np.float32) * rng.uniform(0.01, 30, size=(50, 1)))
    codes, scale, bias = pw.quantize_groups(x, bits)
    levels = (1 << bits) - 1
    g = x.reshape(50, 4, 64)
    c = codes.reshape(50, 4, 64)
    deq = scale[..., None].astype(np.float64) * c + bias[..., None]
    lo = g.min(-1, keepdims=True)
    # half a step, plus what bf16 rounding of the scale (over all levels) and the bias can add
    bound = 0.5 * scale[..., None] + levels * 2.0 ** -8 * scale[..., None] + 2.0 ** -8 * np.abs(lo)
    assert np.all(np.abs(deq - g) <= bound * (1 + 1e-6))
    assert np.all(c[np.arange(50)[:, None], np.arange(4)[None], g.argmin(-1)] == 0)
    # the group's largest value takes the top code; with 8 bits a bf16 scale rounded up by up to
    # 2^-8 can leave it one step below (255 / (1 + 2^-8) rounds to 254)
    top = c[np.arange(50)[:, None], np.arange(4)[None], g.argmax(-1)]
    assert np.all(top == levels) if bits == 4 else np.all(top >= levels - 1)
    assert codes.min() >= 0 and codes.max() <= levels


def test_constant_group_is_exact():
    x = np.full((2, 128), 0.75, dtype=np.float32)
    codes, scale, bias = pw.quantize_groups(x, 4)
    assert not codes.any() and not scale.any() and np.all(bias == 0.75)


@pytest.mark.parametrize("bits", [4, 8])
def test_pack_round_trip_and_layout(bits):
    rng = np.random.default_rng(7)
    codes = rng.integers(0, 1 << bits, size=(3, 128))
    words = pw.pack_codes(codes, bits)
    assert np.array_equal(oracle.unpack_codes(words, bits), codes)
    if bits == 4:
        assert pw.pack_codes(np.arange(8)[None], 4).tolist() == [[0x76543210]]
    else:
        assert pw.pack_codes(np.array([[0, 1, 2, 3]]), 8).tolist() == [[0x03020100]]


def test_append_places_rows_by_block_table():
    NB, HK, BS, D = 3, 2, 4, 64
    pool = np.zeros((NB, HK, BS, D), dtype=np.uint16)
    rows = pw.bf16_round(np.arange(2 * HK * 2 * D, dtype=np.float32).reshape(2, HK, 2, D) / 8)
    # two sequences: lengths 3 and 0, tables [2, 0] and [1]
    tables = np.array([[2, 0], [1, 1]])
    out = pw.append_rows(rows, rows, tables, [3, 0], pool, pool)
    got = out["k_pool"]
    assert np.array_equal(got[2, :, 3], pw.bf16_bits(rows[0, :, 0]))  # position 3 -> block 2 row 3
    assert np.array_equal(got[0, :, 0], pw.bf16_bits(rows[0, :, 1]))  # position 4 -> block 0 row 0
    assert np.array_equal(got[1, :, 0], pw.bf16_bits(rows[1, :, 0]))
    assert np.array_equal(got[1, :, 1], pw.bf16_bits(rows[1, :, 1]))
    assert int((got != 0).any(axis=-1).sum()) == 4 * HK


def test_append_then_dequantise_reads_back_the_rows():
    rng = np.random.default_rng(3)
    NB, HK, BS, D, bits = 4, 2, 32, 128, 4
    words = np.zeros((NB, HK, BS, D * bits // 32), dtype=np.int32)
    planes = {k: np.zeros((NB, HK, BS, D // 64), dtype=np.uint16) for k in ("ks", "kb", "vs", "vb")}
    rows = pw.bf16_round(rng.normal(size=(1, HK, 3, D)).astype(np.float32))
    out = pw.append_rows(rows, rows, np.array([[3, 1]]), [31], words, words, bits=bits,
                         k_scales=planes["ks"], k_biases=planes["kb"], v_scales=planes["vs"], v_biases=planes["vb"])
    f = lambda u: (u.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    back = oracle.dequantize(out["k_pool"][3, :, 31], f(out["k_scales"][3, :, 31]), f(out["k_biases"][3, :, 31]), bits, 64)
    codes, sc, bi = pw.quantize_groups(rows[0, :, 0], bits)
    assert np.array_equal(back, sc.repeat(64, -1).astype(np.float64) * codes + bi.repeat(64, -1))
    assert np.max(np.abs(back - rows[0, :, 0])) <= 0.6 * sc.max()
