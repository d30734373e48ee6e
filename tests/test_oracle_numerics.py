"""Pins for the oracle's bf16 conversion and int4 packing (CPU only)."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import bf16, int4

GOLD = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- bf16

def test_bf16_known_values():
    f = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, np.inf, -np.inf, 0.0, -0.0],
                 dtype=np.float32)
    assert list(bf16.to_bf16(f)) == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x7F80, 0xFF80, 0x0000, 0x8000]
    assert bf16.to_bf16(np.array([np.nan], np.float32))[0] & 0x7FC0 == 0x7FC0


def test_bf16_matches_library_conversion():
    rng = np.random.default_rng(1)
    f = (rng.standard_normal(200_000) * np.exp(rng.uniform(-20, 20, 200_000))).astype(np.float32)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bf16.to_bf16(f), ref)
    back = bf16.bf16_to_f32(ref)
    assert np.array_equal(back, torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_f64_to_bf16_has_no_double_rounding():
    # 1 + 2^-8 + 2^-40 lies above the bf16 midpoint 1 + 2^-8, so it rounds up to 1 + 2^-7;
    # rounding through fp32 first would land exactly on the midpoint and tie to 1.0.
    x = np.array([1.0 + 2 ** -8 + 2 ** -40, 1.0 + 2 ** -8, -(1.0 + 2 ** -8 + 2 ** -40)])
    assert list(bf16.f64_to_bf16(x)) == [0x3F81, 0x3F80, 0xBF81]


# ---------------------------------------------------------------- int4

def test_nibble_order_known_answer():
    codes = np.array([[1, 2, 3, 4, 5, 6, 7, 8] * 8], dtype=np.uint8)
    words = int4.pack_codes(codes)
    assert words.shape == (1, 8)
    assert int(words[0, 0]) == 0x87654321
    assert np.array_equal(int4.unpack_codes(words), codes)


def _exact_groups(rng, rows, groups):
    """Weights w = b + s*q built from bf16 s, b and codes that include 0 and 15."""
    q = rng.integers(0, 16, size=(rows, groups, 64))
    q[:, :, 0] = 0
    q[:, :, 1] = 15
    s = bf16.bf16_to_f32(bf16.to_bf16(rng.uniform(0.05, 0.15, (rows, groups)).astype(np.float32)))
    b = bf16.bf16_to_f32(bf16.to_bf16(rng.uniform(-1.0, -0.5, (rows, groups)).astype(np.float32)))
    w = (b[:, :, None] + s[:, :, None] * q.astype(np.float32)).astype(np.float32)
    # s*q has <= 12 significant bits and |b| ~ |s*q|, so every w is exact in fp32
    assert np.array_equal(w.astype(np.float64), b[:, :, None].astype(np.float64)
                          + s[:, :, None].astype(np.float64) * q)
    return w.reshape(rows, groups * 64), q.reshape(rows, groups * 64), s, b


def test_pack_round_trip_is_exact():
    rng = np.random.default_rng(2)
    w, q, s, b = _exact_groups(rng, 16, 4)
    codes, ps, pb = int4.quantize_groups(w)
    assert np.array_equal(codes, q)
    assert np.array_equal(bf16.bf16_to_f32(ps), s)
    assert np.array_equal(bf16.bf16_to_f32(pb), b)
    assert np.array_equal(int4.dequantize(*int4.pack(w)), w.astype(np.float64))


def test_pack_error_bound():
    rng = np.random.default_rng(3)
    w = (rng.standard_normal((64, 256)) * 0.02).astype(np.float32)
    q, s, b = int4.pack(w)
    what = int4.dequantize(q, s, b)
    g = w.reshape(64, 4, 64).astype(np.float64)
    lo, hi = g.min(2), g.max(2)
    sf, bfv = bf16.bf16_to_f64(s), bf16.bf16_to_f64(b)
    s_exact = (hi - lo) / 15.0
    # half a step of rounding, plus the bias rounding, plus 15 steps of scale rounding
    bound = sf / 2 + np.abs(lo - bfv) + 15 * np.abs(s_exact - sf) + 1e-7
    err = np.abs(w.astype(np.float64) - what).reshape(64, 4, 64).max(2)
    assert np.all(err <= bound)
    codes = int4.unpack_codes(q)
    assert codes.min() == 0 and codes.max() == 15


def test_constant_group_has_zero_scale_and_zero_codes():
    w = np.full((2, 64), 0.375, dtype=np.float32)
    codes, s, b = int4.quantize_groups(w)
    assert np.all(codes == 0)
    assert np.all(s == 0)
    assert np.all(bf16.bf16_to_f32(b) == np.float32(0.375))
    assert np.all(int4.dequantize(*int4.pack(w)) == 0.375)


def test_column_slab_layout_is_a_permutation():
    rng = np.random.default_rng(4)
    w = rng.standard_normal((24, 128)).astype(np.float32)
    q, s, b = int4.pack(w)
    codes = int4.unpack_codes(q)
    q_cs, s_cs, b_cs = int4.to_column_slab(q, s, b)
    assert q_cs.shape == (4, 24, 4) and s_cs.shape == (2, 24)
    for c in range(4):
        for r in range(24):
            for i in range(4):
                for n in range(8):
                    assert (int(q_cs[c, r, i]) >> (4 * n)) & 0xF == codes[r, 32 * c + 8 * i + n]
    assert np.array_equal(s_cs[1, 5], s[5, 1]) and np.array_equal(b_cs[0, 7], b[7, 0])


def test_page_byte_counts():
    g = json.load(open(os.path.join(GOLD, "page_numbers.json")))
    d, F, E, L = g["d"], g["F"], g["E"], g["layers"]
    w_gate = np.zeros((F, d), np.float32)
    w_down = np.zeros((d, F), np.float32)
    nbytes = 0
    for w in (w_gate, w_gate, w_down):
        q, s, b = int4.pack(w)
        nbytes += q.nbytes + s.nbytes + b.nbytes
    assert nbytes == 1_769_472
    assert round(nbytes / 1e6, 2) == g["expert_bytes_MB_printed"]
    assert round(E * nbytes / 1e6) == g["layer_expert_bytes_MB_printed"]
    assert round(L * E * nbytes / 1e9) == g["stack_expert_bytes_GB_printed"]
    assert round(L * E * nbytes / 2 ** 30, 1) == g["stack_expert_bytes_GiB_printed"]
    assert round(4 * nbytes / 1e6) == g["k4_layer_expert_bytes_MB_printed"]
    assert d + 2 * E == g["head_feature_dim_printed"]


@pytest.mark.parametrize("val", [1e-30, 3.0e-3, 7.0])
def test_pack_rounding_of_scale_happens_before_codes(val):
    # A group whose exact step (hi-lo)/15 is not bf16-representable: codes must be
    # chosen against the rounded step, so the top weight may clamp at 15.
    w = np.linspace(0, val, 64, dtype=np.float32)[None, :]
    codes, s, b = int4.quantize_groups(w)
    sf = float(bf16.bf16_to_f32(s)[0, 0])
    bfv = float(bf16.bf16_to_f32(b)[0, 0])
    expect = np.clip(np.rint((w[0] - np.float32(bfv)) / np.float32(sf)), 0, 15)
    assert np.array_equal(codes[0], expect.astype(np.uint8))
