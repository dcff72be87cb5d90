"""Pins for the oracle's E4M3 codec and fp8 cache write (CPU only)."""
import numpy as np
import pytest
import torch

from oracle.fp8 import (dequantize_ref, e4m3_decode, e4m3_encode,
                        quantize_ref, reshape_and_cache_fp8_ref,
                        scaled_fp8_quant_ref)


def test_decode_matches_torch_float8_e4m3fn():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).float().double().numpy()
    got = e4m3_decode(np.arange(256))
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.nanmax(got) == 448.0 and np.nanmin(got) == -448.0
    assert e4m3_decode([1])[0] == 2.0 ** -9        # smallest subnormal


def test_round_trip_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    assert np.array_equal(e4m3_encode(e4m3_decode(codes)), codes)


def test_encode_matches_torch_cast_in_range():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * s
                        for s in (1e-3, 0.05, 1, 30, 200)])
    x = x[np.abs(x) < 440].astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8)
    assert np.array_equal(e4m3_encode(x.astype(np.float64)), ref.numpy())


def test_ties_saturation_and_specials():
    # 1.0625 lies halfway between 1.0 (code 0x38) and 1.125 (0x39): even
    assert e4m3_encode([1.0625])[0] == 0x38
    assert e4m3_encode([1.1875])[0] == 0x3A        # between 0x39 and 0x3A
    assert e4m3_encode([1e6, -1e6]).tolist() == [0x7E, 0xFE]
    assert e4m3_encode([464.0])[0] == 0x7E         # beyond 448 saturates
    assert e4m3_encode([np.nan])[0] == 0x7F
    assert e4m3_encode([-0.0])[0] == 0x80
    assert e4m3_encode([2.0 ** -10])[0] == 0x00     # halfway to 2^-9: even


def test_quantize_divides_in_float32():
    x = np.float32(0.3)
    s = np.float32(0.7)
    assert quantize_ref([x], s)[0] == e4m3_encode([np.float64(x / s)])[0]


def test_fp8_cache_write_round_trip_within_half_ulp():
    rng = np.random.default_rng(1)
    NB, BS, H, D, T = 6, 16, 2, 32, 40
    key = rng.standard_normal((T, H, D)).astype(np.float32)
    val = rng.standard_normal((T, H, D)).astype(np.float32)
    slots = rng.permutation(NB * BS)[:T]
    kc = np.zeros((NB, BS, H, D), np.uint8)
    vc = np.zeros_like(kc)
    reshape_and_cache_fp8_ref(key, val, kc, vc, slots, 0.02, 0.05)
    flat = kc.reshape(NB * BS, H, D)
    back = e4m3_decode(flat[slots]) * 0.02
    rel = np.abs(back - key) / np.maximum(np.abs(key), 2.0 ** -6 * 0.02)
    assert rel.max() <= 2.0 ** -4 + 1e-9            # 3 mantissa bits


def test_scaled_fp8_quant_hand_values():
    # quotients 0.6, -3.4, 1000, 0 (scale 0.5): 0.6 is nearer 0.625 (0x32)
    # than 0.5625; 3.4 nearer 3.5 (0x46) than 3.25; 1000 saturates to 448
    codes = scaled_fp8_quant_ref([[0.3, -1.7], [500.0, 0.0]], 0.5)
    assert codes.tolist() == [[0x32, 0xC6], [0x7E, 0x00]]
    assert e4m3_decode([0x32, 0xC6]).tolist() == [0.625, -3.5]


def test_scaled_fp8_quant_keeps_shape_and_reads_back():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((5, 4, 32)).astype(np.float32)
    s = 0.01
    codes = scaled_fp8_quant_ref(q, s)
    assert codes.shape == q.shape and codes.dtype == np.uint8
    flat = scaled_fp8_quant_ref(q.reshape(5, 128), s)
    assert np.array_equal(codes.reshape(5, 128), flat)
    back = dequantize_ref(codes, s)
    rel = np.abs(back - q) / np.maximum(np.abs(q), 2.0 ** -6 * s)
    assert rel.max() <= 2.0 ** -4 + 1e-9            # 3 mantissa bits
    # the read-back value is the code's value times the float32 scale
    assert back[0, 0, 0] == e4m3_decode([codes[0, 0, 0]])[0] * \
        np.float64(np.float32(s))
