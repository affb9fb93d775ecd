"""Pins for the oracle's element-format decoders and its E4M3 encoder.

Each decoder is checked over every code against an independent library
conversion (numpy binary16, torch bfloat16 and float8_e4m3fn); the encoder is
checked against torch's conversion and against properties of round-to-nearest
that hold whatever the implementation.
"""
import numpy as np
import torch


def _same(a, b):
    return np.array_equal(np.isnan(a), np.isnan(b)) and np.array_equal(a[~np.isnan(a)], b[~np.isnan(b)])


def test_f16_decode_all_codes(oracle_mod):
    codes = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle_mod.decode_elements(codes, oracle_mod.F16)
    want = codes.view(np.float16).astype(np.float64)
    assert _same(got, want)


def test_bf16_decode_all_codes(oracle_mod):
    codes = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle_mod.decode_elements(codes, oracle_mod.BF16)
    want = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert _same(got, want)


def test_e4m3_decode_all_codes(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    got = oracle_mod.decode_elements(codes, oracle_mod.E4M3)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert _same(got, want)
    # format facts: largest finite 448, smallest subnormal 2^-9, one NaN code per sign
    assert np.nanmax(got) == 448.0 and got[1] == 2.0 ** -9
    assert np.isnan(got).sum() == 2 and np.isnan(got[0x7F]) and np.isnan(got[0xFF])


def test_e4m3_encode_round_trip(oracle_mod):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle_mod.decode_elements(codes, oracle_mod.E4M3).astype(np.float32)
    assert np.array_equal(oracle_mod.e4m3_encode(vals), codes)


def test_e4m3_encode_matches_torch(oracle_mod):
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(200_000).astype(np.float32) * np.float32(60.0),
        rng.standard_normal(50_000).astype(np.float32) * np.float32(0.01),
        (rng.uniform(-500, 500, 50_000)).astype(np.float32),
    ])
    # exact midpoints between neighbouring codes: ties go to the even code
    pos = oracle_mod.decode_elements(np.arange(0, 0x7F, dtype=np.uint8), oracle_mod.E4M3)
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids])
    got = oracle_mod.e4m3_encode(x)
    want = torch.from_numpy(x).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, want)


def test_e4m3_encode_is_nearest(oracle_mod):
    """Whatever the tie rule, the chosen code is a nearest finite value."""
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(20_000) * 30).astype(np.float32)
    got = oracle_mod.decode_elements(oracle_mod.e4m3_encode(x), oracle_mod.E4M3)
    table = oracle_mod.decode_elements(np.arange(256, dtype=np.uint8), oracle_mod.E4M3)
    table = table[~np.isnan(table)]
    best = np.min(np.abs(table[None, :] - x[:, None].astype(np.float64)), axis=1)
    assert np.array_equal(np.abs(got - x.astype(np.float64)), best)


def test_e4m3_encode_saturates_and_nan(oracle_mod):
    x = np.array([448.0, 449.0, 464.0, 1e30, np.inf, -np.inf, -1e30, np.nan, 0.0, -0.0], np.float32)
    got = oracle_mod.e4m3_encode(x)
    assert list(got) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F, 0x00, 0x80]
