"""Pins for the oracle's number formats: OCP E4M3, BF16, FP16, exp2.

Each conversion written from its definition in ``oracle/`` is checked here
against something other than itself: the OCP table's landmark values, torch's
own float8/bfloat16 casts, and Python's correctly rounded binary16 packing.
"""
import math
import os
import struct

import numpy as np
import pytest
import torch

from oracle import sage_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _torch_e4m3_bytes(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def test_e4m3_decode_all_256_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    mine = O.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().double().numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])
    assert np.array_equal(np.signbit(mine[ok]), np.signbit(ref[ok]))
    assert set(np.flatnonzero(np.isnan(mine))) == {0x7F, 0xFF}


def test_e4m3_ocp_landmarks():
    rows = [l.split() for l in open(os.path.join(GOLD, "e4m3_ocp_landmarks.txt"))
            if l.strip() and not l.startswith("#")]
    for hexcode, val in rows:
        c = int(hexcode, 16)
        v = float(val)
        assert O.e4m3_decode(np.array([c], np.uint8))[0] == v
        assert math.copysign(1, O.e4m3_decode(np.array([c], np.uint8))[0]) == math.copysign(1, v)
        assert int(O.e4m3_encode(np.array([v]))[0]) == c


def test_e4m3_encode_roundtrips_every_finite_code():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    assert np.array_equal(O.e4m3_encode(O.e4m3_decode(codes)), codes)


def test_e4m3_encode_midpoints_and_neighbours_match_torch():
    mags = np.sort(np.unique(np.abs(O.e4m3_decode(np.arange(127, dtype=np.uint8)))))
    mids = (mags[:-1] + mags[1:]) / 2                        # exact ties (float32-exact)
    xs = np.concatenate([mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
                         np.nextafter(mids.astype(np.float32), np.float32(1e9)), mags])
    xs = np.concatenate([xs, -xs]).astype(np.float32)
    assert np.array_equal(O.e4m3_encode(xs), _torch_e4m3_bytes(xs))


def test_e4m3_encode_random_matches_torch():
    rng = np.random.default_rng(7)
    x = (rng.choice([-1, 1], 400_000) * np.exp2(rng.uniform(-14, 8.85, 400_000))).astype(np.float32)
    x = x[np.abs(x) < 464]                                   # torch turns >= 464 into NaN
    assert np.array_equal(O.e4m3_encode(x), _torch_e4m3_bytes(x))


def test_e4m3_encode_saturates_to_448():
    big = np.array([448.0, 463.9, 464.0, 480.0, 1e6, 3.4e38, np.inf], np.float64)
    assert np.all(O.e4m3_encode(big) == 0x7E)
    assert np.all(O.e4m3_encode(-big) == 0xFE)
    assert O.e4m3_encode(np.array([np.nan]))[0] == 0x7F


def test_bf16_rne_matches_torch():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(200_000).astype(np.float32) * np.float32(37.0)
    # exact ties: low 16 bits == 0x8000 with both parities of the kept LSB
    u = rng.integers(0x3F000000, 0x47000000, 20_000, dtype=np.uint64).astype(np.uint32)
    ties = ((u & np.uint32(0xFFFF0000)) | np.uint32(0x8000)).view(np.float32)
    x = np.concatenate([x, ties, -ties])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.uint16).numpy()
    assert np.array_equal(O.f32_to_bf16_bits(x), ref)
    back = O.bf16_bits_to_f32(ref)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_f16_round_matches_correctly_rounded_pack():
    # struct's 'e' format rounds a double to binary16 directly (ties to even).
    rng = np.random.default_rng(11)
    x = rng.standard_normal(20_000) * 3000.0
    halfs = np.array([struct.unpack("<e", struct.pack("<e", v))[0] for v in x])
    assert np.array_equal(O.f16_round(x), halfs)
    # ties between neighbouring halves: 1 + 2^-11 lies between 1 and 1 + 2^-10
    ties = np.array([1 + 2 ** -11, 1 + 3 * 2 ** -11, 2048 + 1.0, 2048 + 3.0])
    tie_ref = np.array([struct.unpack("<e", struct.pack("<e", v))[0] for v in ties])
    assert np.array_equal(O.f16_round(ties), tie_ref)
    assert list(tie_ref) == [1.0, 1 + 2 ** -9, 2048.0, 2052.0]


def test_exp2_f32_integer_and_fractional_arguments():
    ints = np.arange(-126, 128, dtype=np.float32)
    assert np.array_equal(O.exp2_f32(ints), np.ldexp(np.float32(1), ints.astype(int)).astype(np.float32))
    x = np.array([-0.5, 0.5, -3.25, 8.807354922057604], np.float32)
    ref = np.array([np.float32(math.pow(2.0, float(v))) for v in x], np.float32)
    assert np.array_equal(O.exp2_f32(x), ref)
    assert O.exp2_f32(np.array([-np.inf], np.float32))[0] == 0.0


@pytest.mark.parametrize("val,code", [(1.125, 0x39), (-1.125, 0xB9), (0.0625, 0x18)])
def test_e4m3_spot_values(val, code):
    assert O.e4m3_encode(np.array([val]))[0] == code
