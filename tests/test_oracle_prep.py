"""Pins for the oracle's preparation stage: K mean, smoothing, INT8 Q/K, FP8 V.

The stage list is from the Experiment Log, "Phase 0 Import And Verification"
(Q/K preparation, K smoothing, INT8 quantization, FP8 V).  Constants and
orders are readings (K-mean chunk order, block sizes 128/64, S_V = 1.125);
these tests check the oracle against hand-derived values, exact rational
arithmetic and properties that any correct implementation of those readings
must have.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import sage_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")
F32 = np.float32


def _gold_k_mean_cases():
    rows = [l.split() for l in open(os.path.join(GOLD, "k_mean_order.txt"))
            if l.strip() and not l.startswith("#")]
    return {r[0]: (int(r[1]), float(r[2])) for r in rows}


def _case_tokens(name, n):
    x = np.ones(n, np.float32)
    if name == "A":
        x[:] = [2.0 ** 24, 1, 1, -(2.0 ** 24)]
    else:
        x[0] = 2.0 ** 24
    return x


@pytest.mark.parametrize("case", ["A", "B", "C"])
def test_k_mean_summation_order_golden(case):
    n, expect = _gold_k_mean_cases()[case]
    x = _case_tokens(case, n)
    k = np.zeros((n, 4), np.float32)
    k[:, 2] = x
    mean = O.k_channel_mean(k, n)
    assert mean[2] == np.float32(expect)
    assert np.all(mean[[0, 1, 3]] == 0)


def test_k_mean_exact_for_small_integers():
    # every partial sum is a small integer -> FP32 sums are exact -> mean is the
    # correctly rounded quotient of the exact sum
    rng = np.random.default_rng(0)
    for n in (1, 5, 63, 64, 65, 200, 777):
        k = rng.integers(-100, 100, (n, 16)).astype(np.float32)
        mean = O.k_channel_mean(k, n)
        exact = k.astype(np.int64).sum(0)
        for d in range(16):
            assert mean[d] == np.float32(Fraction(int(exact[d]), n).__float__()) or \
                abs(Fraction(float(mean[d])) - Fraction(int(exact[d]), n)) <= \
                Fraction(float(np.spacing(mean[d]))) / 2


def test_k_mean_close_to_rational_mean_random():
    rng = np.random.default_rng(1)
    n = 1000
    k = (rng.standard_normal((n, 8)) * 3 + 5).astype(np.float32)
    mean = O.k_channel_mean(k, n)
    for d in range(8):
        exact = sum(Fraction(float(v)) for v in k[:, d]) / n
        # recursive-summation bound: (chunk + chunks) * eps * sum|x| / n
        bound = (64 + n / 64 + 1) * 2.0 ** -24 * float(np.abs(k[:, d]).sum()) / n
        assert abs(float(Fraction(float(mean[d])) - exact)) <= bound


def test_k_mean_ignores_rows_beyond_kv_len_and_handles_empty():
    rng = np.random.default_rng(2)
    k = rng.standard_normal((100, 8)).astype(np.float32)
    k2 = k.copy()
    k2[70:] = 1e30
    assert np.array_equal(O.k_channel_mean(k, 70), O.k_channel_mean(k2, 70))
    assert np.all(O.k_channel_mean(k, 0) == 0)
    # leading axes are independent heads
    kk = np.stack([k, 2 * k])
    m = O.k_channel_mean(kk, 100)
    assert np.array_equal(m[0], O.k_channel_mean(k, 100))
    assert np.array_equal(m[1], O.k_channel_mean(2 * k, 100))


def test_smoothed_keys_have_zero_channel_mean():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 2, 64, 128)).astype(np.float32)
    k = (rng.standard_normal((1, 2, 300, 128)) + rng.standard_normal((1, 2, 1, 128)) * 4).astype(np.float32)
    prep = O.prepare(q, k, k)
    deq = prep.k8.astype(np.float64) * np.repeat(prep.k_scale, 64, axis=-1)[..., :300, None]
    # dequantized smoothed keys average to ~0 per channel (quantization noise only),
    # while the raw keys carry the large offset
    assert np.abs(deq.mean(axis=2)).max() < 0.02
    assert np.abs(k.mean(axis=2)).max() > 1.0
    assert np.allclose(prep.k_mean, k.mean(axis=2), atol=1e-5)


@pytest.mark.parametrize("block", [128, 64])
def test_int8_block_quantization_properties(block):
    rng = np.random.default_rng(4)
    n, valid = 3 * block + 17, 3 * block + 5
    x = (rng.standard_normal((n, 128)) * rng.uniform(0.1, 10, (n, 1))).astype(np.float32)
    codes, scales = O.quantize_int8_blocks(x, valid, block)
    assert codes.dtype == np.int8 and scales.dtype == np.float32
    assert len(scales) == (n + block - 1) // block
    assert np.all(codes[valid:] == 0)
    assert np.all(np.abs(codes.astype(int)) <= 127)
    for b in range((valid + block - 1) // block):
        r0, r1 = b * block, min((b + 1) * block, valid)
        blk = x[r0:r1].astype(np.float64)
        amax = np.abs(blk).max()
        assert scales[b] == np.float32(np.float32(amax) / np.float32(127))
        # the element of largest magnitude maps to +-127
        i = np.unravel_index(np.abs(blk).argmax(), blk.shape)
        assert abs(int(codes[r0:r1][i])) == 127
        # round-to-nearest: dequantized error at most half a step (plus FP32 slack)
        err = np.abs(blk - codes[r0:r1].astype(np.float64) * float(scales[b]))
        assert err.max() <= float(scales[b]) * (0.5 + 1e-5)
    assert np.all(scales[(valid + block - 1) // block:] == 0)


def test_int8_block_boundaries_are_independent():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((256, 128)).astype(np.float32)
    c0, s0 = O.quantize_int8_blocks(x, 256, 64)
    x2 = x.copy()
    x2[130, 7] = 1000.0                                      # row 130 lives in block 2
    c1, s1 = O.quantize_int8_blocks(x2, 256, 64)
    changed = np.flatnonzero(s0 != s1)
    assert list(changed) == [2]
    assert np.array_equal(c0[:128], c1[:128]) and np.array_equal(c0[192:], c1[192:])
    # a huge value in an invalid row changes nothing
    x3 = x.copy()
    x3[200:] = 1e9
    c3, s3 = O.quantize_int8_blocks(x3, 200, 64)
    c4, s4 = O.quantize_int8_blocks(x, 200, 64)
    assert np.array_equal(c3, c4) and np.array_equal(s3, s4)


def test_int8_zero_block_and_ties_to_even():
    x = np.zeros((64, 128), np.float32)
    codes, scales = O.quantize_int8_blocks(x, 64, 64)
    assert np.all(codes == 0) and scales[0] == 0
    # amax 127 -> inv = 1 -> x*inv = x; halves round to even
    x[0, :6] = [127.0, 0.5, 1.5, 2.5, -0.5, -2.5]
    codes, scales = O.quantize_int8_blocks(x, 64, 64)
    assert scales[0] == 1.0
    assert list(codes[0, :6]) == [127, 0, 2, 2, 0, -2]


def test_v_fp8_per_channel_properties():
    rng = np.random.default_rng(6)
    n, valid = 300, 290
    v = (rng.standard_normal((n, 128)) * rng.uniform(0.01, 50, (1, 128))).astype(np.float32)
    v[:, 5] = 0.0                                             # an all-zero channel
    codes, scale = O.quantize_v_fp8(v, valid)
    assert np.all(codes[valid:] == 0)
    assert scale[5] == 0 and np.all(codes[:, 5] == 0)
    dec = O.e4m3_decode(codes[:valid])
    amax = np.abs(v[:valid]).max(0)
    for d in range(128):
        if d == 5:
            continue
        assert scale[d] == np.float32(np.float32(amax[d]) / np.float32(O.S_V))
        # the channel maximum lands on +-1.125 exactly (e4m3 code 0x39/0xB9)
        assert np.abs(dec[:, d]).max() == 1.125
        # e4m3 relative rounding error <= 2^-4 for normals; absolute <= 2^-10 near 0
        x = v[:valid, d].astype(np.float64) * (O.S_V / float(amax[d]))
        err = np.abs(dec[:, d] - x)
        assert np.all(err <= np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10) * (1 + 1e-6))
    # channels are independent: scaling one channel changes only that channel
    v2 = v.copy()
    v2[:, 9] *= 8
    codes2, scale2 = O.quantize_v_fp8(v2, valid)
    assert np.flatnonzero(scale2 != scale).tolist() == [9]
    assert np.array_equal(np.delete(codes2, 9, 1), np.delete(codes, 9, 1))


def test_prepare_shapes_and_varlen_padding():
    rng = np.random.default_rng(8)
    B, H, N = 2, 3, 200
    q = rng.standard_normal((B, H, N, 128)).astype(np.float32)
    k = rng.standard_normal((B, H, N, 128)).astype(np.float32)
    v = rng.standard_normal((B, H, N, 128)).astype(np.float32)
    p = O.prepare(q, k, v, q_len=[200, 77], kv_len=[200, 130])
    assert p.q8.shape == (B, H, N, 128) and p.q_scale.shape == (B, H, 2)
    assert p.k_scale.shape == (B, H, 4) and p.v_scale.shape == (B, H, 128)
    assert np.all(p.q8[1, :, 77:] == 0) and np.all(p.k8[1, :, 130:] == 0)
    assert np.all(p.v8[1, :, 130:] == 0)
    assert np.all(p.q_scale[1, :, 1] == 0) and np.all(p.k_scale[1, :, 3] == 0)
    # a batch item's preparation does not depend on the other item
    p1 = O.prepare(q[1:], k[1:], v[1:], q_len=[77], kv_len=[130])
    assert np.array_equal(p1.k8[0], p.k8[1]) and np.array_equal(p1.k_mean[0], p.k_mean[1])
