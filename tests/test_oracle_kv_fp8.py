"""Pins for the oracle's E4M3 key / value cache (oracle/kv_fp8.py): hand-worked
codes from the format's definition, every finite code round-tripped, the
rounding rule at midpoints (ties to the even mantissa) and at saturation,
agreement with a library conversion (PyTorch's float8_e4m3fn), the relative
error bound of a round trip, and the page scales on a hand-made cache."""

import numpy as np
import pytest
import torch

from oracle.kv_fp8 import (E4M3_MAX, dequantize_cache, e4m3_decode, e4m3_encode, page_scales,
                           quantize_cache, tree_attention_fp8)
from oracle.tree_attn import tree_attention


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x80, -0.0), (0x38, 1.0), (0xB8, -1.0), (0x40, 2.0), (0x3C, 1.5),
    (0x7E, 448.0), (0xFE, -448.0), (0x08, 2.0 ** -6), (0x07, 7 * 2.0 ** -9),
    (0x01, 2.0 ** -9), (0x30, 0.5), (0x39, 1.125), (0x50, 8.0),
])
def test_hand_worked_codes(code, value):
    # value = (1 + m/8) 2^(e-7), or m/8 2^-6 for e = 0
    assert e4m3_decode(np.array([code]))[0] == value
    if value != 0.0 or code == 0x00:
        assert e4m3_encode(np.array([value]))[0] == code


def test_nan_codes_and_saturation():
    assert np.isnan(e4m3_decode(np.array([0x7F, 0xFF]))).all()
    assert e4m3_encode(np.array([1e6]))[0] == 0x7E
    assert e4m3_encode(np.array([-500.0]))[0] == 0xFE
    assert e4m3_encode(np.array([464.0]))[0] == 0x7E     # past the top: saturate


def test_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F and c != 0x80], dtype=np.uint8)
    assert np.array_equal(e4m3_encode(e4m3_decode(codes)), codes)


def test_midpoints_round_to_even_mantissa():
    # between 1.0 (0x38, mantissa 0) and 1.125 (0x39, mantissa 1): 1.0625 -> 1.0;
    # between 1.125 and 1.25 (0x3A): 1.1875 -> 1.25 (mantissa 2 is even)
    assert e4m3_encode(np.array([1.0625]))[0] == 0x38
    assert e4m3_encode(np.array([1.1875]))[0] == 0x3A
    # a hair off the midpoint goes to the nearer one
    assert e4m3_encode(np.array([1.0626]))[0] == 0x39
    # subnormal midpoint 1.5 * 2^-9 between 0x01 and 0x02: even mantissa 2
    assert e4m3_encode(np.array([1.5 * 2.0 ** -9]))[0] == 0x02


def test_agrees_with_pytorch_float8_e4m3fn():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * 50, rng.standard_normal(5000) * 0.01,
                        rng.uniform(-448, 448, 5000)])
    ours = e4m3_encode(x)
    lib = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, lib)
    assert np.array_equal(e4m3_decode(ours),
                          torch.from_numpy(ours).view(torch.float8_e4m3fn).to(torch.float64).numpy())


def test_round_trip_error_bound():
    # normal range: half a unit in the last place, |err| <= 2^-4 |x|;
    # subnormal range: |err| <= 2^-10 (half the spacing 2^-9)
    rng = np.random.default_rng(1)
    x = rng.uniform(-448, 448, 100000)
    err = np.abs(e4m3_decode(e4m3_encode(x)) - x)
    normal = np.abs(x) >= 2.0 ** -6
    assert (err[normal] <= 2.0 ** -4 * np.abs(x[normal])).all()
    assert (err[~normal] <= 2.0 ** -10).all()


def test_page_scales_and_cache_round_trip():
    x = np.zeros((2, 300, 4))
    x[0, 5, 1] = 8.96                      # page 0 of head 0: amax 8.96
    x[0, 200, 2] = -4.48                   # page 1 of head 0
    x[1, 299, 3] = 44.8                    # page 2 of head 1; head 1 pages 0, 1 empty
    s = page_scales(x)
    assert s.shape == (2, 3)
    np.testing.assert_allclose(s[0], [8.96 / 448, 4.48 / 448, 1.0])
    np.testing.assert_allclose(s[1], [1.0, 1.0, 44.8 / 448])
    codes = quantize_cache(x, s)
    assert codes[0, 5, 1] == 0x7E and codes[0, 200, 2] == 0xFE and codes[1, 299, 3] == 0x7E
    np.testing.assert_allclose(dequantize_cache(codes, s), x, rtol=0, atol=1e-12)


def test_fp8_attention_is_the_definition_on_decoded_values():
    rng = np.random.default_rng(2)
    m, hq, hkv, d, S = 5, 4, 2, 16, 260
    parents = [-1, 0, 0, 1, 2]
    mask = np.zeros((m, 1), dtype=np.uint64)
    for i in range(m):
        if i:
            mask[i] = mask[parents[i]]
        mask[i, 0] |= np.uint64(1) << np.uint64(i)
    kx, vx = rng.standard_normal((hkv, S, d)), rng.standard_normal((hkv, S, d))
    ks, vs = page_scales(kx), page_scales(vx)
    kc, vc = quantize_cache(kx, ks), quantize_cache(vx, vs)
    q = rng.standard_normal((m, hq, d))
    tk, tv = rng.standard_normal((m, hkv, d)), rng.standard_normal((m, hkv, d))
    got = tree_attention_fp8(q, kc, ks, vc, vs, tk, tv, mask, S)
    want = tree_attention(q, dequantize_cache(kc, ks), dequantize_cache(vc, vs), tk, tv, mask, S)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)
    # and close to the unquantized attention (E4M3 keeps 3 mantissa bits)
    assert np.abs(got - tree_attention(q, kx, vx, tk, tv, mask, S)).max() < 0.1
