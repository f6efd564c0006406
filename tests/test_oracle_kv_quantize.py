"""Pins of the oracle's FP8 cache-write quantiser (oracle_f32_to_e4m3,
oracle_kv_quantize), on the CPU.

The E4M3 rounding is pinned to the OCP E4M3 value set and a library routine
(torch's float8_e4m3fn conversion, round to nearest even): every finite code
round-trips, every midpoint between neighbouring codes goes to the even
code, and random values agree with torch.  The row quantiser is pinned to its
error bound and special cases (the largest element maps to +-448, a zero row
has scale 0).
"""
import numpy as np
import pytest
import torch

import oracle


def _value(code):
    return oracle.e4m3_to_f64(code)


def test_every_finite_code_round_trips():
    for c in range(256):
        if (c & 0x7F) == 0x7F:  # NaN
            continue
        assert oracle.f32_to_e4m3(np.float32(_value(c))) == c, hex(c)


def test_midpoints_round_to_even_code():
    for c in range(0, 0x7E):  # neighbours c, c + 1 on the positive side
        lo, hi = _value(c), _value(c + 1)
        mid = (lo + hi) / 2
        assert np.float32(mid) == mid  # exact in binary32
        even = c if c % 2 == 0 else c + 1
        assert oracle.f32_to_e4m3(np.float32(mid)) == even, hex(c)
        assert oracle.f32_to_e4m3(np.float32(-mid)) == even | 0x80
        # just off the midpoint goes to the nearer one
        assert oracle.f32_to_e4m3(np.nextafter(np.float32(mid), np.float32(0))) == c
        assert oracle.f32_to_e4m3(np.nextafter(np.float32(mid), np.float32(1e9))) == c + 1


def test_saturation_and_signed_zero():
    assert oracle.f32_to_e4m3(np.float32(448.0)) == 0x7E
    assert oracle.f32_to_e4m3(np.float32(1e30)) == 0x7E
    assert oracle.f32_to_e4m3(np.float32(-1e30)) == 0xFE
    assert oracle.f32_to_e4m3(np.float32(0.0)) == 0x00
    assert oracle.f32_to_e4m3(np.float32(-0.0)) == 0x80
    assert oracle.f32_to_e4m3(np.float32(2.0 ** -11)) == 0x00  # below half the
    assert oracle.f32_to_e4m3(np.float32(-(2.0 ** -11))) == 0x80  # smallest step


def test_random_values_agree_with_torch():
    rng = np.random.default_rng(3)
    v = np.concatenate([
        rng.uniform(-448, 448, 4000),
        rng.standard_normal(2000) * rng.choice([1e-3, 1e-2, 1, 10, 100], 2000),
        np.ldexp(rng.uniform(1, 2, 1000), rng.integers(-12, 9, 1000)),
    ]).astype(np.float32)
    v = v[np.abs(v) <= 448]  # torch does not saturate (overflow gives NaN)
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.f32_to_e4m3(x) for x in v], np.uint8)
    # torch keeps the sign of a value that rounds to zero as well
    np.testing.assert_array_equal(got, want)


def test_row_quantiser_bounds_and_special_cases():
    rng = np.random.default_rng(4)
    rows = rng.standard_normal((6, 576)).astype(np.float32)
    rows[1] *= 1e-20
    rows[2] *= 3e4
    rows[3] = 0.0
    rows[4, 17] = 40.0  # one large element
    codes, scales = oracle.kv_quantize(rows)
    assert scales[3] == 0.0 and not codes[3].any()
    for r in (0, 1, 2, 4, 5):
        amax = np.abs(rows[r]).max()
        assert scales[r] == np.float32(amax) / np.float32(448.0)
        k = int(np.abs(rows[r]).argmax())
        assert codes[r, k] & 0x7F == 0x7E  # the largest element is +-448
        deq = np.array([_value(c) for c in codes[r]]) * float(scales[r])
        err = np.abs(deq - rows[r].astype(np.float64))
        # E4M3: half a step of 3 mantissa bits (2^-4 relative) for normals,
        # half the subnormal step 2^-9 (in units of the scale) below 2^-6
        bound = np.maximum(np.abs(rows[r]) * 2.0 ** -4, float(scales[r]) * 2.0 ** -10)
        assert (err <= bound * (1 + 1e-6)).all(), r
