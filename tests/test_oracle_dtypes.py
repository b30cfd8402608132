"""Pins of the oracle's FP32 -> FP8 E4M3 and FP32 -> INT8 conversions and of its
E8 reconstruction in those dtypes (EntroPack section 3.7 and appendix B.1), against
the OCP E4M3 format's own definition (values written out here from the bit
fields), its textbook landmarks, midpoints, and numpy's round-half-even."""
import numpy as np
import pytest

import oracle as O
import synth


def e4m3_value(code: int) -> float:
    """Magnitude of E4M3 code 0..126 from its fields: bias 7, subnormals at exponent 0."""
    e, m = code >> 3, code & 7
    return (m / 8) * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)


def test_e4m3_landmarks():
    # smallest subnormal, smallest normal, one, largest finite (S.1111.110)
    assert list(O.f32_to_e4m3([2.0 ** -9, 2.0 ** -6, 1.0, 448.0])) == [0x01, 0x08, 0x38, 0x7E]
    assert list(O.f32_to_e4m3([-2.0 ** -9, -1.0, -448.0])) == [0x81, 0xB8, 0xFE]
    assert list(O.f32_to_e4m3([0.0, -0.0])) == [0x00, 0x80]


def test_e4m3_every_code_round_trips():
    vals = np.array([e4m3_value(c) for c in range(127)], dtype=np.float64)
    assert (np.diff(vals) > 0).all()  # the codes are ordered by magnitude
    assert np.array_equal(O.f32_to_e4m3(vals.astype(np.float32)), np.arange(127, dtype=np.uint8))
    assert np.array_equal(O.f32_to_e4m3(-vals[1:].astype(np.float32)), np.arange(1, 127, dtype=np.uint8) | 0x80)


def test_e4m3_midpoints_round_to_even():
    for c in range(126):
        lo, hi = e4m3_value(c), e4m3_value(c + 1)
        mid = np.float32((lo + hi) / 2)
        assert float(mid) == (lo + hi) / 2  # exact: at most 5 significant bits
        even = c if c % 2 == 0 else c + 1
        got = O.f32_to_e4m3([mid, np.nextafter(mid, np.float32(np.inf)), np.nextafter(mid, np.float32(0))])
        assert list(got) == [even, c + 1, c], c


def test_e4m3_saturates():
    big = np.array([448.0, 449.0, 463.9, 464.0, 480.0, 1e30, np.inf], dtype=np.float32)
    assert (O.f32_to_e4m3(big) == 0x7E).all()
    assert (O.f32_to_e4m3(-big) == 0xFE).all()


def test_s8_matches_numpy_rint_and_clip():
    rng = np.random.default_rng(2)
    v = np.concatenate([rng.normal(0, 60, 4000), np.arange(-130, 130) + 0.5, [0.5, -0.5, 1e9, -1e9]])
    v = v.astype(np.float32)
    want = np.clip(np.rint(v.astype(np.float64)), -128, 127).astype(np.int8)
    assert np.array_equal(O.f32_to_s8(v), want)


@pytest.mark.parametrize("dtype", ["bf16", "e4m3", "int8"])
def test_reconstruct_dtypes_with_power_of_two_scales(dtype):
    """Power-of-two scales make v = q / 2 * s * r_i exact in FP32, so each dtype's
    output is its conversion of that exact value."""
    q2 = synth.e8_points(91, 16, 256)
    r = (2.0 ** (np.arange(16) % 7 - 2)).astype(np.float32)
    s = 2.0 ** -3 if dtype != "int8" else 2.0
    v = (q2.astype(np.float64) / 2 * s * r[:, None]).astype(np.float32)
    got = O.e8_reconstruct(q2, s, r, dtype)
    if dtype == "bf16":
        assert np.array_equal(got, O.e8_reconstruct_bf16(q2, s, r))
        assert np.array_equal((got.astype(np.uint32) << 16).view(np.float32), v)
    elif dtype == "e4m3":
        assert np.array_equal(got.ravel(), O.f32_to_e4m3(v))
    else:
        assert np.array_equal(got, np.clip(np.rint(v.astype(np.float64)), -128, 127).astype(np.int8))
