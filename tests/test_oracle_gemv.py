"""Pins for the oracle's FP64 GEMV and its storage-type conversions: exact integer
cases, agreement with numpy's float64 matmul, row selection, and the IEEE
conversions against numpy / torch."""
import numpy as np
import pytest
import torch

import oracle as O
import synth


def f32_to_bf16_bits(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_exact_integer_case():
    rng = np.random.default_rng(0)
    wi = rng.integers(-8, 9, (13, 77))
    xi = rng.integers(-4, 5, (3, 77))
    w = f32_to_bf16_bits(wi.astype(np.float32))
    x = f32_to_bf16_bits(xi.astype(np.float32))
    y, a = O.gemv_bf16(w, x)
    assert np.array_equal(y, (xi @ wi.T).astype(np.float64))
    assert np.array_equal(a, (np.abs(xi) @ np.abs(wi).T).astype(np.float64))


def test_matches_numpy_float64():
    w = synth.llama_bf16(2000, 300, 1024)
    x = synth.make_x(2000, 4, 1024)
    y, a = O.gemv_bf16(w, x)
    wf = synth.bf16_to_f32(w).astype(np.float64)
    xf = synth.bf16_to_f32(x).astype(np.float64)
    ref = xf @ wf.T
    mag = np.abs(xf) @ np.abs(wf).T
    assert (np.abs(y - ref) <= 1e-12 * mag).all()
    assert np.allclose(a, mag, rtol=1e-12)


def test_row_selection():
    w = synth.llama_bf16(2005, 50, 64)
    x = synth.make_x(1, 2, 64)
    y, a = O.gemv_bf16(w, x)
    rows = np.array([49, 0, 7, 7])
    ys, as_ = O.gemv_bf16(w, x, rows=rows)
    assert np.array_equal(ys, y[:, rows]) and np.array_equal(as_, a[:, rows])


def test_rans_gemv_matches_numpy():
    codes, scales = synth.make_rans_case(1, 40, 300)
    x = synth.make_x(4001, 2, 300)
    y, a = O.gemv_rans(codes, scales, x)
    s = scales.view(np.float16).astype(np.float64)
    wv = codes.astype(np.float64) * np.repeat(s, 128, axis=1)[:, :300]
    xf = synth.bf16_to_f32(x).astype(np.float64)
    assert np.allclose(y, xf @ wv.T, rtol=1e-12, atol=1e-15)
    assert np.allclose(a, np.abs(xf) @ np.abs(wv).T, rtol=1e-12)


def test_f16_to_f32_all_patterns():
    h = np.arange(65536, dtype=np.uint16)
    want = h.view(np.float16).astype(np.float32)
    got = np.array([O.f16_to_f32(int(v)) for v in h[::7]], np.float32)
    ref = want[::7]
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_bf16_rne_against_torch():
    rng = np.random.default_rng(3)
    vals = np.concatenate([rng.standard_normal(2000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 2000),
                           np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 3.0e38, -1e-40, np.inf], np.float32)])
    # values exactly halfway between two BF16 numbers
    halfway = ((rng.integers(0, 1 << 15, 200).astype(np.uint32) << 16) | 0x8000).view(np.float32)
    vals = np.concatenate([vals, halfway[np.isfinite(halfway)]])
    got = np.array([O.f32_to_bf16_rne(float(v)) for v in vals], np.uint16)
    assert np.array_equal(got, f32_to_bf16_bits(vals))
