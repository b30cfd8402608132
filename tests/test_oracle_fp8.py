"""Pins of the oracle's FP8 path (MINE section 4, "Escapes": a top-t decoding table
that always holds 0, escaped values coded as 0 and restored from a sparse
correction stream): the E4M3 decode against the format's bit fields, the table
selection against brute force, round trips, escape counts, record placement, the
tile codec's invariants and the dequantisation / GEMV against exact arithmetic."""

import numpy as np
import pytest

import oracle as O
import synth


def e4m3_field_value(code: int) -> float:
    s, e, m = code >> 7, (code >> 3) & 15, code & 7
    v = (m / 8) * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
    return -v if s else v


def test_e4m3_decode_all_codes():
    vals = O.e4m3_to_f32(np.arange(256))
    for c in range(256):
        if c & 0x7F == 0x7F:
            assert np.isnan(vals[c])
        else:
            assert vals[c] == e4m3_field_value(c), c
    assert vals[0x00] == 0 and not np.signbit(vals[0x00]) and np.signbit(vals[0x80])
    assert vals[0x7E] == 448 and vals[0x01] == 2.0 ** -9 and vals[0x38] == 1.0
    finite = [c for c in range(256) if c & 0x7F != 0x7F]
    assert np.array_equal(O.f32_to_e4m3(vals[finite]), np.array(finite, dtype=np.uint8))


@pytest.mark.parametrize("seed", range(6))
def test_table_is_the_top_t_with_zero(seed):
    rng = np.random.default_rng(seed)
    counts = np.zeros(256, np.uint64)
    present = rng.choice(256, size=int(rng.integers(1, 120)), replace=False)
    counts[present] = rng.integers(1, 50, size=present.size)  # many ties
    for t in (1, 2, 5, 17, 64, 256):
        tab = O.fp8_table(counts, t)
        assert tab[0] == 0 and (np.diff(tab.astype(int)) > 0).all()
        others = [c for c in range(1, 256) if counts[c]]
        assert len(tab) == min(t, 1 + len(others))
        chosen = set(int(c) for c in tab[1:])
        # brute force: the chosen set is the first t - 1 of the others sorted by (-count, code)
        want = sorted(others, key=lambda c: (-int(counts[c]), c))[: len(tab) - 1]
        assert chosen == set(want), (t, chosen ^ set(want))


@pytest.mark.parametrize("t", [1, 2, 16, 64, 256])
@pytest.mark.parametrize("n,tile", [(4096, 4096), (3 * 4096 + 640, 1024), (128, 128)])
def test_round_trip_and_escapes(t, n, tile):
    codes = synth.fp8_codes(900 + t, 1, n).ravel()
    f = O.Fp8(codes, t=t, prob_bits=12, tile=tile)
    out, rc = f.decode()
    assert rc == 0 and np.array_equal(out, codes)
    table = set(int(c) for c in f.table)
    outside = np.array([c not in table for c in codes])
    assert f.n_records == int(outside.sum())
    # records: ascending positions per tile, each at an escaped position with its true code
    recs, off = f.records, f.rec_off
    for tt in range(f.n_tiles):
        r = recs[off[tt]:off[tt + 1]]
        pos = (r & 0xFFFF).astype(np.int64)
        assert (np.diff(pos) > 0).all()
        gpos = tt * tile + pos
        assert outside[gpos].all() and np.array_equal((r >> 16).astype(np.uint8), codes[gpos])
        assert outside[tt * tile:(tt + 1) * tile].sum() == len(r)
    # the symbol histogram: escapes count as symbol 0 (code 0x00)
    assert int(f.counts[0]) == int((codes == 0).sum() + outside.sum())


def test_stored_size_bounds_the_cross_entropy():
    codes = synth.fp8_codes(77, 1, 16 * 4096).ravel()
    for t in (16, 256):
        f = O.Fp8(codes, t=t, prob_bits=12, tile=4096)
        bound = float(f.counts.sum()) * O.cross_entropy(f.counts, f.freqs, 12)
        assert 16 * f.payload_words + 32 * 32 * f.n_tiles >= bound


def test_corrupt_payload_is_detected():
    codes = synth.fp8_codes(78, 1, 8192).ravel()
    f = O.Fp8(codes, t=32)
    f.flip_payload_bit(7, 5)
    out, rc = f.decode()
    assert rc != 0 or not np.array_equal(out, codes)


def test_dequant_and_gemv_exact_cases():
    """Power-of-two row scales make value * r exact in FP32 (BF16 then rounds the
    4-bit mantissa exactly); the GEMV against an exact float64 product."""
    codes = synth.fp8_codes(79, 16, 384)
    r = (2.0 ** (np.arange(16) % 5 - 9)).astype(np.float32)
    w = O.fp8_dequant_bf16(codes, r)
    vals = O.e4m3_to_f32(codes.ravel()).reshape(codes.shape).astype(np.float64)
    assert np.array_equal(synth.bf16_to_f32(w).astype(np.float64), vals * r[:, None])
    x = synth.make_x(80, 3, 384)
    xf = synth.bf16_to_f32(x).astype(np.float64)
    y, a = O.gemv_fp8(codes, r, x)
    assert np.allclose(y, xf @ (vals * r[:, None]).T, rtol=1e-13, atol=1e-13)
    assert np.allclose(a, np.abs(xf) @ np.abs(vals * r[:, None]).T, rtol=1e-13, atol=1e-13)
