"""Pins for the oracle's rANS tile codec: round trips (including ragged and
degenerate tiles), the stored-state invariant (every lane returns to 2^16 and
consumes exactly its tile's words), frequency normalisation, brute force over
tiny alphabets, and the cross-entropy size bound."""
import itertools

import numpy as np
import pytest

import oracle as O
import synth

M = 4096


@pytest.mark.parametrize("n", [0, 1, 5, 31, 32, 33, 4095, 4096, 4097, 3 * 4096 + 1000])
def test_round_trip_and_final_states(n):
    c = synth.codes_i8(4000 + n, (n,))
    r = O.Rans(c)
    out, fin, rc = r.decode()
    assert rc == 0
    assert np.array_equal(out, c)
    assert (fin == 1 << 16).all()
    assert r.n_tiles == (n + 4095) // 4096


def test_frequencies_normalised():
    for seed in range(20):
        rng = np.random.default_rng(seed)
        counts = np.zeros(16, np.uint64)
        k = int(rng.integers(1, 17))
        counts[rng.choice(16, k, replace=False)] = rng.integers(1, 10 ** rng.integers(1, 8), k)
        f = O.rans_freqs(counts)
        assert int(f.sum()) == M
        assert ((f > 0) == (counts > 0)).all()
        share = M * counts.astype(np.float64) / float(counts.sum())
        present = counts > 0
        # every present symbol within a few units of its exact share M * p
        # (the floor of 1 for rare symbols is paid for by the largest ones)
        lifted = int((present & (share < 1)).sum())
        assert (np.abs(f[present] - share[present]) <= 1 + lifted).all()


def test_single_symbol_alphabet_is_free():
    c = np.full(10000, 3, np.int8)
    r = O.Rans(c)
    assert r.freqs[3 + 8] == M and r.payload_words == 0
    out, fin, rc = r.decode()
    assert rc == 0 and np.array_equal(out, c)


def test_brute_force_tiny_alphabets():
    for alphabet in ([0, 1], [-8, 7], [-1, 0, 2]):
        for L in range(1, 9):
            for seq in itertools.product(alphabet, repeat=L):
                c = np.array(seq, np.int8)
                r = O.Rans(c, tile=32)
                out, fin, rc = r.decode()
                assert rc == 0 and np.array_equal(out, c)


def test_lane_interleave_within_tile():
    """Position q = 32 j + l belongs to lane l: encoding a tile whose lanes are
    constant must give every lane a state history independent of the others."""
    c = np.tile(np.arange(-8, 8, dtype=np.int8).repeat(2), 4096 // 32)  # lane l always holds code l//2 - 8
    r = O.Rans(c)
    out, fin, rc = r.decode()
    assert rc == 0 and np.array_equal(out, c)


def test_size_against_cross_entropy():
    c = synth.codes_i8(4000, (2048, 2048)).ravel()
    r = O.Rans(c)
    ce = O.cross_entropy(r.counts, r.freqs, 12)
    h = O.entropy(r.counts)
    assert ce >= h
    stored_bits = 16 * r.payload_words + 32 * 32 * r.n_tiles
    assert stored_bits >= c.size * ce
    # the coder adds little beyond the per-lane state: within 0.5% + the state words
    assert 16 * r.payload_words <= c.size * ce * 1.005 + 32 * 16 * r.n_tiles


def test_corrupted_payload_detected_or_differs():
    c = synth.codes_i8(4001, (3 * 4096,))
    for frac in (0.0, 0.1, 0.5, 0.99):
        r = O.Rans(c)
        word = int(frac * (r.payload_words - 1))
        r.flip_payload_bit(word, 7)
        try:
            out, fin, rc = r.decode(strict=False)
        except ValueError:
            continue  # an impossible state was detected
        assert rc != 0 or not np.array_equal(out, c)


def test_dequant_bf16_matches_numpy_conversions():
    codes, scales = synth.make_rans_case(0, 8, 384)
    got = O.rans_dequant_bf16(codes, scales)
    s32 = scales.view(np.float16).astype(np.float32)
    w = codes.astype(np.float32) * np.repeat(s32, 128, axis=1)[:, :384]
    import torch
    want = torch.from_numpy(w).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


# ------------------------------------------------------------------ FP4 values
# The FP4 E2M1 value set as the OCP Microscaling specification tabulates it (the
# magnitudes of exponent fields 0..3 with mantissa bit 0, 1), written out here, not
# derived from the oracle's formula.
E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_values_match_the_format_table():
    vals = [O.e2m1_value(c) for c in range(16)]
    assert vals[:8] == E2M1_MAGNITUDES
    assert vals[8:] == [-m for m in E2M1_MAGNITUDES]
    assert np.signbit(vals[8])  # pattern 8 is -0


def test_fp4_dequant_and_gemv_match_numpy():
    codes, scales = synth.make_fp4_case(4300, 8, 384)
    table = np.array(E2M1_MAGNITUDES + [-m for m in E2M1_MAGNITUDES], dtype=np.float32)
    s32 = np.repeat(scales.view(np.float16).astype(np.float32), 128, axis=1)[:, :384]
    w = table[codes.astype(np.int64)] * s32  # exact in FP32
    import torch
    want = torch.from_numpy(w).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.rans_dequant_bf16(codes, scales, values="fp4"), want)
    x = synth.make_x(4301, 3, 384)
    xf = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    y, a = O.gemv_rans(codes, scales, x, values="fp4")
    assert np.allclose(y, xf @ w.astype(np.float64).T, rtol=1e-12, atol=1e-12)
    assert np.allclose(a, np.abs(xf[:, None, :] * w.astype(np.float64)[None]).sum(-1), rtol=1e-12, atol=1e-12)
    # the integer reading of the same patterns differs (a dropped mode would not)
    assert not np.array_equal(O.rans_dequant_bf16(codes - 8, scales), want)


# ---------------------------------------------------------------- pair symbols
@pytest.mark.parametrize("n", [0, 64, 4096, 4160, 3 * 4096 + 1024])
def test_pair_round_trip_and_final_states(n):
    c = synth.codes_i8(4100 + n, (n,))
    r = O.Rans(c, k=2)
    out, fin, rc = r.decode()
    assert rc == 0
    assert np.array_equal(out, c)
    assert (fin == 1 << 16).all()


def test_pair_symbols_are_a_lanes_consecutive_steps():
    """Symbol = 16 (c[32 (2m) + l] + 8) + (c[32 (2m + 1) + l] + 8) inside a tile:
    the oracle's pair histogram equals the one counted here from the layout."""
    n, tile = 3 * 4096 + 1024, 4096
    c = synth.codes_i8(4200, (n,)).astype(np.int64) + 8
    want = np.zeros(256, np.int64)
    for base in range(0, n, tile):
        t = c[base:base + tile].reshape(-1, 32)  # step, lane
        want += np.bincount((16 * t[0::2] + t[1::2]).ravel(), minlength=256)
    r = O.Rans((c - 8).astype(np.int8), k=2, tile=tile)
    assert np.array_equal(r.counts.astype(np.int64), want)


def test_pair_mode_needs_whole_pairs():
    with pytest.raises(ValueError):
        O.Rans(np.zeros(96, np.int8), k=2)  # 96 codes: lanes would hold 3 steps
    with pytest.raises(ValueError):
        O.Rans(np.zeros(128, np.int8), k=2, tile=96)


def test_pair_random_tiny_alphabets():
    rng = np.random.default_rng(3)
    for alphabet in ([0, 1], [-8, 7], [-1, 0, 2]):
        for _ in range(50):
            c = rng.choice(np.array(alphabet, np.int8), 64 * int(rng.integers(1, 4)))
            r = O.Rans(c, k=2, tile=64)
            out, fin, rc = r.decode()
            assert rc == 0 and np.array_equal(out, c)


def test_pair_frequencies_normalised():
    rng = np.random.default_rng(5)
    for _ in range(10):
        counts = np.zeros(256, np.uint64)
        k = int(rng.integers(2, 200))
        counts[rng.choice(256, k, replace=False)] = rng.integers(1, 10 ** rng.integers(1, 7), k)
        f = O.rans_freqs(counts)
        assert f.size == 256 and int(f.sum()) == M
        assert ((f > 0) == (counts > 0)).all()


def test_pair_size_against_cross_entropy():
    """Pairs of i.i.d. codes: the pair histogram's entropy per code equals the
    single-code entropy, and 12-bit pair frequencies cost at most 0.02 bit per
    code over single-code ones on the discretised N(0, 1.1) codes."""
    c = synth.codes_i8(4000, (2048, 2048)).ravel()
    r1, r2 = O.Rans(c), O.Rans(c, k=2)
    ce1 = O.cross_entropy(r1.counts, r1.freqs, 12)
    ce2 = O.cross_entropy(r2.counts, r2.freqs, 12) / 2
    h1, h2 = O.entropy(r1.counts), O.entropy(r2.counts) / 2
    assert abs(h2 - h1) < 2e-3
    assert ce2 >= h2 and ce2 <= ce1 + 0.02
    assert 16 * r2.payload_words <= c.size * ce2 * 1.005 + 32 * 16 * r2.n_tiles


def test_table_bits_uniform_alphabet_takes_the_smallest_table():
    """Every table size represents a uniform 16-symbol distribution exactly (cross
    entropy 4 bits at any b >= 4), so the table's own size decides: b = 9."""
    counts = np.full(16, 1000, dtype=np.uint64)
    assert O.rans_table_bits(counts) == 9
    for b in (9, 10, 11, 12):
        assert abs(O.cross_entropy(counts, O.rans_freqs(counts, b), b) - 4.0) < 1e-12


def test_table_bits_rare_symbols_need_the_largest_table():
    """One dominant symbol and 15 singletons: at 2^b slots the singletons take at
    least 15 slots, so the dominant symbol costs about -log2(1 - 15/2^b) bits; over
    10^8 symbols that gap dwarfs the table sizes and the largest table wins."""
    counts = np.ones(16, dtype=np.uint64)
    counts[8] = 10 ** 8
    assert O.rans_table_bits(counts) == 12
    # the scores follow the closed form closely enough to order the candidates
    n = float(counts.sum())
    for b in (9, 12):
        ce = O.cross_entropy(counts, O.rans_freqs(counts, b), b)
        f = O.rans_freqs(counts, b)
        assert f[8] == (1 << b) - 15
        assert abs(ce - (-(1e8 / n) * np.log2(f[8] / 2 ** b) + 15 / n * b)) < 1e-9


def test_table_bits_stops_after_a_one_percent_rise():
    """The scan stops at the first candidate scoring more than 1% above the best so
    far.  One symbol of 10^6 and 15 singletons: 2^10 slots beat 2^9 (the singletons'
    15 slots cost the big symbol half as much), 2^11 costs more than 1% over 2^10 in
    table entries, so the scan stops there and never scores 2^12; put 2^12 right
    after 2^9 and the scan stops before reaching 2^10."""
    counts = np.ones(16, dtype=np.uint64)
    counts[8] = 10 ** 6
    n = float(counts.sum())
    score = {b: n * O.cross_entropy(counts, O.rans_freqs(counts, b), b) + 32 * (1 << b) for b in (9, 10, 11, 12)}
    assert score[10] < score[9] and score[11] > 1.01 * score[10] and score[12] > 1.01 * score[9]
    assert O.rans_table_bits(counts) == 10
    assert O.rans_table_bits(counts, candidates=(9, 12, 10)) == 9


@pytest.mark.parametrize("sigma", [0.4, 1.1, 3.0])
def test_table_bits_estimate_bounds_the_coded_size(sigma):
    """The chosen table's score is a lower bound: the oracle's stored stream (16-bit
    payload words and 32-bit final states) is at least n * H(P, Q_b) bits."""
    rng = np.random.default_rng(int(sigma * 10))
    c = np.clip(np.round(rng.normal(0, sigma, 64 * 4096)), -8, 7).astype(np.int8)
    counts = np.bincount(c.astype(np.int64) + 8, minlength=16).astype(np.uint64)
    b = O.rans_table_bits(counts)
    r = O.Rans(c, prob_bits=b)
    assert np.array_equal(r.freqs, O.rans_freqs(counts, b))
    stored = 16 * r.payload_words + 32 * 32 * r.n_tiles  # payload words and the 32 final states per tile
    assert stored >= c.size * O.cross_entropy(counts, r.freqs, b)
