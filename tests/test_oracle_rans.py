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
