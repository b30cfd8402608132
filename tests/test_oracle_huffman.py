"""Pins for the oracle's Huffman pieces: the pages' worked examples (DFloat11
Fig. 13 and Fig. 14), Kraft equality, prefix-freeness, optimality by brute force,
the Shannon bounds, and the special cases."""
import itertools
import math

import numpy as np
import pytest

import oracle as O
from conftest import read_golden


def kraft(lengths):
    return sum(2.0 ** -int(l) for l in lengths if l)


def cost(counts, lengths):
    return sum(int(c) * int(l) for c, l in zip(counts, lengths))


def brute_force_optimal(counts, max_len):
    """Minimum sum(c*l) over all length vectors in [1, max_len] with Kraft sum <= 1."""
    best = None
    n = len(counts)
    for ls in itertools.product(range(1, max_len + 1), repeat=n):
        if sum(2.0 ** -l for l in ls) <= 1.0 + 1e-12:
            c = sum(a * b for a, b in zip(counts, ls))
            best = c if best is None else min(best, c)
    return best


def test_fig13_canonical_code_and_flat_lut():
    g = read_golden("dfloat11_fig13_flat_lut.txt")
    lengths = [int(v) for v in g["lengths"]]
    codes = O.canonical_codes(lengths)[:6]
    assert codes.tolist() == [int(v) for v in g["codes"]]
    lut = O.flat_lut(lengths, codes, 4)
    assert lut.tolist() == [int(v) for v in g["lut"]]


def test_fig13_lengths_from_frequencies():
    # Frequencies for which Huffman's merge rule yields exactly A:1 B:3 C:3 D:3 E:4 F:4.
    assert O.huffman_textbook([8, 2, 2, 2, 1, 1])[:6].tolist() == [1, 3, 3, 3, 4, 4]


def test_fig14_hierarchical_luts():
    g = read_golden("dfloat11_fig14_hier_lut.txt")
    lengths = [1, 3, 3, 3, 4, 4]
    codes = O.canonical_codes(lengths)[:6]
    t = O.hier_luts(lengths, codes, 2)
    assert t.shape == (3, 4)
    for k in range(3):
        want = [256 + int(v[1:]) if v.startswith("T") else int(v) for v in g[f"table{k}"]]
        assert t[k].tolist() == want


def test_hier_lut_walk_matches_flat_lut():
    """Every 12-bit string decodes to the same first symbol through the b=4
    hierarchy as through the flat table."""
    rng = np.random.default_rng(5)
    counts = rng.integers(1, 1000, 40) ** 2
    lengths = O.code_lengths(counts, 12)
    codes = O.canonical_codes(lengths)
    flat = O.flat_lut(lengths, codes, 12)
    t = O.hier_luts(lengths, codes, 4)
    for s in range(1 << 12):
        v = t[0][s >> 8]
        i = 1
        while v >= 256:
            v = t[v - 256][(s >> (8 - 4 * i)) & 0xF]
            i += 1
        assert v == flat[s]


@pytest.mark.parametrize("seed", range(20))
def test_kraft_equality_and_prefix_free(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(2, 257))
    counts = np.zeros(256, np.uint64)
    idx = rng.choice(256, n, replace=False)
    counts[idx] = rng.geometric(0.05, n) ** rng.integers(1, 4)
    for lengths in (O.huffman_textbook(counts), O.package_merge(counts, max(8, int(math.ceil(math.log2(n)))) + 1)):
        assert kraft(lengths) == 1.0
        assert (lengths[counts == 0] == 0).all() and (lengths[counts > 0] > 0).all()
        codes = O.canonical_codes(lengths)
        words = [format(int(codes[s]), f"0{int(lengths[s])}b") for s in range(256) if lengths[s]]
        words.sort()
        # sorted lexicographically, a prefix can only be a prefix of its successor
        for a, b in zip(words, words[1:]):
            assert not b.startswith(a)


@pytest.mark.parametrize("seed", range(30))
def test_optimal_against_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(2, 7))
    counts = [int(v) for v in rng.integers(1, 60, n) ** int(rng.integers(1, 3))]
    tb = O.huffman_textbook(counts)[:n]
    assert cost(counts, tb) == brute_force_optimal(counts, n - 1)
    for L in range(max(1, math.ceil(math.log2(n))), n):
        pm = O.package_merge(counts, L)[:n]
        assert max(pm) <= L and kraft(pm) == 1.0
        assert cost(counts, pm) == brute_force_optimal(counts, L)


def test_package_merge_agrees_with_textbook_when_unconstrained():
    rng = np.random.default_rng(7)
    for _ in range(10):
        counts = (rng.pareto(1.2, 200) * 100).astype(np.uint64) + 1
        tb = O.huffman_textbook(counts)
        pm = O.package_merge(counts, 30)
        assert cost(counts, tb) == cost(counts, pm)


def test_length_limit_binds_on_geometric_histogram():
    counts = [2 ** (40 - i) for i in range(30)]  # textbook lengths 1..29
    tb = O.huffman_textbook(counts)
    assert tb.max() == 29
    lim = O.code_lengths(counts, 24)
    assert lim.max() == 24 and kraft(lim) == 1.0
    assert cost(counts, lim) >= cost(counts, tb)
    # with the limit the result is still the package-merge optimum
    assert cost(counts, lim) == cost(counts, O.package_merge(counts, 24))


def test_shannon_bounds_on_exponent_histogram():
    import synth
    w = synth.gauss_bf16(1001, (256, 1024), 0.02)
    counts = np.bincount(((w >> 7) & 0xFF).ravel(), minlength=256)
    lengths = O.code_lengths(counts, 24)
    h = O.entropy(counts)
    avg = cost(counts, lengths) / counts.sum()
    assert h <= avg < h + 1.0


def test_special_cases():
    one = np.zeros(256, np.uint64)
    one[77] = 5
    assert O.huffman_textbook(one)[77] == 1 and O.huffman_textbook(one).sum() == 1
    assert O.huffman_textbook(np.zeros(256, np.uint64)).sum() == 0
    two = np.zeros(256, np.uint64)
    two[[3, 200]] = [1, 1000]
    assert sorted(O.huffman_textbook(two)[[3, 200]].tolist()) == [1, 1]
    flat = np.ones(256, np.uint64)
    assert (O.huffman_textbook(flat) == 8).all()
    with pytest.raises(ValueError):
        O.package_merge(flat, 7)  # 2^7 < 256 symbols


def test_entropy_closed_forms():
    assert O.entropy([1] * 8) == pytest.approx(3.0, abs=1e-15)
    assert O.entropy([1, 3]) == pytest.approx(2 - 0.75 * math.log2(3), abs=1e-15)
    assert O.entropy([5]) == 0.0
    # discretised N(0, 1.1^2) clipped to [-8, 7]: p_k from the normal CDF
    sd = 1.1
    cdf = lambda t: 0.5 * (1 + math.erf(t / (sd * math.sqrt(2))))
    p = []
    for k in range(-8, 8):
        lo = -math.inf if k == -8 else k - 0.5
        hi = math.inf if k == 7 else k + 0.5
        p.append((1.0 if hi == math.inf else cdf(hi)) - (0.0 if lo == -math.inf else cdf(lo)))
    h_closed = -sum(q * math.log2(q) for q in p if q > 0)
    import synth
    c = synth.codes_i8(4000, (2048, 2048)).ravel().astype(np.int64) + 8
    h_emp = O.entropy(np.bincount(c, minlength=16))
    assert abs(h_emp - h_closed) < 2e-3
    assert h_closed == pytest.approx(2.2328, abs=1e-3)
