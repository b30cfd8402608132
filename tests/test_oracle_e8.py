"""Pins of the oracle's E8 lattice fields and 17-table rANS tile codec (EntroPack
sections 3.2, 3.3, 3.6, 3.7, appendix A.3) against closed forms, brute force and
invariants -- none of them the oracle's own formulas re-typed."""
import itertools

import numpy as np
import pytest

import oracle as O


def e8_roots_doubled():
    """The 240 minimal vectors of E8, doubled: 112 of shape (+-2, +-2, 0^6) and 128
    of shape (+-1)^8 with an even number of -1."""
    roots = []
    for i, j in itertools.combinations(range(8), 2):
        for si, sj in itertools.product((2, -2), repeat=2):
            v = [0] * 8
            v[i], v[j] = si, sj
            roots.append(v)
    for signs in itertools.product((1, -1), repeat=8):
        if signs.count(-1) % 2 == 0:
            roots.append(list(signs))
    return np.array(roots, dtype=np.int8)


def random_points(rng, n, spread=2.0):
    """n doubled E8 points: z in Z^8 with an even sum (D8), coset c, q = 2 z + c."""
    z = np.clip(np.round(rng.normal(0, spread, size=(n, 8))), -14, 13).astype(np.int64)
    odd = z.sum(axis=1) % 2 == 1
    z[odd, 7] += 1  # into D8
    c = rng.integers(0, 2, size=(n, 1))
    return (2 * z + c).astype(np.int8)


def test_roots_are_lattice_points_and_round_trip():
    roots = e8_roots_doubled()
    assert len(roots) == 240
    assert (np.sum(roots.astype(np.int64) ** 2, axis=1) == 8).all()  # norm^2 = 2, doubled
    for q in roots:
        f = O.e8_fields(q)
        assert f is not None
        assert np.array_equal(O.e8_point(f), q)
    # the other half of the (+-1)^8 vectors (odd number of -1) is not in E8
    for signs in itertools.product((1, -1), repeat=8):
        if signs.count(-1) % 2 == 1:
            assert O.e8_fields(np.array(signs, dtype=np.int8)) is None


def test_brute_force_box_membership_and_count():
    """All q in {-2..2}^8: a point is in 2 E8 iff its coordinates share one parity c
    and sum((q - c) / 2) is even.  There are (3^8 + 1) / 2 = 3281 such points with
    even q and 2^7 = 128 with odd q (q in {-1, 1}^8, an even number of -1)."""
    valid = 0
    for q in itertools.product(range(-2, 3), repeat=8):
        qa = np.array(q, dtype=np.int8)
        c = q[0] & 1
        member = all((x & 1) == c for x in q) and (sum((x - c) // 2 for x in q) % 2 == 0)
        f = O.e8_fields(qa)
        assert (f is not None) == member, q
        if member:
            valid += 1
            assert np.array_equal(O.e8_point(f), qa)
    assert valid == 3281 + 128


@pytest.mark.parametrize("n,tile", [(1, 32), (31, 32), (1000, 64), (5000, 512), (8192, 512)])
def test_codec_round_trip_and_invariants(n, tile):
    rng = np.random.default_rng(n + tile)
    q = random_points(rng, n)
    e = O.E8(q, prob_bits=11, tile=tile)
    out, fin, rc = e.decode()
    assert rc == 0 and np.array_equal(out, q)
    assert (fin == 1 << 16).all()
    assert e.n_tiles == (n + tile - 1) // tile


def test_coset_conditioned_counts():
    """Table 0 counts the cosets; table 1 + 8 c + f counts field f of the points of
    coset c: per coset, histograms of z_1..z_7 (+16) and of m (+16) computed here
    from q directly."""
    rng = np.random.default_rng(7)
    q = random_points(rng, 4000).astype(np.int64)
    e = O.E8(q.astype(np.int8))
    counts = e.counts.astype(np.int64)
    c = q[:, 0] & 1
    assert np.array_equal(counts[0, :2], np.bincount(c, minlength=2))
    assert not counts[0, 2:].any()
    z = (q - c[:, None]) // 2
    m = (z[:, 7] - (z[:, :7].sum(axis=1) % 2)) // 2
    for cc in (0, 1):
        sel = c == cc
        for f in range(7):
            assert np.array_equal(counts[1 + 8 * cc + f], np.bincount(z[sel, f] + 16, minlength=32)), (cc, f)
        assert np.array_equal(counts[1 + 8 * cc + 7], np.bincount(m[sel] + 16, minlength=32)), cc


def test_stored_size_bounds_the_cross_entropy():
    """The stored stream (16-bit words and 32-bit final states) is at least the sum
    over the 17 tables of n_t * H(P_t, Q_t)."""
    rng = np.random.default_rng(11)
    q = random_points(rng, 20000, spread=1.5)
    e = O.E8(q, prob_bits=11, tile=512)
    bound = 0.0
    for t in range(O.E8_TABLES):
        n_t = float(e.counts[t].sum())
        if n_t:
            bound += n_t * O.cross_entropy(e.counts[t], e.freqs[t], 11)
    assert 16 * e.payload_words + 32 * 32 * e.n_tiles >= bound
    # and coset conditioning never costs: the conditioned tables' ideal cost is at
    # most that of one table per field (the sum of mutual informations is >= 0)
    cond = sum(O.entropy(e.counts[t]) * float(e.counts[t].sum()) for t in range(1, 17) if e.counts[t].sum())
    uncond = sum(O.entropy(e.counts[1 + f] + e.counts[9 + f]) * float((e.counts[1 + f] + e.counts[9 + f]).sum())
                 for f in range(8))
    assert cond <= uncond + 1e-6


def test_corrupt_payload_is_detected():
    rng = np.random.default_rng(3)
    q = random_points(rng, 2048)
    e = O.E8(q, tile=512)
    e.flip_payload_bit(5, 3)
    try:
        out, fin, rc = e.decode(strict=False)
        assert rc != 0 or not np.array_equal(out, q)
    except ValueError:
        pass


def test_reconstruction_exact_with_power_of_two_scales():
    """With s and r_i powers of two every product is exact: w = q / 2 * s * r_i."""
    rng = np.random.default_rng(5)
    q = random_points(rng, 64 * 32).reshape(64, 256)
    r = (2.0 ** rng.integers(-6, 3, size=64)).astype(np.float32)
    s = 2.0 ** -5
    w = O.e8_reconstruct_bf16(q, s, r)
    expect = q.astype(np.float64) / 2 * s * r[:, None].astype(np.float64)
    got = (w.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(got, expect)
