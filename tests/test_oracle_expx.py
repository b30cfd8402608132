"""Pins of the oracle's BF16-exponent codec (rANS tiles, top-t table, escape records,
pair symbols): MINE section 4 (BF16 handling: exponent coded, sign and mantissa a
plain byte; "Escapes"; "Pair" with t^2 <= M) and section 4.2 ("Tuning t").

Each pin checks the oracle against something other than its own arithmetic:
round trips (every one of the 65536 BF16 patterns), the escape set as the
definition gives it, the k = 1 stream against the separately pinned FP8 top-t
codec run on the exponent bytes, the coded size against the cross-entropy bound,
a closed-form choice of t, and a brute-force pair histogram."""
import math

import numpy as np
import pytest

import oracle as O
import synth


def exps(w):
    return ((np.asarray(w, dtype=np.uint16) >> 7) & 0xFF).astype(np.int64)


def llama_padded(seed, n, k):
    return O.pad_rows(synth.llama_bf16(seed, n, k)).ravel()


@pytest.mark.parametrize("k,t,b,tile", [(1, 256, 12, 4096), (1, 8, 12, 4096), (1, 1, 12, 128), (2, 16, 12, 4096),
                                        (2, 6, 9, 1024), (2, 1, 12, 64), (1, 24, 10, 4096)])
def test_round_trip_llama_weights(k, t, b, tile):
    w = llama_padded(900 + t, 37, 1000)  # ragged: 37 rows of 1024 padded columns, short last tile
    o = O.Expx(w, t=t, prob_bits=b, tile=tile, k=k)
    out, rc = o.decode()
    assert rc == 0
    assert np.array_equal(out, w)
    assert int(o.freqs.sum()) == 1 << b


@pytest.mark.parametrize("k,t", [(1, 256), (2, 16), (1, 1), (2, 4)])
def test_round_trip_all_patterns(k, t):
    w = np.arange(65536, dtype=np.uint16)
    rng = np.random.default_rng(5)
    w = w[rng.permutation(65536)]
    o = O.Expx(w, t=t, prob_bits=12, tile=4096, k=k)
    out, rc = o.decode()
    assert rc == 0 and np.array_equal(out, w)


def test_escape_set_is_the_exponents_outside_the_table():
    """Records are exactly the positions whose exponent is not among exponent 0 and
    the t - 1 most frequent others (ties to the lower exponent), ascending within a
    tile, with the true exponent."""
    w = llama_padded(901, 64, 2048)
    t, tile = 7, 2048
    o = O.Expx(w, t=t, prob_bits=12, tile=tile, k=1)
    e = exps(w)
    cnt = np.bincount(e, minlength=256)
    others = sorted([v for v in range(1, 256) if cnt[v]], key=lambda v: (-cnt[v], v))[: t - 1]
    kept = sorted({0, *others})
    assert list(o.table) == kept
    want = []
    for base in range(0, w.size, tile):
        for p in range(min(tile, w.size - base)):
            if e[base + p] not in kept:
                want.append(p | (int(e[base + p]) << 16))
    assert list(o.records) == want
    assert o.n_records == int(np.isin(e, kept, invert=True).sum()) > 0


@pytest.mark.parametrize("t", [256, 12, 3])
def test_single_symbols_equal_the_fp8_codec_on_exponent_bytes(t):
    """With k = 1 the exponent stream is the FP8 top-t codec applied to the exponent
    bytes (same table rule, same tiles): identical table, frequencies, states, words
    and records."""
    w = llama_padded(902, 48, 1536)
    # (the FP8 codec refuses bytes x1111111, its NaN: move exponent 127 to 126)
    w = np.where(exps(w) == 127, (w & 0x807F) | (126 << 7), w).astype(np.uint16)
    o = O.Expx(w, t=t, prob_bits=11, tile=4096, k=1)
    f = O.Fp8(exps(w).astype(np.uint8), t=t, prob_bits=11, tile=4096)
    assert list(o.table) == list(f.table)
    assert np.array_equal(o.freqs, f.freqs)
    assert np.array_equal(o.states, f.states) and np.array_equal(o.offsets, f.offsets)
    assert np.array_equal(o.payload(), f.payload())
    assert np.array_equal(o.records, f.records)


@pytest.mark.parametrize("k,t", [(1, 256), (2, 16), (2, 8)])
def test_coded_size_meets_the_cross_entropy_bound(k, t):
    """16 bits per payload word plus the 32 initial states per tile against the
    cross-entropy of the symbol stream under the stored table, sum c_s log2(M / f_s):
    within 0.5% above it, and no lower than it minus the states' share."""
    w = llama_padded(903, 256, 4096)
    o = O.Expx(w, t=t, prob_bits=12, tile=4096, k=k)
    M = 1 << o.prob_bits
    c, f = o.counts.astype(np.float64), o.freqs.astype(np.float64)
    bound = float(np.sum(c[c > 0] * (np.log2(M) - np.log2(f[c > 0]))))
    coded = 16.0 * o.payload_words
    states = 32 * 32 * o.n_tiles
    assert bound - states <= coded <= 1.005 * bound
    # and the bound itself is at least the stream's Shannon entropy (Gibbs)
    p = c[c > 0] / c.sum()
    assert bound >= c.sum() * float(-(p * np.log2(p)).sum()) - 1e-6


def test_pair_histogram_brute_force():
    """k = 2 on one short tile: symbol = rank(e at step 2m) * tsize + rank(e at step
    2m + 1) of lane l (position 32 j + l is lane l's step j), counted by hand."""
    w = llama_padded(904, 1, 256)[:256].copy()
    w[5] = 0x7F80  # exponent 255: certainly outside a small table
    t = 4
    o = O.Expx(w, t=t, prob_bits=10, tile=256, k=2)
    table = list(o.table)
    rank = {v: i for i, v in enumerate(table)}
    e = exps(w)
    ts = o.tsize
    want = np.zeros(ts * ts, dtype=np.uint64)
    for l in range(32):
        for m in range(256 // 64):
            r0 = rank.get(int(e[32 * (2 * m) + l]), 0)
            r1 = rank.get(int(e[32 * (2 * m + 1) + l]), 0)
            want[r0 * ts + r1] += 1
    assert np.array_equal(o.counts, want)
    assert 5 in [int(r) & 0xFFFF for r in o.records]


def test_choose_t_closed_form():
    """Weights whose exponents are 0 or one other value: t = 1 leaves a stream of one
    symbol (0 bits) and escapes every nonzero weight at 32 bits; t = 2 codes the two
    exponents at the binary entropy of their shares, with no escapes."""
    w = np.zeros(8192, dtype=np.uint16)
    w[::3] = 0x3F80  # 1.0: exponent 127
    w[1::3] = 0xBF81
    nz = np.count_nonzero(exps(w))
    assert O.expx_bound(w, 1, 1) == pytest.approx(32.0 * nz)
    p = nz / w.size
    h2 = -(p * math.log2(p) + (1 - p) * math.log2(1 - p))
    assert O.expx_bound(w, 1, 2) == pytest.approx(w.size * h2, rel=2e-3)
    assert O.expx_choose_t(w, 1, 256) == 2
    assert O.expx_choose_t(w, 2, 16) == 2


@pytest.mark.parametrize("k,t_max", [(1, 64), (2, 16)])
def test_chosen_t_is_near_the_smallest_actual_size(k, t_max):
    """The t chosen by the bound codes within 1% of the best actual size (payload
    words and records) over every t."""
    w = llama_padded(905, 64, 4096)
    tc = O.expx_choose_t(w, k, t_max)
    sizes = {}
    for t in range(1, t_max + 1):
        o = O.Expx(w, t=t, prob_bits=12, tile=4096, k=k)
        sizes[t] = 16 * o.payload_words + 32 * o.n_records
    assert sizes[tc] <= 1.01 * min(sizes.values())
    assert O.expx_bound(w, k, tc) <= min(O.expx_bound(w, k, t) for t in range(1, t_max + 1)) + 1e-6


def test_pair_mode_needs_t_squared_within_the_table():
    w = np.arange(65536, dtype=np.uint16)
    assert O.expx_bound(w, 2, 256, prob_bits=12) == -1.0
    with pytest.raises(ValueError):
        O.Expx(w, t=100, prob_bits=12, tile=4096, k=2)


def test_flipped_payload_bit_is_detected():
    w = llama_padded(906, 32, 4096)
    o = O.Expx(w, t=16, prob_bits=12, tile=4096, k=2)
    o.flip_payload_bit(o.payload_words // 2, 3)
    out, rc = o.decode()
    assert rc != 0 or not np.array_equal(out, w)
