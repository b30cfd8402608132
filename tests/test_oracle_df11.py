"""Pins for the oracle's DFloat11 codec: exact round trip of every BF16 pattern,
an independent bit-by-bit tree-walk decode of its stream, the Gaps /
BlockOutputPos definitions, the rate bounds, and corruption behaviour."""
import numpy as np
import pytest

import oracle as O
import synth


def exps(w):
    return ((w >> 7) & 0xFF).astype(np.int64)


def tree_walk_decode(stream_bits: str, lengths, codes, count):
    """Decode `count` symbols bit by bit with a dict of codewords (no LUTs)."""
    table = {format(int(codes[s]), f"0{int(lengths[s])}b"): s for s in range(256) if lengths[s]}
    out, cur = [], ""
    for bit in stream_bits:
        cur += bit
        if cur in table:
            out.append(table[cur])
            cur = ""
            if len(out) == count:
                break
    return out


def bits_of(stream: np.ndarray) -> str:
    return "".join(format(int(b), "08b") for b in stream)


def test_all_65536_bf16_patterns_round_trip():
    w = np.arange(65536, dtype=np.uint16)
    d = O.DF11(w)
    assert (d.lengths == 8).all()  # every exponent occurs 256 times
    assert np.array_equal(d.decode(), w)


@pytest.mark.parametrize("n_bytes,threads", [(8, 256), (8, 4), (2, 3), (1, 1), (16, 32)])
def test_round_trip_shapes_and_chunkings(n_bytes, threads):
    w = synth.llama_bf16(2003, 37, 129)
    d = O.DF11(w, n_bytes=n_bytes, threads=threads)
    assert np.array_equal(d.decode(), w.ravel())


@pytest.mark.parametrize("n", [0, 1, 2, 7, 31, 4097])
def test_round_trip_ragged_lengths(n):
    w = synth.gauss_bf16(11, (n,), 0.02)
    d = O.DF11(w)
    assert np.array_equal(d.decode(), w)


def test_stream_is_canonical_codewords_msb_first():
    w = synth.llama_bf16(2001, 16, 200)
    d = O.DF11(w)
    e = exps(w.ravel())
    want = "".join(format(int(d.codes[s]), f"0{int(d.lengths[s])}b") for s in e)
    got = bits_of(d.stream)
    assert got[: len(want)] == want
    assert set(got[len(want):]) <= {"0"}  # zero padding
    assert d.payload_bits == len(want)
    # independent decode of the exponents by walking codewords bit by bit
    assert tree_walk_decode(got, d.lengths, d.codes, e.size) == e.tolist()


def test_gaps_and_block_output_pos_definitions():
    w = synth.llama_bf16(2002, 64, 100)
    n_bytes, T = 4, 8
    d = O.DF11(w, n_bytes=n_bytes, threads=T)
    starts = np.concatenate([[0], np.cumsum(d.lengths[exps(w.ravel())])[:-1]])
    chunk_bits = 8 * n_bytes
    last_start = starts[-1]
    for c in range(d.n_chunks):
        c0 = c * chunk_bits
        if c0 > last_start:
            continue  # padding chunk
        first = starts[np.searchsorted(starts, c0)]
        assert d.gaps[c] == min(first - c0, chunk_bits)
    bp = d.block_pos
    for b in range(d.n_blocks):
        b0 = b * chunk_bits * T
        assert bp[b] == np.searchsorted(starts, b0)
    assert bp[-1] == w.size


def test_symbol_sequences_brute_force():
    """All exponent sequences of length <= 6 over a 3-value alphabet round-trip, and
    the stream equals the concatenated codewords."""
    import itertools
    alphabet = [120, 121, 127]
    for L in range(1, 7):
        for seq in itertools.product(alphabet, repeat=L):
            w = np.array([(e << 7) | (i * 37 % 128) | ((i & 1) << 15) for i, e in enumerate(seq)], np.uint16)
            d = O.DF11(w, n_bytes=1, threads=2)
            assert np.array_equal(d.decode(), w)
            want = "".join(format(int(d.codes[e]), f"0{int(d.lengths[e])}b") for e in seq)
            assert bits_of(d.stream)[: len(want)] == want


@pytest.mark.parametrize("make", [lambda: synth.make_weights(synth.single_1024()),
                                  lambda: synth.llama_bf16(2001, 1024, 4096)])
def test_rate_bounds(make):
    w = make()
    d = O.DF11(w)
    n = w.size
    h = O.entropy(d.counts)
    assert d.payload_bits >= n * h  # Shannon lower bound (DFloat11 Eq. (2))
    assert d.payload_bits < n * (h + 1)  # Huffman redundancy below one bit
    # payload (coded exponents + raw sign/mantissa byte) within 1% of the
    # Shannon payload bound n * (8 + H(exponent))
    assert d.payload_bits + 8 * n <= 1.01 * n * (8 + h)
    assert np.array_equal(d.decode(), w.ravel())


def test_corrupted_stream_is_detected_or_differs():
    w = synth.llama_bf16(2004, 32, 256)
    for bit in (3, 1000, 5001):
        d = O.DF11(w)
        d.flip_stream_bit(bit)
        try:
            out = d.decode()
        except ValueError:
            continue
        assert not np.array_equal(out, w.ravel())


def test_max_code_length_24_is_honoured():
    # Fibonacci counts give the deepest Huffman tree: 29 bits for 30 symbols
    fib = [1, 1]
    while len(fib) < 30:
        fib.append(fib[-1] + fib[-2])
    assert O.huffman_textbook(fib).max() == 29
    e = np.concatenate([np.full(f, 100 + i) for i, f in enumerate(fib)])
    w = (e.astype(np.uint16) << 7) | (np.arange(e.size) % 128).astype(np.uint16)
    d = O.DF11(w)
    assert d.lengths.max() == 24
    assert np.array_equal(d.decode(), w)
