"""CPU-only tests of the C ABI: exported symbols, argument validation, the host
encoders (through host-only matrices and their serialised form), the untrusted-
input validator, and agreement of the library's code lengths / rANS frequencies
with the oracle's (same tie rules, independent implementations)."""
import ctypes
import os
import re
import struct

import numpy as np
import pytest

import oracle as O
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ec():
    from lossless_entropy_coded_gb300 import build
    build.build()
    import lossless_entropy_coded_gb300 as ec
    return ec


def declared_functions():
    src = open(os.path.join(ROOT, "include", "ec.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ec_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(ec):
    names = declared_functions()
    assert len(names) >= 14
    lib = ctypes.CDLL(ec.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ec.h but not exported"
    assert set(ec.EXPORTS) == set(names)


def test_strerror_codes(ec):
    for c in range(-7, 1):
        assert ec.strerror(c) and ec.strerror(c) != "unknown error"
    assert ec.strerror(-99) == "unknown error"


def rc_of(fn, *a):
    from lossless_entropy_coded_gb300 import _ec
    h = ctypes.c_void_p()
    return fn(*a, ctypes.byref(h)), h


def test_argument_validation(ec):
    from lossless_entropy_coded_gb300 import _ec
    lib = ec.lib
    w = np.zeros(16, np.uint16)
    bad = [(-1, 4, None, _ec.EC_ERR_SHAPE), (4, -1, None, _ec.EC_ERR_SHAPE),
           (2 ** 62, 1024, None, _ec.EC_ERR_OVERFLOW),
           (4, 4, _ec.HuffParams(0, 128), _ec.EC_ERR_INVALID_ARG),
           (4, 4, _ec.HuffParams(25, 128), _ec.EC_ERR_INVALID_ARG),
           (4, 4, _ec.HuffParams(24, 100), _ec.EC_ERR_INVALID_ARG)]
    for n, k, prm, want in bad:
        h = ctypes.c_void_p()
        rc = lib.ec_encode_bf16(w.ctypes.data, n, k, ctypes.byref(prm) if prm else None, -1, ctypes.byref(h))
        assert rc == want, (n, k, rc)
        assert not h.value
    assert lib.ec_encode_bf16(None, 4, 4, None, -1, ctypes.byref(ctypes.c_void_p())) == _ec.EC_ERR_INVALID_ARG
    assert lib.ec_encode_bf16(w.ctypes.data, 4, 4, None, -1, None) == _ec.EC_ERR_INVALID_ARG
    codes = np.array([[0, 8]], np.int8)
    sc = np.zeros((1, 1), np.uint16)
    h = ctypes.c_void_p()
    assert lib.ec_encode_rans(codes.ctypes.data, sc.ctypes.data, 1, 2, None, -1, ctypes.byref(h)) == _ec.EC_ERR_INVALID_ARG
    assert lib.ec_encode_rans(codes.ctypes.data, sc.ctypes.data, 1, 2, ctypes.byref(_ec.RansParams(12, 4096, 64, 0)),
                              -1, ctypes.byref(h)) == _ec.EC_ERR_UNSUPPORTED
    assert lib.ec_encode_rans(codes.ctypes.data, sc.ctypes.data, 1, 2, ctypes.byref(_ec.RansParams(8, 4096, 128, 0)),
                              -1, ctypes.byref(h)) == _ec.EC_ERR_INVALID_ARG
    # host-only matrices are rejected by the device entry points
    W = ec.encode_bf16(synth.gauss_bf16(1, (4, 8), 0.02), device=-1)
    assert lib.ec_gemv(W.handle, None, None, 1, None) == _ec.EC_ERR_INVALID_ARG
    assert lib.ec_gemv(W.handle, None, None, 0, None) == _ec.EC_ERR_INVALID_ARG
    assert lib.ec_gemv(W.handle, None, None, 65, None) == _ec.EC_ERR_UNSUPPORTED


# --------------------------------------------------------------- blob reader
HDR = struct.Struct("<IIii" + "q" * 10 + "i" * 6 + "Ii" + "qqq" + "iiiii")


HDR_KEYS = ["magic", "version", "kind", "steps", "n_rows", "k_cols", "k_pad", "n_tiles", "table_off",
            "table_words", "scales_off", "tile_off_off", "records_off", "blob_bytes", "max_code_bytes",
            "prob_bits", "max_words", "max_len", "rans_tuple", "window_code_bytes", "e8_scale_bits",
            "fp8_table_size", "esc_off_off", "esc_records_off", "n_escapes", "huff_flags", "huff_sub_tables",
            "huff_fill", "max_code_area", "rans_values"]


def hdr_offset(key: str) -> int:
    """Byte offset of a header field (the fields are naturally aligned: no padding)."""
    return struct.calcsize("<" + HDR.format[1:][: HDR_KEYS.index(key)])


def parse(blob: bytes):
    meta_size = 8 + 8 + 8 + 256 * 8 + 256 + 256 * 4 + 4 * 8 + 8
    dev = blob[meta_size:]
    f = HDR.unpack_from(dev, 0)
    keys = HDR_KEYS
    h = dict(zip(keys, f))
    return h, dev


def huff_pos(i: int, l: int) -> int:
    """Position in its tile of symbol i of lane l: 8 consecutive positions of every 256."""
    return 256 * (i // 8) + 8 * l + i % 8


def raw_sign_mantissa(raw_t: np.ndarray, S: int) -> np.ndarray:
    """Sign/mantissa bytes [symbol][lane] of a tile's raw section: lane-transposed
    16-byte chunks, and inside each group of four symbols i..i+3 the bits laid out so
    that a little-endian word r holds [w(i+1)|w(i)] under 0x807F807F and [w(i+3)|w(i+2)]
    under the same mask after rotating right by 8."""
    S16 = (S + 15) // 16 * 16
    g = raw_t.reshape(S16 // 16, 32, 4, 4)  # [chunk][lane][group][byte]
    b0, b1, b2, b3 = (g[..., j].astype(np.int64) for j in range(4))
    sm = np.stack([(b1 & 0x80) | (b0 & 0x7F),   # symbol i:   sign in byte 1, mantissa in byte 0
                   (b3 & 0x80) | (b2 & 0x7F),   # symbol i+1: sign in byte 3, mantissa in byte 2
                   (b2 & 0x80) | (b1 & 0x7F),   # symbol i+2: sign in byte 2, mantissa in byte 1
                   (b0 & 0x80) | (b3 & 0x7F)],  # symbol i+3: sign in byte 0, mantissa in byte 3
                  axis=-1)  # [chunk][lane][group][symbol in group]
    return sm.transpose(0, 2, 3, 1).reshape(S16, 32)[:S]


def area_bits(words: np.ndarray) -> str:
    """The code area as a string of bits in stream order (LSB first within each word)."""
    return "".join(format(int(x), "032b")[::-1] for x in words)


def tile_layout(h, dev, t):
    """(record offset, symbols per lane, sign/mantissa bytes, record count, code area offset,
    code area end) of tile t: lane starts (lane 0's slot holds the window record count),
    raw bytes, the code area, then the records (padded to 16 bytes)."""
    T = 32 * h["steps"]
    toff = np.frombuffer(dev, np.uint32, h["n_tiles"] + 1, h["tile_off_off"])
    rec = h["records_off"] + int(toff[t]) * 16
    S = min(T, h["n_rows"] * h["k_pad"] - t * T) // 32
    raw_bytes = 32 * ((S + 15) // 16 * 16)
    nrec = int(np.frombuffer(dev, np.uint16, 1, rec)[0])
    area_off = rec + 64 + raw_bytes
    area_end = h["records_off"] + int(toff[t + 1]) * 16 - 16 * ((4 * nrec + 15) // 16)
    return rec, S, raw_bytes, nrec, area_off, area_end


def lane_starts(dev, rec):
    st = np.frombuffer(dev, np.uint16, 32, rec).astype(np.int64).copy()
    st[0] = 0  # lane 0 starts at the area's first byte
    return st


def tile_records(h, dev, t, with_sm=False):
    """Window records of tile t: (position, true exponent, coded exponent[, sign/mantissa byte])
    from 13-bit position | sign and mantissa << 13 | exponent << 21."""
    rec, S, raw_bytes, nrec, _, area_end = tile_layout(h, dev, t)
    assert nrec == 0 or h["huff_flags"] & 1
    er = np.frombuffer(dev, np.uint32, nrec, area_end)
    out = []
    for i in range(nrec):
        r = int(er[i])
        assert r >> 29 == 0
        rec = (r & 0x1FFF, (r >> 21) & 0xFF, h["huff_fill"])
        out.append(rec + ((r >> 13) & 0xFF,) if with_sm else rec)
    return out


def read_huffman(blob: bytes, lengths: np.ndarray) -> np.ndarray:
    """Reconstruct the BF16 matrix from a Huffman blob with a bit-by-bit reader
    (canonical codewords, first bit first), then apply the window records."""
    h, dev = parse(blob)
    codes = O.canonical_codes(lengths)
    table = {(int(lengths[s]), int(codes[s])): s for s in range(256) if lengths[s]}
    n, k, kp, steps = h["n_rows"], h["k_cols"], h["k_pad"], h["steps"]
    T = 32 * steps
    toff = np.frombuffer(dev, np.uint32, h["n_tiles"] + 1, h["tile_off_off"])
    flat = np.zeros(n * kp, np.uint16)
    for t in range(h["n_tiles"]):
        rec, S, raw_bytes, _, area_off, area_end = tile_layout(h, dev, t)
        start = lane_starts(dev, rec)
        raw = raw_sign_mantissa(np.frombuffer(dev, np.uint8, raw_bytes, rec + 64), S)
        bits = area_bits(np.frombuffer(dev, np.uint32, (area_end - area_off) // 4, area_off))
        expo = {}
        for l in range(32):
            pos = 8 * int(start[l])
            for i in range(S):
                L, c = 0, 0
                while (L, c) not in table:
                    c = (c << 1) | (bits[pos] == "1")
                    L += 1
                    pos += 1
                    assert L <= 24
                expo[huff_pos(i, l)] = table[(L, c)]
        sm_of = {}
        for q, e_true, e_coded, sm in tile_records(h, dev, t, with_sm=True):
            assert expo[q] == e_coded
            expo[q] = e_true
            sm_of[q] = sm
        for l in range(32):
            for i in range(S):
                q = huff_pos(i, l)
                r = int(raw[i, l])
                assert sm_of.get(q, r) == r  # a record carries the weight's own sign and mantissa
                flat[t * T + q] = ((r & 0x80) << 8) | (expo[q] << 7) | (r & 0x7F)
    return flat.reshape(n, kp)[:, :k]


def walk_pair_table(blob: bytes):
    """Decode a Huffman blob the way a GPU lane does: two exponents per lookup of
    the pair table (indexed by the next 12 stream bits, the first at bit 0); an open
    entry (only without window records) takes a second lookup, and codewords longer
    than the window walk the sub-tables.  Window records then replace the coded
    exponents.  Returns the exponent of every padded position and whether every
    lane ended in the last byte before the next lane's start."""
    h, dev = parse(blob)
    tab = np.frombuffer(dev, np.uint32, h["table_words"], h["table_off"])
    pair, sub = tab[:4096], tab[4096:]
    T = 32 * h["steps"]
    n_pad = h["n_rows"] * h["k_pad"]
    toff = np.frombuffer(dev, np.uint32, h["n_tiles"] + 1, h["tile_off_off"])
    exps = np.zeros(n_pad, np.int64)
    ends_ok = True
    records = bool(h["huff_flags"] & 1)

    def win(bits, p, n):  # the next n stream bits, the first at bit 0
        return sum(1 << j for j in range(n) if bits[p + j] == "1")

    def long_cw(bits, p, ent):  # sub-table walk for a codeword longer than the window
        t, used = (ent >> 7) & 0x1FF, 12
        while True:
            e = int(sub[256 * t + win(bits, p + used, 8)])
            if not e & 0x80000000:
                break
            t, used = e & 0xFFFF, (e >> 16) & 31
        assert not e & 0x40000000
        return (e & 0xFFFF) >> 7, (e >> 16) & 31

    for t in range(h["n_tiles"]):
        rec, S, _, _, area_off, area_end = tile_layout(h, dev, t)
        start = lane_starts(dev, rec)
        words = np.frombuffer(dev, np.uint32, (area_end - area_off) // 4, area_off)
        bits = area_bits(words) + "0" * 64
        for l in range(32):
            p = 8 * int(start[l])
            for s in range(S // 2):
                e = int(pair[win(bits, p, 12)])
                if not e & 0x80000000:
                    x0, x1, adv = (e >> 7) & 255, (e >> 23) & 255, e & 15
                else:
                    assert not records, "an open pair entry in a stream with window records"
                    l0 = (e >> 16) & 15
                    x0, l0 = ((e >> 7) & 255, l0) if l0 else long_cw(bits, p, e)
                    f = int(pair[win(bits, p + l0, 12)])
                    l1 = (f >> 16) & 15
                    x1, l1 = ((f >> 7) & 255, l1) if l1 else long_cw(bits, p + l0, f)
                    adv = l0 + l1
                exps[t * T + huff_pos(2 * s, l)] = x0
                exps[t * T + huff_pos(2 * s + 1, l)] = x1
                p += adv
            if l < 31:
                ends_ok &= 8 * int(start[l + 1]) - 8 < p <= 8 * int(start[l + 1])
            else:
                ends_ok &= p + 64 <= 32 * len(words)
        for q, e_true, e_coded in tile_records(h, dev, t):
            assert exps[t * T + q] == e_coded
            exps[t * T + q] = e_true
    return exps, ends_ok


@pytest.mark.parametrize("hier", [False, True])
@pytest.mark.parametrize("case", ["llama", "fib24", "fib12", "fib12_256", "one_symbol", "all_patterns"])
def test_pair_table_walk_decodes_exponents(ec, case, hier):
    if case == "llama":
        w = synth.llama_bf16(2010, 24, 2048)
        W = ec.encode_bf16(w, device=-1, hierarchical=hier)
    elif case.startswith("fib"):
        steps = 256 if case.endswith("_256") else 0  # 8192-position tiles: records past position 4095
        case = case[:5]
        fib = [1, 1]
        while len(fib) < 30:
            fib.append(fib[-1] + fib[-2])
        e = np.concatenate([np.full(f, 100 + i) for i, f in enumerate(fib)])[: 64 * 4096]
        rng = np.random.default_rng(1)
        rng.shuffle(e)
        w = ((e.astype(np.uint16) << 7) | (np.arange(e.size) % 128).astype(np.uint16)).reshape(-1, 4096)[:8]
        W = ec.encode_bf16(w, max_code_len=int(case[3:]), tile_steps=steps, device=-1, hierarchical=hier)
        if steps and not hier:
            h0, d0 = parse(W.serialize())
            assert max(q for t in range(h0["n_tiles"]) for q, *_ in tile_records(h0, d0, t)) >= 4096
        # L=24: codewords longer than the window reach the sub-tables (or, with window
        # records, are coded as the shortest codeword and recorded);
        # L=12: the longest codeword fills the window exactly
        assert W.code_lengths().max() > 12 if case == "fib24" else W.code_lengths().max() == 12
    elif case == "one_symbol":
        w = np.full((3, 512), 0x3F80, np.uint16)
        W = ec.encode_bf16(w, device=-1, hierarchical=hier)
    else:
        w = np.arange(65536, dtype=np.uint16).reshape(256, 256)
        W = ec.encode_bf16(w, device=-1, hierarchical=hier)
    blob = W.serialize()
    h, _ = parse(blob)
    # window records unless asked otherwise, or unless two shortest codewords overflow
    # the window (the uniform histogram of all patterns: every codeword is 8 bits)
    assert h["huff_flags"] == (0 if hier or case == "all_patterns" else 1)
    if h["huff_flags"]:
        assert h["huff_sub_tables"] == 0
        if case in ("llama", "fib24"):
            assert h["n_escapes"] > 0
    elif case == "fib24":
        assert h["huff_sub_tables"] > 0
    exps, ends_ok = walk_pair_table(blob)
    kp = W.stats()["k_pad"]
    want = np.zeros((w.shape[0], kp), np.int64)
    want[:, : w.shape[1]] = (w >> 7) & 0xFF
    assert np.array_equal(exps.reshape(w.shape[0], kp), want)
    assert ends_ok


@pytest.mark.parametrize("hier", [False, True])
def test_window_records_bound(ec, hier):
    """Window records replace exactly the symbols of pairs whose codewords overflow the
    12-bit window: the record count equals what the code lengths imply (one record when
    the shortest codeword fits beside the first, else one or two)."""
    w = synth.llama_bf16(2011, 64, 4096)
    W = ec.encode_bf16(w, device=-1, hierarchical=hier)
    h, dev = parse(W.serialize())
    lens = W.code_lengths().astype(np.int64)
    if hier:
        assert h["huff_flags"] == 0 and h["n_escapes"] == 0
        return
    fill = int(np.argmin(np.where(lens > 0, lens, 99)))
    lf = lens[fill]
    e = ((w >> 7) & 0xFF).astype(np.int64)  # 4096 columns: one tile per row, no padding
    n_rec = 0
    for row in e:
        lanes = row.reshape(16, 32, 8).transpose(1, 0, 2).reshape(32, -1)  # [lane][symbol]
        for seq in lanes:
            a, b = lens[seq[0::2]], lens[seq[1::2]]
            over = a + b > 12
            first_fits = a + lf <= 12
            n_rec += int((over & first_fits).sum()) + int((over & ~first_fits).sum()) + int(
                (over & ~first_fits & (lf + b > 12)).sum())
    assert h["n_escapes"] == n_rec
    st = W.stats()
    assert 8 * 4 * h["n_escapes"] / w.size < 0.2  # records cost well under 0.2 bit per weight


@pytest.mark.parametrize("shape,steps", [((7, 13), 128), ((3, 300), 32), ((40, 1024), 64), ((2, 4097), 128),
                                         ((6, 8192), 256), ((5, 14336), 224), ((3, 5000), 240)])
def test_huffman_blob_reads_back(ec, shape, steps):
    w = synth.llama_bf16(2007, *shape)
    W = ec.encode_bf16(w, tile_steps=steps, device=-1)
    got = read_huffman(W.serialize(), W.code_lengths())
    assert np.array_equal(got, w)


def test_all_bf16_patterns_blob_reads_back(ec):
    w = np.arange(65536, dtype=np.uint16).reshape(128, 512)  # k_pad = K: no padding, uniform histogram
    W = ec.encode_bf16(w, device=-1)
    assert (W.code_lengths() == 8).all()
    assert np.array_equal(read_huffman(W.serialize(), W.code_lengths()), w)


@pytest.mark.parametrize("seed", range(8))
def test_code_lengths_match_oracle(ec, seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(2, 60))
    exps = rng.choice(np.arange(80, 140), n, replace=False)
    counts = np.floor(2.0 ** rng.uniform(0, 15, n)).astype(np.int64) + 1  # skewed, deep trees
    e = np.repeat(exps, counts)
    w = (e.astype(np.uint16) << 7) | (np.arange(e.size) % 128).astype(np.uint16)
    k = 512  # a multiple of the row alignment: no padding columns
    rows = (w.size + k - 1) // k
    pad = rows * k - w.size
    # pad with an exponent already present so the histogram matches the oracle's
    w = np.concatenate([w, np.full(pad, int(exps[0]) << 7, np.uint16)]).reshape(rows, k)
    for L in (24, 12, 9):
        if 2 ** L < n:
            continue
        W = ec.encode_bf16(w, max_code_len=L, device=-1)
        cnt = np.bincount(((w >> 7) & 0xFF).ravel(), minlength=256)
        assert np.array_equal(W.code_lengths(), O.code_lengths(cnt, L)), L


def test_rans_frequencies_match_oracle(ec):
    for seed in range(5):
        codes, scales = synth.make_rans_case(0, 64, 512)
        codes = np.clip(codes + seed - 2, -8, 7).astype(np.int8)
        W = ec.encode_rans(codes, scales, device=-1)
        h, dev = parse(W.serialize())
        tab = np.frombuffer(dev, np.uint32, h["table_words"], h["table_off"])
        sym = tab & 15
        freq_lib = np.bincount(sym, minlength=16)
        want = O.rans_freqs(np.bincount(codes.ravel().astype(np.int64) + 8, minlength=16))
        assert np.array_equal(freq_lib, want)
        assert ((tab >> 16) == want[sym]).all()


def rans_padded(codes: np.ndarray, k_pad: int) -> np.ndarray:
    """The codes laid out as the library encodes them: rows padded to k_pad with code 0."""
    n, k = codes.shape
    out = np.zeros((n, k_pad), dtype=np.int8)
    out[:, :k] = codes
    return out


@pytest.mark.parametrize("tuple_", [1, 2])
@pytest.mark.parametrize("shape,tile", [((64, 1000), 4096), ((7, 300), 128), ((3, 4096), 1024), ((1, 1), 4096)])
def test_rans_blob_matches_oracle_stream(ec, tuple_, shape, tile):
    """The library's table, tile states and payload words equal the oracle's own
    encoding of the padded code layout, word for word (single and pair symbols)."""
    codes, scales = synth.make_rans_case(3, *shape)
    W = ec.encode_rans(codes, scales, tile_syms=tile, device=-1, codes_per_symbol=tuple_)
    h, dev = parse(W.serialize())
    assert h["rans_tuple"] == tuple_
    r = O.Rans(rans_padded(codes, h["k_pad"]), 12, tile, k=tuple_)
    tab = np.frombuffer(dev, np.uint32, h["table_words"], h["table_off"]).astype(np.int64)
    freqs = r.freqs.astype(np.int64)
    cum = np.concatenate([[0], np.cumsum(freqs)[:-1]])
    if tuple_ == 1:
        sym, bias, f = tab & 15, (tab >> 4) & 0xFFF, tab >> 16
    else:
        sym, bias, f = tab & 0xFF, (tab >> 8) & 0xFFF, (tab >> 20) + 1
    assert np.array_equal(np.bincount(sym, minlength=r.nsym), freqs)
    assert np.array_equal(f, freqs[sym])
    assert np.array_equal(bias, np.arange(4096) - cum[sym])
    assert h["n_tiles"] == r.n_tiles
    toff = np.frombuffer(dev, np.uint32, h["n_tiles"] + 1, h["tile_off_off"]).astype(np.int64)
    ooff = r.offsets.astype(np.int64)
    for t in range(h["n_tiles"]):
        base = h["records_off"] + 16 * toff[t]
        st = np.frombuffer(dev, np.uint32, 32, base)
        assert np.array_equal(st, r.states[t]), t
        nw = int(ooff[t + 1] - ooff[t])
        words = np.frombuffer(dev, np.uint16, 8 * (toff[t + 1] - toff[t]) - 64, base + 128)
        ow = np.ctypeslib.as_array(
            (ctypes.c_uint16 * max(1, int(ooff[-1]))).from_address(O._L().orc_rans_payload_mut(r._h)))
        assert np.array_equal(words[:nw], ow[ooff[t]:ooff[t + 1]]), t
        assert len(words) - nw < 8 and not words[nw:].any()


@pytest.mark.parametrize("tuple_", [1, 2])
@pytest.mark.parametrize("case", ["gauss", "gauss_1024", "uniform", "peaked", "rare"])
def test_rans_automatic_table_size_matches_oracle(ec, tuple_, case):
    """prob_bits = 0: the library picks the table size the oracle's MINE rule picks
    from the histogram of the padded layout (single codes or pairs).  Small streams
    take 2^9 (the table dominates); 1024 x 4096 Gaussian codes take 2^10 / 2^11."""
    rng = np.random.default_rng(len(case) * 7 + tuple_)
    shape = (48, 1024)
    if case == "gauss_1024":
        codes = np.clip(np.round(np.random.default_rng(1).normal(0, 1.1, size=(1024, 4096))), -8, 7).astype(np.int8)
        scales = np.full((1024, 32), 0x2000, np.uint16)
        expect = {1: 10, 2: 11}[tuple_]
    elif case == "gauss":
        codes, scales = synth.make_rans_case(0, *shape)
    else:
        if case == "uniform":
            codes = rng.integers(-8, 8, size=shape)
        elif case == "peaked":
            codes = np.clip(np.round(rng.normal(0, 0.35, size=shape)), -8, 7)
        else:
            codes = np.zeros(shape)
            codes.flat[rng.choice(codes.size, 6, replace=False)] = [-8, -5, 3, 5, 6, 7]
        codes = codes.astype(np.int8)
        scales = np.full((shape[0], shape[1] // 128), 0x2000, np.uint16)
    W = ec.encode_rans(codes, scales, prob_bits=0, device=-1, codes_per_symbol=tuple_)
    h, _ = parse(W.serialize())
    padded = rans_padded(codes, h["k_pad"])
    counts = O.Rans(padded, 12, 4096, k=tuple_).counts
    assert h["prob_bits"] == O.rans_table_bits(counts)
    if case == "gauss_1024":
        assert h["prob_bits"] == expect


def test_rans_pair_limits(ec):
    from lossless_entropy_coded_gb300 import _ec
    codes, sc = synth.make_rans_case(0, 4, 256)
    h = ctypes.c_void_p()
    for prm, want in [((13, 4096, 128, 2), _ec.EC_ERR_INVALID_ARG), ((12, 4096, 128, 3), _ec.EC_ERR_INVALID_ARG),
                      ((12, 4096, 128, -1), _ec.EC_ERR_INVALID_ARG)]:
        assert _ec.lib.ec_encode_rans(codes.ctypes.data, sc.ctypes.data, 4, 256, ctypes.byref(_ec.RansParams(*prm)),
                                     -1, ctypes.byref(h)) == want, prm
    for b in (9, 12):
        W = ec.encode_rans(codes, sc, prob_bits=b, device=-1, codes_per_symbol=2)
        assert W.stats()["max_code_len"] == b


def corruptions(blob: bytes):
    h, dev = parse(blob)
    meta = len(blob) - len(dev)
    b = bytearray(blob)
    yield "truncated", bytes(b[:-16])
    x = bytearray(b); x[meta] ^= 1
    yield "magic", bytes(x)
    x = bytearray(b); struct.pack_into("<q", x, meta + 16 + 8 * 3, h["n_tiles"] + 1)
    yield "n_tiles", bytes(x)
    toff = meta + h["tile_off_off"]
    x = bytearray(b); struct.pack_into("<I", x, toff + 4, 0xFFFFFF)
    yield "tile offset", bytes(x)
    rec = meta + h["records_off"]
    if h["kind"] == 1:
        x = bytearray(b); struct.pack_into("<H", x, rec + 2 * 31, 0xFFFF)
        yield "lane start", bytes(x)
        x = bytearray(b); struct.pack_into("<I", x, meta + h["table_off"], 0x80000000 | 0x7FFF)
        yield "table pointer", bytes(x)
        x = bytearray(b); struct.pack_into("<i", x, meta + hdr_offset("window_code_bytes"), -1)
        yield "window size", bytes(x)
    else:
        x = bytearray(b); struct.pack_into("<I", x, meta + h["table_off"], 0 if h["rans_tuple"] == 1 else 0xFFF00)
        yield "slot entry", bytes(x)
        tup = meta + hdr_offset("rans_tuple")
        x = bytearray(b); struct.pack_into("<i", x, tup, 3)
        yield "codes per symbol", bytes(x)
        if h["rans_tuple"] == 2:
            pb = meta + hdr_offset("prob_bits")
            x = bytearray(b); struct.pack_into("<i", x, pb, 13)
            yield "pair precision", bytes(x)


@pytest.mark.parametrize("kind", ["huffman", "rans", "rans_pair"])
def test_deserialize_rejects_structural_corruption(ec, kind):
    if kind == "huffman":
        W = ec.encode_bf16(synth.llama_bf16(2008, 20, 1000), device=-1)
    else:
        W = ec.encode_rans(*synth.make_rans_case(0, 20, 1000), device=-1,
                           codes_per_symbol=2 if kind == "rans_pair" else 1)
    blob = W.serialize()
    W2 = ec.deserialize(blob, device=-1)
    assert W2.stats() == W.stats()
    for name, bad in corruptions(blob):
        with pytest.raises(ec.EcError) as e:
            ec.deserialize(bad, device=-1)
        assert e.value.code == -5, name


@pytest.mark.parametrize("shape,steps", [((300, 4096), 128), ((70, 14336), 0), ((40, 1000), 64), ((5, 300), 16),
                                         ((40, 14336), 224)])
def test_huffman_window_size_matches_tiles(ec, shape, steps):
    """The header's largest 31-row window of one tile column (64 bytes of lane
    starts plus the code area per tile), recomputed from the tile offsets."""
    W = ec.encode_bf16(synth.llama_bf16(3300 + shape[0], *shape), tile_steps=steps, device=-1)
    h, dev = parse(W.serialize())
    toff = np.frombuffer(dev, np.uint32, h["n_tiles"] + 1, h["tile_off_off"]).astype(np.int64) * 16
    code = np.diff(toff) - 64 - 32 * ((h["steps"] + 15) // 16 * 16)
    assert code.max() == h["max_code_bytes"]
    T = 32 * h["steps"]
    if h["k_pad"] % T:
        assert h["window_code_bytes"] == 0
    else:
        R = h["k_pad"] // T
        per = (64 + code).reshape(h["n_rows"], R)
        c = np.vstack([np.zeros((1, R), np.int64), np.cumsum(per, axis=0)])
        wmax = max(int((c[min(r + 31, h["n_rows"])] - c[r]).max()) for r in range(h["n_rows"]))
        assert h["window_code_bytes"] == wmax


def test_gemv_path_dispatch(ec):
    """Which kernels a GEMV takes, decided on the host: tensor cores from batch 6 when
    every tile lies inside a row and k_cols % 8 == 0, else CUDA cores."""
    from lossless_entropy_coded_gb300 import _ec
    if os.environ.get("EC_MMA_MIN_BATCH"):
        pytest.skip("threshold overridden")
    W = ec.encode_bf16(synth.llama_bf16(3400, 64, 4096), device=-1)
    assert [ec.gemv_path(W, b) for b in (1, 5, 6, 32, 64)] == ["cuda_cores"] * 2 + ["tensor_cores"] * 3
    Wodd = ec.encode_bf16(synth.llama_bf16(3401, 8, 13), device=-1)  # rows of x not 16-byte aligned
    assert ec.gemv_path(Wodd, 16) == "cuda_cores"
    Wx = ec.encode_bf16(synth.llama_bf16(3402, 8, 14336), tile_steps=128, device=-1)  # tiles cross rows
    assert ec.gemv_path(Wx, 16) == "cuda_cores"
    Wy = ec.encode_bf16(synth.llama_bf16(3403, 8, 14336), device=-1)  # automatic tiles: 32 steps, inside rows
    assert ec.gemv_path(Wy, 16) == "tensor_cores"
    assert ec.gemv_path([Wy, Wx], 16) == "cuda_cores"  # one matrix without the layout: the whole group
    # tiles inside rows but too wide for the tensor-core kernel's staging pools (31 rows of
    # 8192-weight tiles): CUDA cores
    Ww = ec.encode_bf16(synth.llama_bf16(3404, 64, 8192), tile_steps=256, device=-1)
    assert parse(Ww.serialize())[0]["k_pad"] % (32 * 256) == 0
    assert ec.gemv_path(Ww, 16) == "cuda_cores"
    R = ec.encode_rans(*synth.make_rans_case(0, 8, 4096), device=-1)
    assert ec.gemv_path(R, 16) == "cuda_cores"
    hs = (ctypes.c_void_p * 2)(W.handle.value, R.handle.value)
    assert ec.lib.ec_gemv_path(hs, 2, 16) == _ec.EC_ERR_SHAPE
    assert ec.lib.ec_gemv_path(hs, 1, 0) == _ec.EC_ERR_INVALID_ARG
    assert ec.lib.ec_gemv_path(hs, 1, 65) == _ec.EC_ERR_UNSUPPORTED


def test_tile_width_aux_bounds(ec):
    w = synth.llama_bf16(2001, 1024, 4096)
    for steps, lo, hi in ((128, 0.125, 0.25), (64, 0.25, 0.40)):
        W = ec.encode_bf16(w, tile_steps=steps, device=-1)
        s = W.stats()
        h, _ = parse(W.serialize())
        assert s["n_tiles"] == w.size // (32 * steps)
        # per tile: 64 B of lane starts, each lane's last byte (about 4 bits x 32
        # lanes) and the area's >= 8 zero bytes and 16-byte padding; besides these, the
        # window records (4 bytes each, padded to 16 per tile)
        rec_bytes = 4 * h["n_escapes"] + 12 * h["n_tiles"]
        assert h["huff_flags"] == 1 and 0 < rec_bytes * 8 / w.size < 0.2
        assert lo < (s["aux_bytes"] - rec_bytes) * 8 / w.size < hi, steps


def test_stats_accounting(ec):
    w = synth.llama_bf16(2001, 1024, 4096)
    W = ec.encode_bf16(w, tile_steps=128, device=-1)
    s = W.stats()
    n = w.size
    assert s["k_pad"] == 4096 and s["n_tiles"] == n // 4096
    cnt = np.bincount(((w >> 7) & 0xFF).ravel(), minlength=256)
    lens = W.code_lengths().astype(np.int64)
    assert s["entropy_bits"] == pytest.approx(O.entropy(cnt), rel=1e-12)
    # the stream holds every exponent's codeword except where a window record put the
    # shortest one in its place
    h, dev = parse(W.serialize())
    recs = [r for t in range(h["n_tiles"]) for r in tile_records(h, dev, t)]
    assert len(recs) == h["n_escapes"] > 0
    saved = sum(int(lens[e_true] - lens[e_coded]) for _, e_true, e_coded in recs)
    assert s["payload_bits"] == int((cnt * lens).sum()) - saved
    assert s["raw_bytes"] == n
    assert s["device_bytes"] * 8 / n == pytest.approx(s["bits_per_weight"])
    # aux (lane starts, byte alignment, 16-byte record padding, offsets) well under 0.25 bit per
    # weight, plus the window records
    assert (s["aux_bytes"] - 4 * len(recs)) * 8 / n < 0.25
    assert 10.5 < s["bits_per_weight"] < 11.3
    Wh = ec.encode_bf16(w, tile_steps=128, device=-1, hierarchical=True)
    sh = Wh.stats()
    assert sh["payload_bits"] == int((cnt * lens).sum()) and sh["aux_bytes"] * 8 / n < 0.25


# --------------------------------------------------------------- E8 lattice codec
def e8_padded(q2: np.ndarray, k_pad: int) -> np.ndarray:
    """The points laid out as the library encodes them: rows padded to k_pad with the zero point."""
    n, k = q2.shape
    out = np.zeros((n, k_pad), dtype=np.int8)
    out[:, :k] = q2
    return out


@pytest.mark.parametrize("shape,tile,b", [((3, 256), 32, 11), ((7, 264), 64, 9), ((40, 1024), 512, 11),
                                          ((1, 8), 32, 12), ((5, 4096), 1024, 10), ((33, 776), 96, 11)])
def test_e8_blob_matches_oracle_stream(ec, shape, tile, b):
    """The library's 17 tables, row scales, shared scale, tile states and payload
    words equal the oracle's own encoding of the padded point layout, word for word."""
    q2, r, s = synth.make_e8_case(6000 + shape[1], *shape)
    W = ec.encode_e8(q2, r, s, prob_bits=b, tile_vectors=tile, device=-1)
    h, dev = parse(W.serialize())
    assert h["kind"] == ec.EC_KIND_E8 and h["k_pad"] == (shape[1] + 255) // 256 * 256
    assert h["steps"] == tile // 32 and h["prob_bits"] == b
    assert struct.unpack("<f", struct.pack("<I", h["e8_scale_bits"]))[0] == np.float32(s)
    e = O.E8(e8_padded(q2, h["k_pad"]), prob_bits=b, tile=tile)
    assert h["n_tiles"] == e.n_tiles
    M = 1 << b
    fc = np.frombuffer(dev, np.uint32, O.E8_TABLES * O.E8_ALPHA, h["table_off"]).reshape(O.E8_TABLES, O.E8_ALPHA)
    assert np.array_equal(fc & 0xFFFF, e.freqs)
    cum = np.concatenate([np.zeros((O.E8_TABLES, 1), np.int64), np.cumsum(e.freqs, axis=1)[:, :-1]], axis=1)
    used = e.freqs.sum(axis=1) > 0
    assert np.array_equal((fc >> 16)[used], cum[used])
    ss = np.frombuffer(dev, np.uint8, O.E8_TABLES * M, h["table_off"] + 4 * fc.size).reshape(O.E8_TABLES, M)
    for t in np.nonzero(used)[0]:
        assert np.array_equal(ss[t], np.repeat(np.arange(O.E8_ALPHA), e.freqs[t])), t
    assert np.array_equal(np.frombuffer(dev, np.float32, shape[0], h["scales_off"]), r)
    toff = np.frombuffer(dev, np.uint32, h["n_tiles"] + 1, h["tile_off_off"]).astype(np.int64)
    ooff = e.offsets.astype(np.int64)
    pay = e.payload()
    for t in range(h["n_tiles"]):
        base = h["records_off"] + 16 * toff[t]
        assert np.array_equal(np.frombuffer(dev, np.uint32, 32, base), e.states[t]), t
        nw = int(ooff[t + 1] - ooff[t])
        words = np.frombuffer(dev, np.uint16, 8 * (toff[t + 1] - toff[t]) - 64, base + 128)
        assert np.array_equal(words[:nw], pay[ooff[t]:ooff[t + 1]]), t
        assert len(words) - nw < 8 and not words[nw:].any()
    st = W.stats()
    assert st["kind"] == ec.EC_KIND_E8 and st["n_rows"] == shape[0] and st["k_cols"] == shape[1]


def test_e8_argument_validation(ec):
    from lossless_entropy_coded_gb300 import _ec
    q2, r, s = synth.make_e8_case(17, 4, 256)
    h = ctypes.c_void_p()

    def enc(q, n, k, prm=None, scale=s, rs=r):
        qq = np.ascontiguousarray(q, np.int8)
        return _ec.lib.ec_encode_e8(qq.ctypes.data, rs.ctypes.data, scale, n, k,
                                    ctypes.byref(prm) if prm else None, -1, ctypes.byref(h))

    assert enc(q2, 4, 256) == 0
    _ec.lib.ec_free(h)
    assert enc(q2, 4, 252) == _ec.EC_ERR_SHAPE            # k_cols % 8
    assert enc(q2, -1, 256) == _ec.EC_ERR_SHAPE
    for prm in [(13, 512), (8, 512), (11, 48), (11, 2048), (11, -32)]:
        assert enc(q2, 4, 256, _ec.E8Params(*prm)) == _ec.EC_ERR_INVALID_ARG, prm
    assert enc(q2, 4, 256, scale=float("inf")) == _ec.EC_ERR_INVALID_ARG
    bad_r = r.copy(); bad_r[2] = np.nan
    assert enc(q2, 4, 256, rs=bad_r) == _ec.EC_ERR_INVALID_ARG
    big_r = r.copy(); big_r[1] = 3e38  # finite, but s * r_1 overflows FP32
    assert enc(q2, 4, 256, scale=4.0, rs=big_r) == _ec.EC_ERR_INVALID_ARG
    for v, why in [([1, 1, 1, 1, 1, 1, 1, -1], "odd number of -1 in the odd coset"),
                   ([2, 0, 0, 0, 0, 0, 0, 0], "odd sum in D8"), ([1, 0, 0, 0, 0, 0, 0, 1], "mixed parity"),
                   ([32, 0, 0, 0, 0, 0, 0, 0], "z_1 = 16 out of range"),
                   ([0, 0, 0, 0, 0, 0, 0, -34], "z_8 = -17: m out of range")]:
        qb = q2.copy()
        qb[1, 8:16] = v
        assert enc(qb, 4, 256) == _ec.EC_ERR_INVALID_ARG, why
    # the extremes of every field are accepted: z_j in -16..15, m in -8..7
    qe = np.zeros((4, 256), np.int8)
    qe[0, :8] = [-32, 30, 0, 0, 0, 0, 0, 2]          # c 0, z (-16, 15, 0 x 5, 1): m = 0
    qe[1, :8] = [31, 31, 31, 31, 31, 31, 31, -29]    # c 1, z (15 x 7, -15): odd sum7, m = -8
    qe[2, :8] = [0, 0, 0, 0, 0, 0, 0, -32]           # c 0, z_8 = -16: even sum7, m = -8
    qe[3, :8] = [2, 0, 0, 0, 0, 0, 0, 30]            # c 0, z_8 = 15: odd sum7, m = 7
    assert enc(qe, 4, 256, rs=np.ones(4, np.float32)) == 0
    _ec.lib.ec_free(h)


def test_e8_rejects_structural_corruption(ec):
    q2, r, s = synth.make_e8_case(23, 20, 1000)
    W = ec.encode_e8(q2, r, s, device=-1)
    blob = W.serialize()
    W2 = ec.deserialize(blob, device=-1)
    assert W2.stats() == W.stats() and W2.kind == ec.EC_KIND_E8
    h, dev = parse(blob)
    meta = len(blob) - len(dev)
    M = 1 << h["prob_bits"]
    fc = np.frombuffer(dev, np.uint32, 17 * 32, h["table_off"]).reshape(17, 32)
    ss0 = meta + h["table_off"] + 4 * 17 * 32
    unused = [t for t in range(17) if not (fc[t] & 0xFFFF).any()]
    cases = []
    for name, off, fmt, val in [("precision", meta + hdr_offset("prob_bits"), "<i", 13),
                                ("steps", meta + hdr_offset("steps"), "<i", 33),
                                ("frequency", meta + h["table_off"] + 4 * 40, "<I", int(fc[1, 8]) + 1),
                                ("slot symbol", ss0 + M + 5, "<B", 31),
                                ("tile offset", meta + h["tile_off_off"] + 4, "<I", 0xFFFFFF),
                                ("max words", meta + hdr_offset("max_words"), "<i", 1)]:
        x = bytearray(blob); struct.pack_into(fmt, x, off, val)
        cases.append((name, bytes(x)))
    if unused:
        x = bytearray(blob); struct.pack_into("<B", x, ss0 + unused[0] * M + 3, 7)
        cases.append(("unused table slot", bytes(x)))
    # a consistent coset table with a third symbol: one slot moved from symbol 1 to 2
    f0, f1 = int(fc[0, 0] & 0xFFFF), int(fc[0, 1] & 0xFFFF)
    x = bytearray(blob)
    struct.pack_into("<I", x, meta + h["table_off"] + 4, (f1 - 1) | (f0 << 16))
    struct.pack_into("<I", x, meta + h["table_off"] + 8, 1 | ((M - 1) << 16))
    for s in range(3, 32):
        struct.pack_into("<I", x, meta + h["table_off"] + 4 * s, M << 16)
    struct.pack_into("<B", x, ss0 + M - 1, 2)
    cases.append(("third coset", bytes(x)))
    for name, bad in cases:
        with pytest.raises(ec.EcError) as e:
            ec.deserialize(bad, device=-1)
        assert e.value.code == -5, name


def test_decode_as_argument_checks(ec):
    from lossless_entropy_coded_gb300 import _ec
    assert _ec.lib.ec_decode_as(None, None, 0, None) == _ec.EC_ERR_INVALID_ARG
    q2, r, s = synth.make_e8_case(31, 8, 256)
    W = ec.encode_e8(q2, r, s, device=-1)  # host-only: no device blob
    assert _ec.lib.ec_decode_as(W.handle, None, 1, None) == _ec.EC_ERR_INVALID_ARG


def test_e8_matrices_have_no_gemv(ec):
    """EntroPack decodes to a dense matrix: the GEMV query (and the GEMV) refuse E8 matrices."""
    q2, r, s = synth.make_e8_case(29, 8, 256)
    W = ec.encode_e8(q2, r, s, device=-1)
    with pytest.raises(ec.EcError) as e:
        ec.gemv_path([W], 1)
    assert e.value.code == -4


# --------------------------------------------------------------- FP8 top-t tables with escapes
def fp8_padded(codes: np.ndarray, k_pad: int) -> np.ndarray:
    n, k = codes.shape
    out = np.zeros((n, k_pad), dtype=np.uint8)
    out[:, :k] = codes
    return out


@pytest.mark.parametrize("shape,tile,t,b", [((7, 300), 128, 16, 12), ((64, 1000), 4096, 0, 12),
                                            ((3, 4096), 1024, 2, 9), ((1, 1), 4096, 1, 10),
                                            ((40, 4096), 4096, 64, 11)])
def test_fp8_blob_matches_oracle_stream(ec, shape, tile, t, b):
    """The library's slot table, symbol values, states, payload words and correction
    records equal the oracle's encoding of the padded layout, word for word."""
    codes, r = synth.make_fp8_case(8000 + shape[1], *shape)
    W = ec.encode_fp8(codes, r, top_t=t, prob_bits=b, tile_syms=tile, device=-1)
    h, dev = parse(W.serialize())
    assert h["kind"] == ec.EC_KIND_RANS_FP8 and h["k_pad"] == (shape[1] + 127) // 128 * 128
    o = O.Fp8(fp8_padded(codes, h["k_pad"]), t=t or 256, prob_bits=b, tile=tile)
    assert h["fp8_table_size"] == o.tsize and h["n_tiles"] == o.n_tiles and h["n_escapes"] == o.n_records
    M = 1 << b
    tab = np.frombuffer(dev, np.uint32, M, h["table_off"]).astype(np.int64)
    freqs = o.freqs.astype(np.int64)
    cum = np.concatenate([[0], np.cumsum(freqs)[:-1]])
    sym, bias, f = tab & 0xFF, (tab >> 8) & 0xFFF, (tab >> 20) + 1
    assert np.array_equal(np.bincount(sym, minlength=o.tsize), freqs)
    assert np.array_equal(f, freqs[sym]) and np.array_equal(bias, np.arange(M) - cum[sym])
    vals = np.frombuffer(dev, np.float32, 512, h["table_off"] + 4 * M)
    assert np.array_equal(vals[: o.tsize], O.e4m3_to_f32(o.table)) and not vals[o.tsize:256].any()
    allv = O.e4m3_to_f32(np.arange(256))
    assert np.array_equal(vals[256:], allv, equal_nan=True)
    assert np.array_equal(np.frombuffer(dev, np.float32, shape[0], h["scales_off"]), r)
    toff = np.frombuffer(dev, np.uint32, h["n_tiles"] + 1, h["tile_off_off"]).astype(np.int64)
    ooff, pay = o.offsets.astype(np.int64), o.payload()
    for tt in range(h["n_tiles"]):
        base = h["records_off"] + 16 * toff[tt]
        assert np.array_equal(np.frombuffer(dev, np.uint32, 32, base), o.states[tt]), tt
        nw = int(ooff[tt + 1] - ooff[tt])
        words = np.frombuffer(dev, np.uint16, 8 * (toff[tt + 1] - toff[tt]) - 64, base + 128)
        assert np.array_equal(words[:nw], pay[ooff[tt]:ooff[tt + 1]]), tt
    eoff = np.frombuffer(dev, np.uint32, h["n_tiles"] + 1, h["esc_off_off"])
    assert np.array_equal(eoff, o.rec_off)
    recs = np.frombuffer(dev, np.uint32, h["n_escapes"], h["esc_records_off"])
    assert np.array_equal(recs, o.records)
    if t == 0:
        assert h["n_escapes"] == 0


def test_fp8_argument_validation(ec):
    from lossless_entropy_coded_gb300 import _ec
    codes, r = synth.make_fp8_case(5, 4, 256)
    h = ctypes.c_void_p()

    def enc(c, n, k, prm=None, rs=r):
        cc = np.ascontiguousarray(c, np.uint8)
        return _ec.lib.ec_encode_fp8(cc.ctypes.data, rs.ctypes.data, n, k, ctypes.byref(prm) if prm else None, -1,
                                     ctypes.byref(h))

    assert enc(codes, 4, 256) == 0
    _ec.lib.ec_free(h)
    assert enc(codes, -1, 256) == _ec.EC_ERR_SHAPE
    for prm in [(13, 4096, 0), (8, 4096, 0), (12, 64, 0), (12, 8192, 0), (12, 4096, 257), (12, 4096, -1)]:
        assert enc(codes, 4, 256, _ec.Fp8Params(*prm)) == _ec.EC_ERR_INVALID_ARG, prm
    for nan in (0x7F, 0xFF):
        bad = codes.copy(); bad[2, 9] = nan
        assert enc(bad, 4, 256) == _ec.EC_ERR_INVALID_ARG
    bad_r = r.copy(); bad_r[0] = np.inf
    assert enc(codes, 4, 256, rs=bad_r) == _ec.EC_ERR_INVALID_ARG


def test_fp8_rejects_structural_corruption(ec):
    codes, r = synth.make_fp8_case(6, 20, 1000)
    W = ec.encode_fp8(codes, r, top_t=24, device=-1)
    blob = W.serialize()
    W2 = ec.deserialize(blob, device=-1)
    assert W2.stats() == W.stats() and W2.kind == ec.EC_KIND_RANS_FP8
    h, dev = parse(blob)
    assert h["n_escapes"] > 2
    meta = len(blob) - len(dev)
    er = meta + h["esc_records_off"]
    rec0 = struct.unpack_from("<I", blob, er)[0]
    cases = []
    for name, off, fmt, val in [("table size", meta + hdr_offset("fp8_table_size"), "<i", 0),
                                ("symbol outside the table", meta + h["table_off"], "<I", 200 | (1 << 20)),
                                ("record position", er, "<I", 0xFFFF | (rec0 & 0xFF0000)),
                                ("record high bits", er, "<I", rec0 | 0x01000000),
                                ("record order", er + 4, "<I", rec0),
                                ("record count", meta + hdr_offset("n_escapes"), "<q", h["n_escapes"] - 1),
                                ("record offsets", meta + h["esc_off_off"] + 4, "<I", 0xFFFFFF)]:
        x = bytearray(blob); struct.pack_into(fmt, x, off, val)
        cases.append((name, bytes(x)))
    for name, bad in cases:
        with pytest.raises(ec.EcError) as e:
            ec.deserialize(bad, device=-1)
        assert e.value.code == -5, name


@pytest.mark.parametrize("kind", ["fp8", "e8", "rans", "huffman"])
def test_empty_matrices_round_trip(ec, kind):
    """0 rows: every encoder gives a blob the validator accepts (no tiles, no records)."""
    if kind == "fp8":
        W = ec.encode_fp8(np.zeros((0, 512), np.uint8), np.zeros(0, np.float32), device=-1)
    elif kind == "e8":
        W = ec.encode_e8(np.zeros((0, 256), np.int8), np.zeros(0, np.float32), 1.0, device=-1)
    elif kind == "rans":
        W = ec.encode_rans(np.zeros((0, 512), np.int8), np.zeros((0, 4), np.uint16), device=-1)
    else:
        W = ec.encode_bf16(np.zeros((0, 512), np.uint16), device=-1)
    h, _ = parse(W.serialize())
    assert h["n_tiles"] == 0 and h["n_rows"] == 0
    W2 = ec.deserialize(W.serialize(), device=-1)
    assert W2.stats() == W.stats()


@pytest.mark.parametrize("kind", ["huffman", "rans", "rans_pair", "e8", "fp8"])
def test_validator_survives_random_corruption(ec, kind):
    """Random byte changes anywhere in the metadata part of a blob (header, tables,
    offsets, records): deserialisation accepts or reports EC_ERR_CORRUPT, never
    anything else (and never crashes)."""
    rng = np.random.default_rng(len(kind))
    if kind == "huffman":
        W = ec.encode_bf16(synth.llama_bf16(9001, 24, 1000), device=-1)
    elif kind.startswith("rans"):
        W = ec.encode_rans(*synth.make_rans_case(0, 24, 1000), device=-1, codes_per_symbol=2 if kind == "rans_pair" else 1)
    elif kind == "e8":
        q2, r, s = synth.make_e8_case(9002, 24, 1000)
        W = ec.encode_e8(q2, r, s, tile_vectors=96, device=-1)
    else:
        W = ec.encode_fp8(*synth.make_fp8_case(9003, 24, 1000), top_t=20, device=-1)
    blob = W.serialize()
    h, dev = parse(blob)
    meta = len(blob) - len(dev)
    hot = meta + h["records_off"] + 256  # header, tables, scales, offsets and the first records
    for _ in range(300):
        x = bytearray(blob)
        for _ in range(int(rng.integers(1, 4))):
            x[int(rng.integers(meta, min(hot, len(x))))] = int(rng.integers(0, 256))
        try:
            ec.deserialize(bytes(x), device=-1)
        except ec.EcError as e:
            assert e.code == -5



@pytest.mark.parametrize("tuple_", [1, 2])
def test_fp4_codes_are_the_integer_stream_of_code_minus_8(ec, tuple_):
    """values="fp4": E2M1 patterns 0..15 go through the integer codec as c - 8; the
    header marks the reading and the stream equals the oracle's coding of c - 8."""
    codes, scales = synth.make_fp4_case(3500, 40, 1000)
    W = ec.encode_rans(codes, scales, device=-1, codes_per_symbol=tuple_, values="fp4")
    h, dev = parse(W.serialize())
    assert h["rans_values"] == 1 and h["rans_tuple"] == tuple_
    Wi = ec.encode_rans((codes - 8).astype(np.int8), scales, device=-1, codes_per_symbol=tuple_)
    hi, devi = parse(Wi.serialize())
    assert hi["rans_values"] == 0
    # tables, scales, offsets and tiles byte for byte (the integer blob's stream is
    # the oracle's word for word: test_rans_blob_matches_oracle_stream)
    assert dev[256:] == devi[256:]


def test_fp4_and_int4_code_ranges_are_checked(ec):
    sc = np.full((1, 1), 0x3C00, np.uint16)
    with pytest.raises(ec.EcError):
        ec.encode_rans(np.array([[16]], np.int8), sc, device=-1, values="fp4")
    with pytest.raises(ec.EcError):
        ec.encode_rans(np.array([[-1]], np.int8), sc, device=-1, values="fp4")
    with pytest.raises(ec.EcError):
        ec.encode_rans(np.array([[8]], np.int8), sc, device=-1)
    from lossless_entropy_coded_gb300 import _ec
    import ctypes
    h = ctypes.c_void_p()
    c = np.array([[1]], np.int8)
    assert _ec.lib.ec_encode_rans(c.ctypes.data, sc.ctypes.data, 1, 1, ctypes.byref(_ec.RansParams(12, 4096, 128, 1, 2)),
                                  -1, ctypes.byref(h)) == _ec.EC_ERR_INVALID_ARG
