"""Host side of the BF16-exponent rANS codec (kind 5): the library's blob against
the oracle's encoding of the same padded layout, word for word, its automatic
table size against the oracle's choice, and the validator (no GPU needed).

Source: MINE section 4 (BF16 handling: exponent coded, sign and mantissa a plain
byte; "Escapes"; "Pair" symbols) and section 4.2 ("Tuning t")."""
import ctypes
import struct

import numpy as np
import pytest

import oracle as O
import synth
from test_abi import hdr_offset, parse, raw_sign_mantissa


@pytest.fixture(scope="module")
def ec():
    import lossless_entropy_coded_gb300 as ec
    return ec


CASES = [((7, 300), 128, 3, 12, False), ((64, 1000), 4096, 0, 12, False), ((64, 1000), 4096, 0, 12, True),
         ((3, 4096), 1024, 2, 9, False), ((40, 4096), 4096, 16, 11, False), ((40, 4096), 4096, 40, 11, True),
         ((1, 1), 4096, 1, 10, True), ((33, 2048), 2048, 6, 12, False)]


@pytest.mark.parametrize("shape,tile,t,b,single", CASES)
def test_exp_blob_matches_oracle_stream(ec, shape, tile, t, b, single):
    w = synth.llama_bf16(8100 + shape[1] + t, *shape)
    W = ec.encode_bf16_exp(w, prob_bits=b, tile_syms=tile, top_t=t, single=single, device=-1)
    h, dev = parse(W.serialize())
    assert h["kind"] == ec.EC_KIND_RANS_EXP and h["k_pad"] == (shape[1] + 127) // 128 * 128
    wp = O.pad_rows(w).ravel()
    k = 1 if single else 2
    t_used = t or O.expx_choose_t(wp, k, 256 if single else 16, prob_bits=b, tile=tile)
    o = O.Expx(wp, t=t_used, prob_bits=b, tile=tile, k=k)
    assert h["fp8_table_size"] == o.tsize and h["rans_tuple"] == k
    assert h["n_tiles"] == o.n_tiles and h["n_escapes"] == o.n_records
    M = 1 << b
    tab = np.frombuffer(dev, np.uint32, M, h["table_off"]).astype(np.int64)
    payload, bias, f = tab & 0xFF, (tab >> 8) & 0xFFF, (tab >> 20) + 1
    table = o.table.astype(np.int64)
    if single:  # the entry carries the exponent itself: the oracle's symbol is its rank
        rank = np.full(256, -1)
        rank[table] = np.arange(o.tsize)
        sym = rank[payload]
        assert (sym >= 0).all()
    else:  # 16 r0 + r1 against the oracle's r0 * tsize + r1
        r0, r1 = payload >> 4, payload & 15
        assert (r0 < o.tsize).all() and (r1 < o.tsize).all()
        sym = r0 * o.tsize + r1
        vals = np.frombuffer(dev, np.uint32, 256, h["table_off"] + 4 * M).astype(np.int64)
        for a in range(o.tsize):
            for c in range(o.tsize):
                assert vals[16 * a + c] == (table[a] << 7) | (table[c] << 23)
    freqs = o.freqs.astype(np.int64)
    cum = np.concatenate([[0], np.cumsum(freqs)[:-1]])
    assert np.array_equal(np.bincount(sym, minlength=o.nsym), freqs)
    assert np.array_equal(f, freqs[sym]) and np.array_equal(bias, np.arange(M) - cum[sym])
    toff = np.frombuffer(dev, np.uint32, h["n_tiles"] + 1, h["tile_off_off"]).astype(np.int64)
    ooff, pay = o.offsets.astype(np.int64), o.payload()
    raw_t = 32 * ((h["steps"] + 15) // 16) * 16
    for tt in range(h["n_tiles"]):
        base = h["records_off"] + 16 * toff[tt]
        assert np.array_equal(np.frombuffer(dev, np.uint32, 32, base), o.states[tt]), tt
        nw = int(ooff[tt + 1] - ooff[tt])
        words = np.frombuffer(dev, np.uint16, 8 * (toff[tt + 1] - toff[tt]) - 64, base + 128)
        assert np.array_equal(words[:nw], pay[ooff[tt]:ooff[tt + 1]]), tt
        # sign / mantissa bytes: lane l's symbol i is position 32 i + l
        n_t = min(o.tile, o.n - tt * o.tile)
        raw = np.frombuffer(dev, np.uint8, raw_t, h["scales_off"] + tt * raw_t)
        S = n_t // 32
        sm = raw_sign_mantissa(raw[: 32 * ((S + 15) // 16) * 16], S)  # [symbol][lane]
        assert np.array_equal(sm.ravel(), o.sm[tt * o.tile: tt * o.tile + n_t]), tt
    eoff = np.frombuffer(dev, np.uint32, h["n_tiles"] + 1, h["esc_off_off"])
    assert np.array_equal(eoff, o.rec_off)
    recs = np.frombuffer(dev, np.uint32, h["n_escapes"], h["esc_records_off"]).astype(np.int64)
    orec = o.records.astype(np.int64)
    # the library's record carries the whole BF16 weight, the oracle's the exponent
    assert np.array_equal(recs & 0xFFFF, orec & 0xFFFF)
    assert np.array_equal((recs >> 23) & 0xFF, orec >> 16)
    for tt in range(h["n_tiles"]):
        for j in range(eoff[tt], eoff[tt + 1]):
            assert recs[j] >> 16 == wp[tt * o.tile + (recs[j] & 0xFFFF)]


def test_exp_payload_near_the_entropy(ec):
    """On LLM-like weights the pair code's stream plus records stays within 2% of the
    exponent entropy per weight (DFloat11 Eq. 2 gives the bound) over an 8-bit
    plain byte, and the whole blob is smaller than the Huffman-exponent blob of the
    same 4096 x 4096 matrix (MINE's BF16 results against DFloat11)."""
    w = synth.llama_bf16(8200, 4096, 4096)
    W = ec.encode_bf16_exp(w, device=-1)
    st = W.stats()
    n = w.size
    assert st["payload_bits"] / n <= 1.02 * st["entropy_bits"]
    assert st["bits_per_weight"] < ec.encode_bf16(w, device=-1).stats()["bits_per_weight"]


def test_exp_argument_validation(ec):
    from lossless_entropy_coded_gb300 import _ec
    w = synth.llama_bf16(8300, 4, 256)
    h = ctypes.c_void_p()

    def enc(n, k, prm=None):
        return _ec.lib.ec_encode_bf16_exp(w.ctypes.data, n, k, ctypes.byref(prm) if prm else None, -1, ctypes.byref(h))

    assert enc(4, 256) == 0
    _ec.lib.ec_free(h)
    assert enc(-1, 256) == _ec.EC_ERR_SHAPE
    for prm in [(13, 4096, 0, 0), (8, 4096, 0, 0), (12, 64, 0, 0), (12, 8192, 0, 0), (12, 4096, 17, 0),
                (12, 4096, 257, 1), (12, 4096, -1, 0), (12, 4096, 0, 2)]:
        assert enc(4, 256, _ec.ExpParams(*prm)) == _ec.EC_ERR_INVALID_ARG, prm


def test_exp_serialize_round_trip_and_structural_corruption(ec):
    w = synth.llama_bf16(8400, 20, 1000)
    w[3, 7] = 0x7F80  # an exponent (255) no small table keeps
    W = ec.encode_bf16_exp(w, top_t=5, device=-1)
    blob = W.serialize()
    W2 = ec.deserialize(blob, device=-1)
    assert W2.stats() == W.stats() and W2.kind == ec.EC_KIND_RANS_EXP
    h, dev = parse(blob)
    assert h["n_escapes"] > 2
    meta = len(blob) - len(dev)
    er = meta + h["esc_records_off"]
    rec0 = struct.unpack_from("<I", blob, er)[0]
    M = 1 << h["prob_bits"]
    cases = []
    for name, off, fmt, val in [("table size", meta + hdr_offset("fp8_table_size"), "<i", 0),
                                ("pair symbol outside the table", meta + h["table_off"], "<I", 0xFF | (1 << 20)),
                                ("pair value bits", meta + h["table_off"] + 4 * M, "<I", 1),
                                ("tuple", meta + hdr_offset("rans_tuple"), "<i", 3),
                                ("record position", er, "<I", 0xFFFF | (rec0 & 0xFFFF0000)),
                                ("record order", er + 4, "<I", rec0),
                                ("record count", meta + hdr_offset("n_escapes"), "<q", h["n_escapes"] - 1),
                                ("raw section", meta + hdr_offset("tile_off_off"), "<q", h["scales_off"] + 16)]:
        x = bytearray(blob)
        struct.pack_into(fmt, x, off, val)
        cases.append((name, bytes(x)))
    for name, bad in cases:
        with pytest.raises(ec.EcError) as e:
            ec.deserialize(bad, device=-1)
        assert e.value.code == -5, name


def test_exp_empty_matrix(ec):
    W = ec.encode_bf16_exp(np.zeros((0, 512), np.uint16), device=-1)
    h, _ = parse(W.serialize())
    assert h["n_tiles"] == 0 and h["n_rows"] == 0
    assert ec.deserialize(W.serialize(), device=-1).stats() == W.stats()


def test_exp_validator_survives_random_corruption(ec):
    rng = np.random.default_rng(55)
    W = ec.encode_bf16_exp(synth.llama_bf16(8500, 24, 1000), top_t=6, device=-1)
    blob = W.serialize()
    h, dev = parse(blob)
    meta = len(blob) - len(dev)
    hot = meta + h["records_off"] + 256
    for _ in range(300):
        x = bytearray(blob)
        for _ in range(int(rng.integers(1, 4))):
            x[int(rng.integers(meta, min(hot, len(x))))] = int(rng.integers(0, 256))
        try:
            ec.deserialize(bytes(x), device=-1)
        except ec.EcError as e:
            assert e.code == -5
