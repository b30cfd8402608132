"""CPU oracle for the entropy-coded weight path -- TEST INFRASTRUCTURE ONLY.

The library under lossless_entropy_coded_gb300/ never imports this package.
Only tests/, ``__graft_entry__.smoke()`` and the CPU-baseline leg of bench.py
use it.  The arithmetic lives in ``oracle.c`` (plain C, FP64 sums in index
order); this module only marshals arrays through ctypes.

Functions and the passages they follow (page titles and sections):
  entropy, cross_entropy        DFloat11 Eq.(2); MINE sec. 4.2 "Compressed Size Prediction"
  huffman_textbook              DFloat11 sec. "entropy coding" (Huffman's merge rule)
  package_merge                 Larmore & Hirschberg's optimal length-limited code
  canonical_codes               consistent with DFloat11 Fig. 13
  flat_lut / hier_luts          DFloat11 appendix, Fig. 13 and Fig. 14
  DF11 (encode/decode)          DFloat11 sec. "Dynamic-Length Float", "two-phase kernel", Algorithm 1
  Rans (encode/decode)          EntroPack sec. 3.6 and appendix C.3; Duda's rANS
  rans_table_bits               MINE sec. 4.2 "Launch" (table size by the cross-entropy bound)
  e8_fields / e8_point / E8     EntroPack sec. 3.2, 3.3, 3.6, 3.7, appendix A.3 (E8 fields, 17 tables)
  e8_reconstruct_bf16           EntroPack sec. 3.7 (lattice point x shared scale x row scale)
  Fp8 / fp8_table / e4m3_to_f32 MINE sec. 4 "Escapes" (top-t table, sparse correction records)
  Expx / expx_bound / expx_choose_t / pad_rows
                                MINE sec. 4: BF16 exponents through rANS tiles with a top-t
                                table, escapes and "Pair" symbols; sec. 4.2 "Tuning t"
  fp8_dequant_bf16 / gemv_fp8   FP8 E4M3 weights with FP32 row scales
  e8_reconstruct / f32_to_e4m3 / f32_to_s8
                                EntroPack sec. 3.7 and appendix B.1 (FP8 / INT8 output); the OCP
                                FP8 E4M3 format
  gemv_bf16 / gemv_rans         y = W x with FP64 accumulation
  e2m1_value                    the OCP Microscaling FP4 E2M1 format (MINE "Data Types" names
                                FP4 among the k-tuple types); rans_dequant_bf16 / gemv_rans
                                take values="fp4" for 4-bit codes that are E2M1 patterns

Every function is pinned by tests in tests/test_oracle_*.py against the pages'
worked examples, closed forms, invariants or brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source (plain gcc)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-Wall", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _L():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    vp, i64, i32, f64, u16 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_uint16
    sig = {
        "orc_bf16_to_f64": ([u16], f64),
        "orc_f16_to_f32": ([u16], ctypes.c_float),
        "orc_f32_to_bf16_rne": ([ctypes.c_float], u16),
        "orc_entropy": ([vp, i32], f64),
        "orc_cross_entropy": ([vp, vp, i32, i32], f64),
        "orc_huffman_textbook": ([vp, vp], i32),
        "orc_package_merge": ([vp, i32, vp], i32),
        "orc_code_lengths": ([vp, i32, vp], i32),
        "orc_canonical_codes": ([vp, vp], None),
        "orc_flat_lut": ([vp, vp, i32, vp], i32),
        "orc_hier_luts": ([vp, vp, i32, vp, i32], i32),
        "orc_df11_encode": ([vp, i64, i32, i32, i32], vp),
        "orc_df11_decode": ([vp, vp], i32),
        "orc_df11_free": ([vp], None),
        "orc_df11_info": ([vp, vp], i64),
        "orc_df11_lengths": ([vp], vp),
        "orc_df11_codes": ([vp], vp),
        "orc_df11_counts": ([vp], vp),
        "orc_df11_stream": ([vp], vp),
        "orc_df11_gaps": ([vp], vp),
        "orc_df11_block_pos": ([vp], vp),
        "orc_df11_luts": ([vp], vp),
        "orc_df11_sm_mut": ([vp], vp),
        "orc_df11_stream_mut": ([vp], vp),
        "orc_rans_freqs": ([vp, i32, vp], i32),
        "orc_rans_freqs_n": ([vp, i32, i32, vp], i32),
        "orc_rans_encode": ([vp, i64, i32, i32], vp),
        "orc_rans_encode_k": ([vp, i64, i32, i32, i32], vp),
        "orc_rans_decode": ([vp, vp, vp], i32),
        "orc_rans_free": ([vp], None),
        "orc_rans_info": ([vp, vp], i64),
        "orc_rans_freqs_of": ([vp], vp),
        "orc_rans_counts_of": ([vp], vp),
        "orc_rans_states": ([vp], vp),
        "orc_rans_offsets": ([vp], vp),
        "orc_rans_payload_mut": ([vp], vp),
        "orc_rans_dequant_bf16": ([vp, vp, i64, i64, i32, vp], None),
        "orc_rans_dequant_bf16_v": ([vp, vp, i64, i64, i32, i32, vp], None),
        "orc_gemv_rans_v": ([vp, vp, i64, i64, i32, i32, vp, i32, vp, i64, vp, vp], None),
        "orc_e2m1_value": ([i32], ctypes.c_double),
        "orc_gemv_bf16": ([vp, i64, i64, vp, i32, vp, i64, vp, vp], None),
        "orc_gemv_rans": ([vp, vp, i64, i64, i32, vp, i32, vp, i64, vp, vp], None),
        "orc_e8_fields": ([vp, vp], i32),
        "orc_e8_point": ([vp, vp], None),
        "orc_e8_encode": ([vp, i64, i32, i32], vp),
        "orc_e8_decode": ([vp, vp, vp], i32),
        "orc_e8_free": ([vp], None),
        "orc_e8_info": ([vp, vp], i64),
        "orc_e8_freqs_of": ([vp], vp),
        "orc_e8_counts_of": ([vp], vp),
        "orc_e8_states": ([vp], vp),
        "orc_e8_offsets": ([vp], vp),
        "orc_e8_payload_mut": ([vp], vp),
        "orc_e8_reconstruct_bf16": ([vp, i64, i64, ctypes.c_float, vp, vp], None),
        "orc_e8_reconstruct_as": ([vp, i64, i64, ctypes.c_float, vp, i32, vp], None),
        "orc_f32_to_e4m3_satfinite": ([ctypes.c_float], ctypes.c_uint8),
        "orc_f32_to_s8_rne_sat": ([ctypes.c_float], ctypes.c_int8),
        "orc_e4m3_to_f32": ([ctypes.c_uint8], ctypes.c_float),
        "orc_fp8_table": ([vp, i32, vp], i32),
        "orc_fp8_encode": ([vp, i64, i32, i32, i32], vp),
        "orc_fp8_decode": ([vp, vp], i32),
        "orc_fp8_free": ([vp], None),
        "orc_fp8_info": ([vp, vp], i64),
        "orc_fp8_table_of": ([vp], vp),
        "orc_fp8_freqs_of": ([vp], vp),
        "orc_fp8_counts_of": ([vp], vp),
        "orc_fp8_states": ([vp], vp),
        "orc_fp8_offsets": ([vp], vp),
        "orc_fp8_payload_mut": ([vp], vp),
        "orc_fp8_rec_off": ([vp], vp),
        "orc_fp8_records": ([vp], vp),
        "orc_expx_bound": ([vp, i64, i32, i32, i32, i32], f64),
        "orc_expx_choose_t": ([vp, i64, i32, i32, i32, i32], i32),
        "orc_expx_encode": ([vp, i64, i32, i32, i32, i32], vp),
        "orc_expx_decode": ([vp, vp], i32),
        "orc_expx_free": ([vp], None),
        "orc_expx_info": ([vp, vp], i64),
        "orc_expx_table_of": ([vp], vp),
        "orc_expx_freqs_of": ([vp], vp),
        "orc_expx_counts_of": ([vp], vp),
        "orc_expx_states": ([vp], vp),
        "orc_expx_offsets": ([vp], vp),
        "orc_expx_payload_mut": ([vp], vp),
        "orc_expx_rec_off": ([vp], vp),
        "orc_expx_records": ([vp], vp),
        "orc_expx_sm": ([vp], vp),
        "orc_fp8_dequant_bf16": ([vp, vp, i64, i64, vp], None),
        "orc_gemv_fp8": ([vp, vp, i64, i64, vp, i32, vp, i64, vp, vp], None),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _p(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "arrays passed to the oracle must be C-contiguous"
    return a.ctypes.data


def _view(addr: int, dtype, n: int) -> np.ndarray:
    if n == 0:
        return np.empty(0, dtype=dtype)
    buf = (ctypes.c_char * (n * np.dtype(dtype).itemsize)).from_address(addr)
    return np.frombuffer(buf, dtype=dtype, count=n).copy()


# --------------------------------------------------------------------------- scalars
def bf16_to_f64(h: int) -> float:
    return float(_L().orc_bf16_to_f64(h))


def f16_to_f32(h: int) -> float:
    return float(_L().orc_f16_to_f32(h))


def f32_to_bf16_rne(f: float) -> int:
    return int(_L().orc_f32_to_bf16_rne(f))


# --------------------------------------------------------------------------- entropy
def entropy(counts) -> float:
    c = np.ascontiguousarray(counts, dtype=np.uint64)
    return float(_L().orc_entropy(_p(c), len(c)))


def cross_entropy(counts, freqs, prob_bits: int) -> float:
    c = np.ascontiguousarray(counts, dtype=np.uint64)
    f = np.ascontiguousarray(freqs, dtype=np.uint32)
    return float(_L().orc_cross_entropy(_p(c), _p(f), len(c), prob_bits))


# --------------------------------------------------------------------------- Huffman
def _counts256(counts) -> np.ndarray:
    c = np.zeros(256, dtype=np.uint64)
    cc = np.asarray(counts, dtype=np.uint64)
    c[: len(cc)] = cc
    return c


def huffman_textbook(counts) -> np.ndarray:
    c = _counts256(counts)
    out = np.zeros(256, dtype=np.uint8)
    _L().orc_huffman_textbook(_p(c), _p(out))
    return out


def package_merge(counts, max_len: int) -> np.ndarray:
    c = _counts256(counts)
    out = np.zeros(256, dtype=np.uint8)
    if _L().orc_package_merge(_p(c), max_len, _p(out)) < 0:
        raise ValueError("no prefix code with that length limit")
    return out


def code_lengths(counts, max_len: int = 24) -> np.ndarray:
    c = _counts256(counts)
    out = np.zeros(256, dtype=np.uint8)
    if _L().orc_code_lengths(_p(c), max_len, _p(out)) < 0:
        raise ValueError("no prefix code with that length limit")
    return out


def canonical_codes(lengths) -> np.ndarray:
    ln = np.zeros(256, dtype=np.uint8)
    ln[: len(lengths)] = lengths
    out = np.zeros(256, dtype=np.uint32)
    _L().orc_canonical_codes(_p(ln), _p(out))
    return out


def flat_lut(lengths, codes, L: int) -> np.ndarray:
    ln = np.zeros(256, dtype=np.uint8)
    ln[: len(lengths)] = lengths
    cd = np.zeros(256, dtype=np.uint32)
    cd[: len(codes)] = codes
    out = np.zeros(1 << L, dtype=np.int16)
    if _L().orc_flat_lut(_p(ln), _p(cd), L, _p(out)) < 0:
        raise ValueError("flat LUT needs L >= the longest code")
    return out


def hier_luts(lengths, codes, b: int, max_tables: int = 4096) -> np.ndarray:
    """Returns [k, 2^b] int16: 0..255 symbol, 256+t pointer to table t, -1 unused."""
    ln = np.zeros(256, dtype=np.uint8)
    ln[: len(lengths)] = lengths
    cd = np.zeros(256, dtype=np.uint32)
    cd[: len(codes)] = codes
    buf = np.zeros(max_tables * (1 << b), dtype=np.int16)
    k = _L().orc_hier_luts(_p(ln), _p(cd), b, _p(buf), max_tables)
    if k < 0:
        raise ValueError("too many tables")
    return buf[: k * (1 << b)].reshape(k, 1 << b)


# --------------------------------------------------------------------------- DF11 codec
class DF11:
    """DFloat11-format encoding of a BF16 array (EncodedExponent, PackedSignMantissa,
    Gaps, BlockOutputPos, hierarchical LUTs with b = 8)."""

    def __init__(self, w_bf16: np.ndarray, max_len: int = 24, n_bytes: int = 8, threads: int = 256):
        w = np.ascontiguousarray(w_bf16, dtype=np.uint16).ravel()
        self._w_keepalive = w
        h = _L().orc_df11_encode(_p(w), w.size, max_len, n_bytes, threads)
        if not h:
            raise ValueError("DF11 encode failed")
        self._h = h
        info = np.zeros(8, dtype=np.int64)
        _L().orc_df11_info(h, _p(info))
        (self.n, self.n_bytes, self.threads, self.n_chunks, self.n_blocks, self.stream_bytes,
         self.payload_bits, self.n_luts) = (int(v) for v in info)

    def __del__(self):
        if getattr(self, "_h", None):
            _L().orc_df11_free(self._h)
            self._h = None

    @property
    def lengths(self):
        return _view(_L().orc_df11_lengths(self._h), np.uint8, 256)

    @property
    def codes(self):
        return _view(_L().orc_df11_codes(self._h), np.uint32, 256)

    @property
    def counts(self):
        return _view(_L().orc_df11_counts(self._h), np.uint64, 256)

    @property
    def stream(self):
        return _view(_L().orc_df11_stream(self._h), np.uint8, self.stream_bytes)

    @property
    def gaps(self):
        return _view(_L().orc_df11_gaps(self._h), np.uint16, self.n_chunks)

    @property
    def block_pos(self):
        return _view(_L().orc_df11_block_pos(self._h), np.uint64, self.n_blocks + 1)

    @property
    def luts(self):
        return _view(_L().orc_df11_luts(self._h), np.int16, self.n_luts * 256).reshape(self.n_luts, 256)

    def flip_stream_bit(self, bit: int) -> None:
        addr = _L().orc_df11_stream_mut(self._h)
        b = ctypes.c_uint8.from_address(addr + bit // 8)
        b.value ^= 0x80 >> (bit % 8)

    def decode(self) -> np.ndarray:
        out = np.zeros(self.n, dtype=np.uint16)
        if _L().orc_df11_decode(self._h, _p(out) if self.n else 0) != 0:
            raise ValueError("DF11 decode hit an invalid table entry")
        return out


# --------------------------------------------------------------------------- rANS codec
def rans_freqs(counts, prob_bits: int = 12) -> np.ndarray:
    """Normalised frequencies (sum 2^prob_bits) of a 16- or 256-symbol histogram."""
    nsym = 16 if len(counts) <= 16 else 256
    c = np.zeros(nsym, dtype=np.uint64)
    c[: len(counts)] = counts
    out = np.zeros(nsym, dtype=np.uint32)
    if _L().orc_rans_freqs_n(_p(c), nsym, prob_bits, _p(out)) < 0:
        raise ValueError("cannot normalise")
    return out


def rans_table_bits(counts, candidates=(9, 10, 11, 12), table_entry_bits: int = 32) -> int:
    """MINE section 4.2 ("Launch") table-size tuning: candidate sizes 2^b taken in
    increasing order, each scored by the cross-entropy lower bound of the stored size
    (n * H(P, Q_b) payload bits plus 2^b table entries); stop once a score exceeds
    the best so far by more than 1%, and return the best b."""
    best_b, best = None, None
    for b in candidates:
        try:
            f = rans_freqs(counts, b)
        except ValueError:
            continue
        n = float(np.sum(np.asarray(counts, dtype=np.float64)))
        score = n * cross_entropy(counts, f, b) + table_entry_bits * (1 << b)
        if best is not None and score > 1.01 * best:
            break
        if best is None or score < best:
            best_b, best = b, score
    if best_b is None:
        raise ValueError("no table size holds the alphabet")
    return best_b


class Rans:
    """Independent-tile interleaved rANS encoding of 4-bit codes (-8..7)."""

    def __init__(self, codes: np.ndarray, prob_bits: int = 12, tile: int = 4096, k: int = 1):
        """k = codes per symbol: 1, or 2 for pair symbols (a lane's steps 2m, 2m+1;
        the tile and the code count must then be multiples of 64)."""
        c = np.ascontiguousarray(codes, dtype=np.int8).ravel()
        self._c = c
        self.k = k
        self.nsym = 16 if k == 1 else 256
        h = _L().orc_rans_encode_k(_p(c) if c.size else 0, c.size, prob_bits, tile, k)
        if not h:
            raise ValueError("rANS encode failed")
        self._h = h
        self.prob_bits = prob_bits
        info = np.zeros(4, dtype=np.int64)
        _L().orc_rans_info(h, _p(info))
        self.n, self.n_tiles, self.payload_words, self.tile = (int(v) for v in info)

    def __del__(self):
        if getattr(self, "_h", None):
            _L().orc_rans_free(self._h)
            self._h = None

    @property
    def freqs(self):
        return _view(_L().orc_rans_freqs_of(self._h), np.uint32, self.nsym)

    @property
    def counts(self):
        return _view(_L().orc_rans_counts_of(self._h), np.uint64, self.nsym)

    @property
    def states(self):
        return _view(_L().orc_rans_states(self._h), np.uint32, 32 * self.n_tiles).reshape(self.n_tiles, 32)

    @property
    def offsets(self):
        return _view(_L().orc_rans_offsets(self._h), np.uint32, self.n_tiles + 1)

    def flip_payload_bit(self, word: int, bit: int) -> None:
        addr = _L().orc_rans_payload_mut(self._h)
        w = ctypes.c_uint16.from_address(addr + 2 * word)
        w.value ^= 1 << bit

    def decode(self, strict: bool = True):
        out = np.zeros(self.n, dtype=np.int8)
        fin = np.zeros(max(1, 32 * self.n_tiles), dtype=np.uint32)
        rc = _L().orc_rans_decode(self._h, _p(out) if self.n else 0, _p(fin))
        if rc == -1 or (strict and rc != 0):
            raise ValueError(f"rANS decode failed ({rc})")
        return out, fin[: 32 * self.n_tiles].reshape(self.n_tiles, 32), rc


# --------------------------------------------------------------------------- E8 lattice fields
E8_TABLES, E8_ALPHA = 17, 32


def e8_fields(q) -> np.ndarray | None:
    """Fields (c, z_1+16, .., z_7+16, m+16) of a doubled point q[8]; None if q is not in 2 E8."""
    qq = np.ascontiguousarray(q, dtype=np.int8)
    f = np.zeros(9, dtype=np.int32)
    return f if _L().orc_e8_fields(_p(qq), _p(f)) == 0 else None


def e8_point(fields) -> np.ndarray:
    f = np.ascontiguousarray(fields, dtype=np.int32)
    q = np.zeros(8, dtype=np.int8)
    _L().orc_e8_point(_p(f), _p(q))
    return q


class E8:
    """17-table rANS tile coding of doubled E8 points q [n_vec, 8]."""

    def __init__(self, q: np.ndarray, prob_bits: int = 11, tile: int = 512):
        qq = np.ascontiguousarray(q, dtype=np.int8).reshape(-1, 8)
        self.n_vec = qq.shape[0]
        h = _L().orc_e8_encode(_p(qq) if qq.size else 0, self.n_vec, prob_bits, tile)
        if not h:
            raise ValueError("E8 encode failed")
        self._h = h
        self.prob_bits = prob_bits
        info = np.zeros(4, dtype=np.int64)
        _L().orc_e8_info(h, _p(info))
        _, self.n_tiles, self.payload_words, self.tile = (int(v) for v in info)

    def __del__(self):
        if getattr(self, "_h", None):
            _L().orc_e8_free(self._h)
            self._h = None

    @property
    def freqs(self):
        return _view(_L().orc_e8_freqs_of(self._h), np.uint32, E8_TABLES * E8_ALPHA).reshape(E8_TABLES, E8_ALPHA)

    @property
    def counts(self):
        return _view(_L().orc_e8_counts_of(self._h), np.uint64, E8_TABLES * E8_ALPHA).reshape(E8_TABLES, E8_ALPHA)

    @property
    def states(self):
        return _view(_L().orc_e8_states(self._h), np.uint32, 32 * self.n_tiles).reshape(self.n_tiles, 32)

    @property
    def offsets(self):
        return _view(_L().orc_e8_offsets(self._h), np.uint32, self.n_tiles + 1)

    def payload(self) -> np.ndarray:
        return np.ctypeslib.as_array((ctypes.c_uint16 * max(1, self.payload_words)).from_address(
            _L().orc_e8_payload_mut(self._h)))[: self.payload_words].copy()

    def flip_payload_bit(self, word: int, bit: int) -> None:
        w = ctypes.c_uint16.from_address(_L().orc_e8_payload_mut(self._h) + 2 * word)
        w.value ^= 1 << bit

    def decode(self, strict: bool = True):
        out = np.zeros((self.n_vec, 8), dtype=np.int8)
        fin = np.zeros(max(1, 32 * self.n_tiles), dtype=np.uint32)
        rc = _L().orc_e8_decode(self._h, _p(out) if self.n_vec else 0, _p(fin))
        if rc == -1 or (strict and rc != 0):
            raise ValueError(f"E8 decode failed ({rc})")
        return out, fin[: 32 * self.n_tiles].reshape(self.n_tiles, 32), rc


def e8_reconstruct_bf16(q: np.ndarray, scale: float, row_scales: np.ndarray) -> np.ndarray:
    """BF16 weights of doubled points q [N, K]: bf16(fp32(q * fp32(s * r_i)) * 0.5)."""
    qq = np.ascontiguousarray(q, dtype=np.int8)
    r = np.ascontiguousarray(row_scales, dtype=np.float32)
    n, k = qq.shape
    out = np.zeros((n, k), dtype=np.uint16)
    _L().orc_e8_reconstruct_bf16(_p(qq), n, k, ctypes.c_float(scale), _p(r), _p(out))
    return out


E8_DTYPES = {"bf16": (0, np.uint16), "e4m3": (1, np.uint8), "int8": (2, np.int8)}


def e8_reconstruct(q: np.ndarray, scale: float, row_scales: np.ndarray, dtype: str = "bf16") -> np.ndarray:
    """Weights of doubled points q [N, K] in `dtype` ("bf16" bit patterns as uint16,
    "e4m3" codes as uint8, "int8"): dtype(fp32(fp32(q) * fp32(s * r_i)) * 0.5)."""
    code, nptype = E8_DTYPES[dtype]
    qq = np.ascontiguousarray(q, dtype=np.int8)
    r = np.ascontiguousarray(row_scales, dtype=np.float32)
    n, k = qq.shape
    out = np.zeros((n, k), dtype=nptype)
    _L().orc_e8_reconstruct_as(_p(qq), n, k, ctypes.c_float(scale), _p(r), code, _p(out))
    return out


def f32_to_e4m3(values) -> np.ndarray:
    """FP8 E4M3 codes (uint8) of FP32 values: nearest, ties to even, saturating at 448."""
    v = np.asarray(values, dtype=np.float32).ravel()
    return np.array([_L().orc_f32_to_e4m3_satfinite(float(a)) for a in v], dtype=np.uint8)


def f32_to_s8(values) -> np.ndarray:
    """INT8 of FP32 values: nearest integer, ties to even, saturated to [-128, 127]."""
    v = np.asarray(values, dtype=np.float32).ravel()
    return np.array([_L().orc_f32_to_s8_rne_sat(float(a)) for a in v], dtype=np.int8)


def e4m3_to_f32(codes) -> np.ndarray:
    """FP32 values of FP8 E4M3 codes (NaN for S.1111.111)."""
    c = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([_L().orc_e4m3_to_f32(int(v)) for v in c], dtype=np.float32)


def fp8_table(counts, t: int) -> np.ndarray:
    """The top-t table of a 256-bin code histogram: code 0 and the t - 1 most
    frequent other present codes (ties to the lower code), ascending."""
    cnt = np.ascontiguousarray(counts, dtype=np.uint64)
    out = np.zeros(256, dtype=np.uint8)
    n = _L().orc_fp8_table(_p(cnt), t, _p(out))
    return out[:n].copy()


class Fp8:
    """FP8 codes of the padded layout (flattened) under a top-t table: the symbol
    stream through the tile codec plus per-tile correction records."""

    def __init__(self, codes: np.ndarray, t: int = 256, prob_bits: int = 12, tile: int = 4096):
        c = np.ascontiguousarray(codes, dtype=np.uint8).ravel()
        h = _L().orc_fp8_encode(_p(c) if c.size else 0, c.size, t, prob_bits, tile)
        if not h:
            raise ValueError("FP8 encode failed")
        self._h = h
        self.prob_bits = prob_bits
        info = np.zeros(6, dtype=np.int64)
        _L().orc_fp8_info(h, _p(info))
        self.n, self.n_tiles, self.payload_words, self.tile, self.tsize, self.n_records = (int(v) for v in info)

    def __del__(self):
        if getattr(self, "_h", None):
            _L().orc_fp8_free(self._h)
            self._h = None

    @property
    def table(self):
        return _view(_L().orc_fp8_table_of(self._h), np.uint8, self.tsize)

    @property
    def freqs(self):
        return _view(_L().orc_fp8_freqs_of(self._h), np.uint32, self.tsize)

    @property
    def counts(self):
        return _view(_L().orc_fp8_counts_of(self._h), np.uint64, self.tsize)

    @property
    def states(self):
        return _view(_L().orc_fp8_states(self._h), np.uint32, 32 * self.n_tiles).reshape(self.n_tiles, 32)

    @property
    def offsets(self):
        return _view(_L().orc_fp8_offsets(self._h), np.uint32, self.n_tiles + 1)

    @property
    def rec_off(self):
        return _view(_L().orc_fp8_rec_off(self._h), np.uint32, self.n_tiles + 1)

    @property
    def records(self):
        return _view(_L().orc_fp8_records(self._h), np.uint32, max(1, self.n_records))[: self.n_records]

    def payload(self) -> np.ndarray:
        return np.ctypeslib.as_array((ctypes.c_uint16 * max(1, self.payload_words)).from_address(
            _L().orc_fp8_payload_mut(self._h)))[: self.payload_words].copy()

    def flip_payload_bit(self, word: int, bit: int) -> None:
        w = ctypes.c_uint16.from_address(_L().orc_fp8_payload_mut(self._h) + 2 * word)
        w.value ^= 1 << bit

    def decode(self):
        out = np.zeros(max(1, self.n), dtype=np.uint8)
        rc = _L().orc_fp8_decode(self._h, _p(out))
        return out[: self.n], rc


def pad_rows(w: np.ndarray, align: int = 128) -> np.ndarray:
    """BF16 patterns [n_rows, k_cols] with each row padded by zero weights to a
    multiple of `align` columns (the padded layout of the rANS codecs)."""
    n, k = w.shape
    kp = -(-k // align) * align if k else 0
    out = np.zeros((n, kp), dtype=np.uint16)
    out[:, :k] = w
    return out


def expx_bound(w: np.ndarray, k: int, t: int, prob_bits: int = 12, tile: int = 4096) -> float:
    """Size bound in bits of the exponent codec with table size t (-1: the table cannot hold the symbols)."""
    f = np.ascontiguousarray(w, dtype=np.uint16).ravel()
    return float(_L().orc_expx_bound(_p(f) if f.size else None, f.size, k, t, prob_bits, tile))


def expx_choose_t(w: np.ndarray, k: int, t_max: int, prob_bits: int = 12, tile: int = 4096) -> int:
    """The smallest t in 1..t_max whose size bound is least (MINE sec. 4.2 "Tuning t")."""
    f = np.ascontiguousarray(w, dtype=np.uint16).ravel()
    return int(_L().orc_expx_choose_t(_p(f) if f.size else None, f.size, k, t_max, prob_bits, tile))


class Expx:
    """BF16 patterns of the padded layout (flattened): exponents through rANS tiles
    under a top-t table (single values, k = 1, or pairs of a lane's consecutive
    steps, k = 2), escaped exponents as per-tile records, sign and mantissa as one
    plain byte per weight (MINE sec. 4, BF16 handling, "Escapes", "Pair")."""

    def __init__(self, w: np.ndarray, t: int = 256, prob_bits: int = 12, tile: int = 4096, k: int = 1):
        f = np.ascontiguousarray(w, dtype=np.uint16).ravel()
        h = _L().orc_expx_encode(_p(f) if f.size else None, f.size, t, prob_bits, tile, k)
        if not h:
            raise ValueError("exponent codec: encode failed")
        self._h = h
        self.prob_bits = prob_bits
        info = np.zeros(8, dtype=np.int64)
        _L().orc_expx_info(h, _p(info))
        (self.n, self.n_tiles, self.payload_words, self.tile, self.tsize, self.n_records, self.nsym,
         self.k) = (int(v) for v in info)

    def __del__(self):
        if getattr(self, "_h", None):
            _L().orc_expx_free(self._h)
            self._h = None

    @property
    def table(self):
        return _view(_L().orc_expx_table_of(self._h), np.uint8, self.tsize)

    @property
    def freqs(self):
        return _view(_L().orc_expx_freqs_of(self._h), np.uint32, self.nsym)

    @property
    def counts(self):
        return _view(_L().orc_expx_counts_of(self._h), np.uint64, self.nsym)

    @property
    def states(self):
        return _view(_L().orc_expx_states(self._h), np.uint32, 32 * self.n_tiles).reshape(self.n_tiles, 32)

    @property
    def offsets(self):
        return _view(_L().orc_expx_offsets(self._h), np.uint32, self.n_tiles + 1)

    @property
    def rec_off(self):
        return _view(_L().orc_expx_rec_off(self._h), np.uint32, self.n_tiles + 1)

    @property
    def records(self):
        return _view(_L().orc_expx_records(self._h), np.uint32, max(1, self.n_records))[: self.n_records]

    @property
    def sm(self):
        return _view(_L().orc_expx_sm(self._h), np.uint8, max(1, self.n))[: self.n]

    def payload(self) -> np.ndarray:
        return np.ctypeslib.as_array((ctypes.c_uint16 * max(1, self.payload_words)).from_address(
            _L().orc_expx_payload_mut(self._h)))[: self.payload_words].copy()

    def flip_payload_bit(self, word: int, bit: int) -> None:
        w = ctypes.c_uint16.from_address(_L().orc_expx_payload_mut(self._h) + 2 * word)
        w.value ^= 1 << bit

    def decode(self):
        out = np.zeros(max(1, self.n), dtype=np.uint16)
        rc = _L().orc_expx_decode(self._h, _p(out))
        return out[: self.n], rc


def fp8_dequant_bf16(codes: np.ndarray, row_scales: np.ndarray) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    r = np.ascontiguousarray(row_scales, dtype=np.float32)
    n, k = c.shape
    out = np.zeros((n, k), dtype=np.uint16)
    _L().orc_fp8_dequant_bf16(_p(c), _p(r), n, k, _p(out))
    return out


def gemv_fp8(codes: np.ndarray, row_scales: np.ndarray, x: np.ndarray, rows=None):
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    s = np.ascontiguousarray(row_scales, dtype=np.float32)
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.uint16)
    n, k = c.shape
    batch = x.shape[0]
    r, nsel = _rows_arg(rows)
    nr = nsel if r is not None else n
    y = np.zeros((batch, nr), dtype=np.float64)
    a = np.zeros((batch, nr), dtype=np.float64)
    _L().orc_gemv_fp8(_p(c), _p(s), n, k, _p(x), batch, _p(r) if r is not None else None, nsel, _p(y), _p(a))
    return y, a


_VALUES = {"int4": 0, "fp4": 1}


def e2m1_value(code: int) -> float:
    """The FP4 E2M1 value of a 4-bit pattern (OCP Microscaling definition)."""
    return float(_L().orc_e2m1_value(int(code)))


def rans_dequant_bf16(codes: np.ndarray, scales: np.ndarray, group: int = 128, values: str = "int4") -> np.ndarray:
    """BF16 of value(code) * scale: values "int4" (codes in [-8, 7]) or "fp4" (E2M1 patterns 0..15)."""
    c = np.ascontiguousarray(codes, dtype=np.int8)
    s = np.ascontiguousarray(scales, dtype=np.uint16)
    n, k = c.shape
    out = np.zeros((n, k), dtype=np.uint16)
    _L().orc_rans_dequant_bf16_v(_p(c), _p(s), n, k, group, _VALUES[values], _p(out))
    return out


# --------------------------------------------------------------------------- GEMV
def _rows_arg(rows):
    if rows is None:
        return None, 0
    r = np.ascontiguousarray(rows, dtype=np.int64)
    return r, r.size


def gemv_bf16(w: np.ndarray, x: np.ndarray, rows=None):
    """FP64 y[b, i] and a[b, i] = sum |w x| for BF16 W [N, K] and x [batch, K]."""
    w = np.ascontiguousarray(w, dtype=np.uint16)
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.uint16)
    n, k = w.shape
    batch = x.shape[0]
    r, nsel = _rows_arg(rows)
    nr = nsel if r is not None else n
    y = np.zeros((batch, nr), dtype=np.float64)
    a = np.zeros((batch, nr), dtype=np.float64)
    _L().orc_gemv_bf16(_p(w), n, k, _p(x), batch, _p(r) if r is not None else None, nsel, _p(y), _p(a))
    return y, a


def gemv_rans(codes: np.ndarray, scales: np.ndarray, x: np.ndarray, group: int = 128, rows=None,
              values: str = "int4"):
    c = np.ascontiguousarray(codes, dtype=np.int8)
    s = np.ascontiguousarray(scales, dtype=np.uint16)
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.uint16)
    n, k = c.shape
    batch = x.shape[0]
    r, nsel = _rows_arg(rows)
    nr = nsel if r is not None else n
    y = np.zeros((batch, nr), dtype=np.float64)
    a = np.zeros((batch, nr), dtype=np.float64)
    _L().orc_gemv_rans_v(_p(c), _p(s), n, k, group, _VALUES[values], _p(x), batch, _p(r) if r is not None else None,
                         nsel, _p(y), _p(a))
    return y, a
