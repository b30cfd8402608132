"""ctypes binding of include/ec.h (argument marshalling only).

Every operation runs in libec.so.  Device buffers are torch CUDA tensors (their
data_ptr()), host inputs are numpy arrays or CPU tensors.  If libec.so is missing
the import fails loudly: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libec.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -m lossless_entropy_coded_gb300.build` "
        "(or __graft_entry__.build()); the library has no fallback path")

lib = ctypes.CDLL(LIB_PATH)

EC_OK = 0
EC_ERR_INVALID_ARG = -1
EC_ERR_SHAPE = -2
EC_ERR_OVERFLOW = -3
EC_ERR_UNSUPPORTED = -4
EC_ERR_CORRUPT = -5
EC_ERR_CUDA = -6
EC_ERR_OOM = -7
EC_MAX_BATCH = 64
EC_MAX_GROUP = 8
EC_KIND_HUFFMAN_BF16 = 1
EC_KIND_RANS_INT4 = 2
EC_KIND_E8 = 3
EC_KIND_RANS_FP8 = 4
EC_KIND_RANS_EXP = 5

EXPORTS = ["ec_encode_bf16", "ec_encode_rans", "ec_decode", "ec_decode_batch", "ec_gemv", "ec_gemv_group",
           "ec_bf16_gemv", "ec_stats", "ec_code_lengths", "ec_serialize", "ec_deserialize", "ec_status", "ec_free",
           "ec_strerror", "ec_gemv_static", "ec_gemv_path", "ec_encode_e8", "ec_decode_as", "ec_encode_fp8",
           "ec_gemm", "ec_gemm_work_bytes", "ec_bf16_gemm", "ec_encode_bf16_exp", "ec_gemm_group",
           "ec_gemm_group_work_bytes"]


class HuffParams(ctypes.Structure):
    _fields_ = [("max_code_len", ctypes.c_int32), ("tile_steps", ctypes.c_int32), ("hierarchical", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class RansParams(ctypes.Structure):
    _fields_ = [("prob_bits", ctypes.c_int32), ("tile_syms", ctypes.c_int32), ("group", ctypes.c_int32),
                ("codes_per_symbol", ctypes.c_int32), ("values", ctypes.c_int32)]


_RANS_VALUES = {"int4": 0, "fp4": 1}  # EC_RANS_VALUES_INT4, EC_RANS_VALUES_FP4_E2M1


class E8Params(ctypes.Structure):
    _fields_ = [("prob_bits", ctypes.c_int32), ("tile_vectors", ctypes.c_int32), ("reserved", ctypes.c_int32 * 2)]


class Fp8Params(ctypes.Structure):
    _fields_ = [("prob_bits", ctypes.c_int32), ("tile_syms", ctypes.c_int32), ("top_t", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class ExpParams(ctypes.Structure):
    _fields_ = [("prob_bits", ctypes.c_int32), ("tile_syms", ctypes.c_int32), ("top_t", ctypes.c_int32),
                ("single", ctypes.c_int32)]


class Stats(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("max_code_len", ctypes.c_int32), ("n_rows", ctypes.c_int64),
                ("k_cols", ctypes.c_int64), ("k_pad", ctypes.c_int64), ("n_tiles", ctypes.c_int64),
                ("payload_bits", ctypes.c_int64), ("raw_bytes", ctypes.c_int64), ("aux_bytes", ctypes.c_int64),
                ("table_bytes", ctypes.c_int64), ("device_bytes", ctypes.c_int64),
                ("bits_per_weight", ctypes.c_double), ("entropy_bits", ctypes.c_double),
                ("coded_bits_per_symbol", ctypes.c_double), ("n_records", ctypes.c_int64)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


_vp, _i64, _i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
_sig = {
    "ec_encode_bf16": ([_vp, _i64, _i64, ctypes.POINTER(HuffParams), _i32, ctypes.POINTER(_vp)], _i32),
    "ec_encode_rans": ([_vp, _vp, _i64, _i64, ctypes.POINTER(RansParams), _i32, ctypes.POINTER(_vp)], _i32),
    "ec_encode_e8": ([_vp, _vp, ctypes.c_float, _i64, _i64, ctypes.POINTER(E8Params), _i32, ctypes.POINTER(_vp)],
                     _i32),
    "ec_encode_fp8": ([_vp, _vp, _i64, _i64, ctypes.POINTER(Fp8Params), _i32, ctypes.POINTER(_vp)], _i32),
    "ec_encode_bf16_exp": ([_vp, _i64, _i64, ctypes.POINTER(ExpParams), _i32, ctypes.POINTER(_vp)], _i32),
    "ec_decode": ([_vp, _vp, _vp], _i32),
    "ec_decode_batch": ([_vp, _vp, _i32, _vp], _i32),
    "ec_decode_as": ([_vp, _vp, _i32, _vp], _i32),
    "ec_gemv": ([_vp, _vp, _vp, _i32, _vp], _i32),
    "ec_gemv_group": ([_vp, _i32, _vp, _vp, _i32, _vp], _i32),
    "ec_bf16_gemv": ([_vp, _i64, _i64, _vp, _vp, _i32, _vp], _i32),
    "ec_gemm": ([_vp, _vp, _vp, _i32, _vp, ctypes.c_size_t, _vp], _i32),
    "ec_gemm_work_bytes": ([_vp, _i32, ctypes.POINTER(ctypes.c_size_t)], _i32),
    "ec_gemm_group": ([_vp, _i32, _vp, _vp, _i32, _vp, ctypes.c_size_t, _vp], _i32),
    "ec_gemm_group_work_bytes": ([_vp, _i32, _i32, ctypes.POINTER(ctypes.c_size_t)], _i32),
    "ec_bf16_gemm": ([_vp, _i64, _i64, _vp, _vp, _i32, _vp, ctypes.c_size_t, _vp], _i32),
    "ec_gemv_static": ([_vp, _vp, _vp, _i32, _vp], _i32),
    "ec_gemv_path": ([_vp, _i32, _i32], _i32),
    "ec_stats": ([_vp, ctypes.POINTER(Stats)], _i32),
    "ec_code_lengths": ([_vp, _vp], _i32),
    "ec_serialize": ([_vp, _vp, _i64, ctypes.POINTER(_i64)], _i32),
    "ec_deserialize": ([_vp, _i64, _i32, ctypes.POINTER(_vp)], _i32),
    "ec_status": ([_vp], _i32),
    "ec_free": ([_vp], None),
    "ec_strerror": ([_i32], ctypes.c_char_p),
}
for _n, (_a, _r) in _sig.items():
    _f = getattr(lib, _n)
    _f.argtypes = _a
    _f.restype = _r


class EcError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {lib.ec_strerror(code).decode()} ({code})")


def _check(rc: int, what: str) -> None:
    if rc != EC_OK:
        raise EcError(rc, what)


def strerror(code: int) -> str:
    return lib.ec_strerror(code).decode()


def _host_ptr(a):
    """(pointer, keepalive) for a C-contiguous host array (numpy or CPU tensor)."""
    if hasattr(a, "data_ptr"):
        assert not a.is_cuda and a.is_contiguous()
        return a.data_ptr(), a
    a = np.ascontiguousarray(a)
    return a.ctypes.data, a


def _stream_ptr(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    return int(stream)


def _dev_ptr(t):
    return 0 if t is None else t.data_ptr()


class Matrix:
    """An encoded matrix resident on one GPU (owns its device blob)."""

    def __init__(self, handle: int, n_rows: int, k_cols: int, kind: int, device: int):
        self.handle = ctypes.c_void_p(handle)
        self.n_rows, self.k_cols, self.kind, self.device = n_rows, k_cols, kind, device

    @property
    def shape(self):
        return (self.n_rows, self.k_cols)

    def stats(self) -> dict:
        s = Stats()
        _check(lib.ec_stats(self.handle, ctypes.byref(s)), "ec_stats")
        return s.as_dict()

    def code_lengths(self) -> np.ndarray:
        out = np.zeros(256, np.uint8)
        _check(lib.ec_code_lengths(self.handle, out.ctypes.data), "ec_code_lengths")
        return out

    def serialize(self) -> bytes:
        """Metadata block + device blob (copied back to the host)."""
        n = ctypes.c_int64()
        _check(lib.ec_serialize(self.handle, None, 0, ctypes.byref(n)), "ec_serialize")
        buf = (ctypes.c_uint8 * n.value)()
        _check(lib.ec_serialize(self.handle, buf, n.value, ctypes.byref(n)), "ec_serialize")
        return bytes(buf)

    def free(self) -> None:
        if self.handle:
            lib.ec_free(self.handle)
            self.handle = ctypes.c_void_p(0)

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def encode_bf16(w, max_code_len: int = 12, tile_steps: int = 0, device: int = 0, hierarchical: bool = False) -> Matrix:
    """Huffman-exponent encode a host BF16 matrix [N, K] (uint16 bit patterns);
    hierarchical=True decodes overflowing pairs through DFloat11's hierarchical tables
    instead of window records."""
    n, k = int(w.shape[0]), int(w.shape[1])
    p, keep = _host_ptr(w)
    prm = HuffParams(max_code_len, tile_steps, 1 if hierarchical else 0)
    h = ctypes.c_void_p()
    _check(lib.ec_encode_bf16(p, n, k, ctypes.byref(prm), device, ctypes.byref(h)), "ec_encode_bf16")
    del keep
    return Matrix(h.value, n, k, EC_KIND_HUFFMAN_BF16, device)


def encode_rans(codes, scales_f16, prob_bits: int = 12, tile_syms: int = 4096, group: int = 128,
                device: int = 0, codes_per_symbol: int = 1, values: str = "int4") -> Matrix:
    """rANS-encode host int8 codes [N, K] with FP16 scales [N, ceil(K/group)]: values
    "int4" takes signed codes in [-8, 7], "fp4" FP4 E2M1 patterns in [0, 15]
    (codes_per_symbol 2: one symbol per pair of a lane's consecutive codes)."""
    n, k = int(codes.shape[0]), int(codes.shape[1])
    pc, kc = _host_ptr(codes)
    ps, ks = _host_ptr(scales_f16)
    prm = RansParams(prob_bits, tile_syms, group, codes_per_symbol, _RANS_VALUES[values])
    h = ctypes.c_void_p()
    _check(lib.ec_encode_rans(pc, ps, n, k, ctypes.byref(prm), device, ctypes.byref(h)), "ec_encode_rans")
    return Matrix(h.value, n, k, EC_KIND_RANS_INT4, device)


def encode_e8(q2, row_scales, scale: float, prob_bits: int = 0, tile_vectors: int = 0,
              device: int = 0) -> Matrix:
    """Encode host int8 doubled E8 points q2 [N, K] (each run of 8 columns is 2 p with
    p in E8) with FP32 row scales [N] and the global scale s; decode gives
    bf16(q2 / 2 * s * r_i).  0 selects the defaults (2^11 slots, 1024 vectors a tile)."""
    n, k = int(q2.shape[0]), int(q2.shape[1])
    pq, kq = _host_ptr(q2)
    pr, kr = _host_ptr(row_scales)
    prm = E8Params(prob_bits, tile_vectors)
    h = ctypes.c_void_p()
    _check(lib.ec_encode_e8(pq, pr, float(scale), n, k, ctypes.byref(prm), device, ctypes.byref(h)), "ec_encode_e8")
    return Matrix(h.value, n, k, EC_KIND_E8, device)


def encode_fp8(codes, row_scales, top_t: int = 0, prob_bits: int = 0, tile_syms: int = 0,
               device: int = 0) -> Matrix:
    """Encode host FP8 E4M3 bytes [N, K] with FP32 row scales [N] under a top-t table
    (top_t 0: every code present; 0 for prob_bits / tile_syms: 12 and 4096)."""
    n, k = int(codes.shape[0]), int(codes.shape[1])
    pc, kc = _host_ptr(codes)
    pr, kr = _host_ptr(row_scales)
    prm = Fp8Params(prob_bits, tile_syms, top_t)
    h = ctypes.c_void_p()
    _check(lib.ec_encode_fp8(pc, pr, n, k, ctypes.byref(prm), device, ctypes.byref(h)), "ec_encode_fp8")
    return Matrix(h.value, n, k, EC_KIND_RANS_FP8, device)


def encode_bf16_exp(w, prob_bits: int = 0, tile_syms: int = 0, top_t: int = 0, single: bool = False,
                    device: int = 0) -> Matrix:
    """Encode a host BF16 matrix [N, K] (uint16 bit patterns) with its exponents as rANS
    symbols under a top-t table (pairs of a lane's consecutive exponents unless single),
    escaped exponents as records, sign and mantissa as plain bytes.  0 selects the
    defaults (2^12 slots, 4096-weight tiles, t chosen by the size bound)."""
    n, k = int(w.shape[0]), int(w.shape[1])
    p, keep = _host_ptr(w)
    prm = ExpParams(prob_bits, tile_syms, top_t, 1 if single else 0)
    h = ctypes.c_void_p()
    _check(lib.ec_encode_bf16_exp(p, n, k, ctypes.byref(prm), device, ctypes.byref(h)), "ec_encode_bf16_exp")
    del keep
    return Matrix(h.value, n, k, EC_KIND_RANS_EXP, device)


def deserialize(data: bytes, device: int = 0) -> Matrix:
    """Validate and load ec_serialize output (device < 0: host-only matrix)."""
    buf = (ctypes.c_uint8 * len(data)).from_buffer_copy(data)
    h = ctypes.c_void_p()
    _check(lib.ec_deserialize(buf, len(data), device, ctypes.byref(h)), "ec_deserialize")
    m = Matrix(h.value, 0, 0, 0, device)
    s = m.stats()
    m.n_rows, m.k_cols, m.kind = s["n_rows"], s["k_cols"], s["kind"]
    return m


def decode(W: Matrix, out, stream=None) -> None:
    _check(lib.ec_decode(W.handle, _dev_ptr(out), _stream_ptr(stream)), "ec_decode")


EC_DTYPE_BF16, EC_DTYPE_FP8_E4M3, EC_DTYPE_INT8 = 0, 1, 2
_DTYPES = {"bf16": EC_DTYPE_BF16, "e4m3": EC_DTYPE_FP8_E4M3, "int8": EC_DTYPE_INT8}


def decode_as(W: Matrix, out, dtype: str = "bf16", stream=None) -> None:
    """ec_decode_as: decode into `out` as "bf16" (2 bytes), "e4m3" or "int8" (1 byte)."""
    _check(lib.ec_decode_as(W.handle, _dev_ptr(out), _DTYPES[dtype], _stream_ptr(stream)), "ec_decode_as")


def decode_batch(Ws, outs, stream=None) -> None:
    n = len(Ws)
    hs = (ctypes.c_void_p * n)(*[W.handle.value for W in Ws])
    os_ = (ctypes.c_void_p * n)(*[_dev_ptr(o) for o in outs])
    _check(lib.ec_decode_batch(hs, os_, n, _stream_ptr(stream)), "ec_decode_batch")


def gemv(W: Matrix, x, y, batch: int = 1, stream=None) -> None:
    _check(lib.ec_gemv(W.handle, _dev_ptr(x), _dev_ptr(y), batch, _stream_ptr(stream)), "ec_gemv")


def gemv_static(W: Matrix, x, y, batch: int = 1, stream=None) -> None:
    """ec_gemv_static: the GEMV with no device or host allocation (fixed built-in
    scratch; serialise calls that could overlap on the GPU)."""
    _check(lib.ec_gemv_static(W.handle, _dev_ptr(x), _dev_ptr(y), batch, _stream_ptr(stream)), "ec_gemv_static")


EC_PATH_CUDA_CORES, EC_PATH_TENSOR_CORES = 1, 2


def gemv_path(Ws, batch: int = 1) -> str:
    """Which kernels gemv_group(Ws, ..., batch) uses: "cuda_cores" or "tensor_cores"."""
    if not isinstance(Ws, (list, tuple)):
        Ws = [Ws]
    hs = (ctypes.c_void_p * len(Ws))(*[W.handle.value for W in Ws])
    rc = lib.ec_gemv_path(hs, len(Ws), batch)
    _check(rc if rc < 0 else 0, "ec_gemv_path")
    return "tensor_cores" if rc == EC_PATH_TENSOR_CORES else "cuda_cores"


def gemv_group(Ws, x, ys, batch: int = 1, stream=None) -> None:
    n = len(Ws)
    hs = (ctypes.c_void_p * n)(*[W.handle.value for W in Ws])
    yp = (ctypes.c_void_p * n)(*[_dev_ptr(y) for y in ys])
    _check(lib.ec_gemv_group(hs, n, _dev_ptr(x), yp, batch, _stream_ptr(stream)), "ec_gemv_group")


def bf16_gemv(w, x, y, batch: int = 1, stream=None) -> None:
    n, k = int(w.shape[0]), int(w.shape[1])
    _check(lib.ec_bf16_gemv(_dev_ptr(w), n, k, _dev_ptr(x), _dev_ptr(y), batch, _stream_ptr(stream)),
           "ec_bf16_gemv")


def gemm_work_bytes(W: Matrix, batch: int) -> int:
    """ec_gemm_work_bytes: the work buffer ec_gemm uses with full-size chunks."""
    n = ctypes.c_size_t(0)
    _check(lib.ec_gemm_work_bytes(W.handle, batch, ctypes.byref(n)), "ec_gemm_work_bytes")
    return int(n.value)


def gemm(W: Matrix, x, y, batch: int, work=None, stream=None) -> None:
    """ec_gemm: y = x W^T for any batch (chunked decode + tensor-core GEMM).  work: a
    device tensor (its bytes are the buffer); None allocates one of gemm_work_bytes."""
    if work is None:
        import torch
        work = torch.empty(gemm_work_bytes(W, batch), dtype=torch.uint8, device=x.device)
    nbytes = work.numel() * work.element_size()
    _check(lib.ec_gemm(W.handle, _dev_ptr(x), _dev_ptr(y), batch, _dev_ptr(work), nbytes, _stream_ptr(stream)),
           "ec_gemm")


def gemm_group_work_bytes(Ws, batch: int) -> int:
    """ec_gemm_group_work_bytes: the work buffer that decodes every packable matrix in one launch."""
    hs = (ctypes.c_void_p * len(Ws))(*[W.handle.value for W in Ws])
    n = ctypes.c_size_t(0)
    _check(lib.ec_gemm_group_work_bytes(hs, len(Ws), batch, ctypes.byref(n)), "ec_gemm_group_work_bytes")
    return int(n.value)


def gemm_group(Ws, xs, ys, batch: int, work=None, stream=None) -> None:
    """ec_gemm_group: ys[m] = xs[m] W_m^T for several matrices, decoded together where
    the work buffer allows (None allocates gemm_group_work_bytes)."""
    n = len(Ws)
    if work is None:
        import torch
        work = torch.empty(gemm_group_work_bytes(Ws, batch), dtype=torch.uint8, device=ys[0].device)
    hs = (ctypes.c_void_p * n)(*[W.handle.value for W in Ws])
    xp = (ctypes.c_void_p * n)(*[_dev_ptr(x) for x in xs])
    yp = (ctypes.c_void_p * n)(*[_dev_ptr(y) for y in ys])
    nbytes = work.numel() * work.element_size()
    _check(lib.ec_gemm_group(hs, n, xp, yp, batch, _dev_ptr(work), nbytes, _stream_ptr(stream)), "ec_gemm_group")


def bf16_gemm(w, x, y, batch: int, work=None, stream=None) -> None:
    """ec_bf16_gemm: the same tensor-core GEMM on a dense BF16 matrix (work: partial sums, optional)."""
    n, k = int(w.shape[0]), int(w.shape[1])
    nbytes = 0 if work is None else work.numel() * work.element_size()
    _check(lib.ec_bf16_gemm(_dev_ptr(w), n, k, _dev_ptr(x), _dev_ptr(y), batch, _dev_ptr(work), nbytes,
                            _stream_ptr(stream)), "ec_bf16_gemm")


def status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    return int(lib.ec_status(_stream_ptr(stream)))
