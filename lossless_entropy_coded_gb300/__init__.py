"""Entropy-coded LLM weights on GB300: lossless Huffman-exponent BF16 and rANS
4-bit codecs with fused decode + GEMV kernels for sm_103a.

The work happens in libec.so (include/ec.h); this package only marshals arguments.
The library is loaded on first use of any attribute below; if libec.so has not been
built the access raises ImportError (there is no fallback path).
"""
_API = ("EC_KIND_E8", "EC_KIND_HUFFMAN_BF16", "EC_KIND_RANS_FP8", "EC_KIND_RANS_EXP", "EC_KIND_RANS_INT4", "EC_MAX_BATCH", "EC_MAX_GROUP", "EcError", "Matrix",
        "bf16_gemm", "bf16_gemv", "decode", "decode_as", "decode_batch", "deserialize", "encode_bf16", "encode_bf16_exp", "encode_e8", "encode_fp8", "encode_rans", "gemm", "gemm_group", "gemm_group_work_bytes", "gemm_work_bytes", "gemv", "gemv_group", "gemv_path", "gemv_static", "lib",
        "status", "strerror", "LIB_PATH", "EXPORTS")

__all__ = list(_API)


def __getattr__(name):
    if name in _API:
        from . import _ec
        return getattr(_ec, name)
    raise AttributeError(name)
