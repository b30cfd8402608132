"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the benchmark.

Only random-number drawing and storage-type rounding live here (FP32 -> BF16
round-to-nearest-even, integer codes, FP64 -> FP16 scales).  None of the
entropy-coding or GEMV arithmetic does: both sides get these arrays as inputs.

Workload recipes (shapes and distributions of the Llama-3.1-8B / 70B linear
layers and the 4-bit rANS case) are in ``WORKLOADS`` and the ``make_*``
functions below.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lib = None

NTHREADS = max(1, min(64, os.cpu_count() or 1))


def build(force: bool = False) -> str:
    """Compile libsynth.so next to its source (plain gcc, no CUDA)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-Wall", "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def _L():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        u64, i64, i32, f64, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        lib.synth_sm64.argtypes = [u64, u64]
        lib.synth_sm64.restype = u64
        lib.synth_subseed.argtypes = [u64, u64]
        lib.synth_subseed.restype = u64
        lib.synth_normal_f64.argtypes = [u64, u64, i64, vp, i32]
        lib.synth_uniform_f64.argtypes = [u64, u64, i64, vp, i32]
        lib.synth_gauss_bf16.argtypes = [u64, i64, f64, vp, i32]
        lib.synth_llama_bf16.argtypes = [u64, i64, i64, f64, f64, f64, f64, vp, vp, i32]
        lib.synth_llama_bf16.restype = i64
        lib.synth_codes_i8.argtypes = [u64, i64, f64, i32, i32, vp, i32]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def sm64(seed: int, n: int) -> int:
    """Output number n of the SplitMix64 stream seeded with `seed`."""
    return int(_L().synth_sm64(seed & (2**64 - 1), n))


def normal_f64(seed: int, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _L().synth_normal_f64(seed, offset, n, _ptr(out), NTHREADS)
    return out


def uniform_f64(seed: int, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _L().synth_uniform_f64(seed, offset, n, _ptr(out), NTHREADS)
    return out


def gauss_bf16(seed: int, shape, std: float) -> np.ndarray:
    """bf16(float(std * z)) as uint16 bit patterns."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.uint16)
    _L().synth_gauss_bf16(seed, n, float(std), _ptr(out), NTHREADS)
    return out.reshape(shape)


def llama_bf16(seed: int, n_rows: int, k_cols: int, base_std: float = 0.02, ln_sigma: float = 0.5,
               outlier_frac: float = 0.001, outlier_std: float = 0.5, return_positions: bool = False):
    """Row-scaled Gaussian weights with a fixed count of outliers, as BF16 bit patterns.

    s_i = base_std * exp(ln_sigma * z_i) (a LogNormal(0, ln_sigma) factor), w_ij ~ N(0, s_i^2),
    then round(outlier_frac * N * K) distinct positions get N(0, outlier_std^2).
    """
    out = np.empty((n_rows, k_cols), dtype=np.uint16)
    m = int(round(outlier_frac * n_rows * k_cols))
    pos = np.empty(max(m, 1), dtype=np.int64)
    got = _L().synth_llama_bf16(seed, n_rows, k_cols, base_std, ln_sigma, outlier_frac, outlier_std,
                                _ptr(out), _ptr(pos), NTHREADS)
    if got < 0:
        raise MemoryError("synth_llama_bf16 failed")
    return (out, pos[:got]) if return_positions else out


def codes_i8(seed: int, shape, std: float = 1.1, lo: int = -8, hi: int = 7) -> np.ndarray:
    """clip(round_half_even(std * z), lo, hi) as int8."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.int8)
    _L().synth_codes_i8(seed, n, float(std), lo, hi, _ptr(out), NTHREADS)
    return out.reshape(shape)


def scales_f16(seed: int, shape, lo: float = 0.005, hi: float = 0.03) -> np.ndarray:
    """FP16 (round-to-nearest-even from FP64) draws of U(lo, hi), as uint16 bit patterns."""
    n = int(np.prod(shape))
    u = uniform_f64(seed, n)
    return (lo + (hi - lo) * u).astype(np.float16).view(np.uint16).reshape(shape)


def bf16_to_f32(a: np.ndarray) -> np.ndarray:
    return (a.astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# Workloads: Llama-3.1-8B decoder-layer linears (q, k, v, o, gate, up, down),
# Llama-3.3-70B-shaped block, 1024x1024 single matrix, 4-bit rANS shapes.
# ---------------------------------------------------------------------------
LAYER_8B = [("q", 4096, 4096), ("k", 1024, 4096), ("v", 1024, 4096), ("o", 4096, 4096),
            ("gate", 14336, 4096), ("up", 14336, 4096), ("down", 4096, 14336)]
BLOCK_70B = [("q", 8192, 8192), ("k", 1024, 8192), ("v", 1024, 8192), ("o", 8192, 8192),
             ("gate", 28672, 8192), ("up", 28672, 8192), ("down", 8192, 28672)]
RANS_SHAPES = [(14336, 4096), (4096, 14336)]
N_LAYERS_8B = 32


@dataclass(frozen=True)
class MatrixSpec:
    name: str
    n_rows: int
    k_cols: int
    seed: int
    kind: str  # "gauss" | "llama"


def single_1024() -> MatrixSpec:
    return MatrixSpec("w1024", 1024, 1024, 1001, "gauss")


def layer_8b(layer: int | None = None) -> list[MatrixSpec]:
    """One 8B layer set; layer=None is the stand-alone set (seeds 2000+i), else layer l of the stack."""
    out = []
    for i, (nm, n, k) in enumerate(LAYER_8B):
        seed = 2000 + i if layer is None else 3000 + 16 * layer + i
        out.append(MatrixSpec(nm if layer is None else f"L{layer}.{nm}", n, k, seed, "llama"))
    return out


def block_70b() -> list[MatrixSpec]:
    return [MatrixSpec(nm, n, k, 5000 + i, "llama") for i, (nm, n, k) in enumerate(BLOCK_70B)]


def make_weights(spec: MatrixSpec) -> np.ndarray:
    if spec.kind == "gauss":
        return gauss_bf16(spec.seed, (spec.n_rows, spec.k_cols), 0.02)
    return llama_bf16(spec.seed, spec.n_rows, spec.k_cols)


def make_x(seed: int, batch: int, k_cols: int) -> np.ndarray:
    """Activations x ~ N(0, 1) as BF16 bit patterns, stream seed + 7."""
    return gauss_bf16(seed + 7, (batch, k_cols), 1.0)


def make_rans_case(shape_index: int, n_rows: int | None = None, k_cols: int | None = None, group: int = 128):
    """4-bit codes ~ clip(rne(N(0, 1.1^2)), -8, 7) and FP16 scales ~ U(0.005, 0.03) per `group` weights."""
    n, k = RANS_SHAPES[shape_index] if n_rows is None else (n_rows, k_cols)
    seed = 4000 + shape_index
    codes = codes_i8(seed, (n, k))
    scales = scales_f16(synth_subseed(seed, 9), (n, (k + group - 1) // group))
    return codes, scales


def fp4_codes(seed: int, shape, std: float = 1.6) -> np.ndarray:
    """4-bit patterns (sign << 3 | k) with k = min(|round_half_even(std * z)|, 7) and the
    sign of z: a skewed histogram over the 16 patterns, most mass on small k (the
    patterns are taken as FP4 E2M1 codes by the codec under test)."""
    c = codes_i8(seed, shape, std=std, lo=-7, hi=7).astype(np.int16)
    return (((c < 0).astype(np.int16) << 3) | np.abs(c)).astype(np.int8)


def make_fp4_case(seed: int, n_rows: int, k_cols: int, group: int = 128):
    """(codes, FP16 scales ~ U(0.005, 0.03) per `group` weights) of an FP4 matrix."""
    return fp4_codes(seed, (n_rows, k_cols)), scales_f16(synth_subseed(seed, 9), (n_rows, (k_cols + group - 1) // group))


def synth_subseed(seed: int, tag: int) -> int:
    return int(_L().synth_subseed(seed, tag))


def e8_points(seed: int, n_rows: int, k_cols: int, std: float = 3.5) -> np.ndarray:
    """Doubled E8 points q = 2 z + c, int8 [n_rows, k_cols] (k_cols % 8 == 0).

    Per run of 8 columns: coset c ~ Bernoulli(1/2); z_j = clip(rne(std * g_j), -15, 14)
    with g ~ N(0, 1); if z_1 + ... + z_8 is odd, coordinate u (uniform in 0..7) moves
    by one toward zero (away from zero if it is 0), which puts z in D8.  std = 3.5 gives
    about 4 bits of entropy per weight."""
    assert k_cols % 8 == 0
    nv = n_rows * (k_cols // 8)
    z = np.clip(np.rint(std * normal_f64(seed, 8 * nv)), -15, 14).astype(np.int16).reshape(nv, 8)
    u = uniform_f64(synth_subseed(seed, 1), 2 * nv).reshape(nv, 2)
    c = (u[:, 0] < 0.5).astype(np.int16)
    odd = np.nonzero(z.sum(axis=1) & 1)[0]
    j = np.minimum((u[odd, 1] * 8).astype(np.int64), 7)
    v = z[odd, j]
    z[odd, j] = np.where(v > 0, v - 1, v + 1)
    return (2 * z + c[:, None]).astype(np.int8).reshape(n_rows, k_cols)


def e8_row_scales(seed: int, n_rows: int, base: float = 0.02, ln_sigma: float = 0.5) -> np.ndarray:
    """FP32 row scales r_i = base * exp(ln_sigma * g_i), g ~ N(0, 1)."""
    return (base * np.exp(ln_sigma * normal_f64(seed, n_rows))).astype(np.float32)


def make_e8_case(seed: int, n_rows: int, k_cols: int, std: float = 3.5, scale: float = 0.125):
    """(q2, row_scales, scale) of an E8 matrix: w = bf16(q2 / 2 * scale * r_i)."""
    return e8_points(seed, n_rows, k_cols, std), e8_row_scales(synth_subseed(seed, 2), n_rows), scale


def fp8_codes(seed: int, n_rows: int, k_cols: int, spread: float = 100.0) -> np.ndarray:
    """FP8 E4M3 bytes [n_rows, k_cols] with the skewed histogram of Gaussian weights
    scaled to the format's range: m = spread * |g|, sign ~ Bernoulli(1/2); the
    exponent field is floor(log2 m) + 7 clipped to 1..15 (field 0 and mantissa
    floor(m / 2^-9) below 2^-6), the mantissa floor(8 (m / 2^e - 1)), and the NaN
    pattern S.1111.111 is avoided (mantissa 6 there)."""
    n = n_rows * k_cols
    m = spread * np.abs(normal_f64(seed, n))
    sign = (uniform_f64(synth_subseed(seed, 3), n) < 0.5).astype(np.uint8)
    with np.errstate(divide="ignore"):
        e = np.clip(np.floor(np.log2(np.maximum(m, 1e-300))), -6, 8)
    mant = np.clip(np.floor(8 * (m / 2.0 ** e - 1)), 0, 7)
    field = (e + 7).astype(np.int64)
    sub = m < 2.0 ** -6
    field[sub] = 0
    mant[sub] = np.clip(np.floor(m[sub] / 2.0 ** -9), 0, 7)
    mant = mant.astype(np.int64)
    mant[(field == 15) & (mant == 7)] = 6
    return ((sign.astype(np.int64) << 7) | (field << 3) | mant).astype(np.uint8).reshape(n_rows, k_cols)


def make_fp8_case(seed: int, n_rows: int, k_cols: int):
    """(codes, row_scales) of an FP8 matrix: weight = value(code) * r_i, r_i ~ 0.02 LogNormal(0, 0.5) / 448."""
    return fp8_codes(seed, n_rows, k_cols), e8_row_scales(synth_subseed(seed, 4), n_rows, base=0.02 / 448)
