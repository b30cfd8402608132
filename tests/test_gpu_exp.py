"""GPU parity of the BF16-exponent rANS codec (kind 5): decode bit-exact with the
original BF16 patterns (the codec is lossless; the oracle's decode of the same
stream gives the same patterns, tests/test_oracle_expx.py), and the fused GEMV
against the oracle's FP64 GEMV at the stated tolerance (relative L2 <= 1e-3,
|err| <= 2e-3 * sum|w x|), with and without escape records.

Source: MINE section 4 (BF16 handling, "Escapes", "Pair") and section 4.2."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from parity import check_gemv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ec():
    import lossless_entropy_coded_gb300 as ec
    return ec


def decode(ec, W):
    out = torch.zeros((W.n_rows, W.k_cols), dtype=torch.int16, device="cuda")
    ec.decode(W, out)
    assert ec.status() == 0
    return out.cpu().numpy().view(np.uint16)


# (shape, top_t (0: automatic), single, tile)
DEC = [((7, 300), 0, False, 4096), ((64, 1000), 3, False, 1024), ((300, 4096), 0, True, 4096),
       ((300, 4096), 5, True, 2048), ((96, 14336), 0, False, 4096), ((33, 2048), 1, False, 128)]


@pytest.mark.parametrize("shape,t,single,tile", DEC)
def test_decode_bit_exact(ec, shape, t, single, tile):
    w = synth.llama_bf16(8600 + shape[1] + t, *shape)
    W = ec.encode_bf16_exp(w, top_t=t, single=single, tile_syms=tile)
    assert np.array_equal(decode(ec, W), w)
    if t and t < 8:
        assert W.stats()["n_records"] > 0


@pytest.mark.parametrize("single", [False, True])
def test_all_patterns_decode(ec, single):
    w = np.arange(65536, dtype=np.uint16)[np.random.default_rng(3).permutation(65536)].reshape(256, 256)
    W = ec.encode_bf16_exp(w, single=single)  # many exponents outside a 16-entry pair table
    assert np.array_equal(decode(ec, W), w)


GEMV = [((7, 300), 0, False), ((64, 1000), 3, False), ((300, 4096), 0, True), ((96, 14336), 0, False),
        ((257, 4096), 2, True), ((520, 14336), 6, False)]


@pytest.mark.parametrize("shape,t,single", GEMV)
@pytest.mark.parametrize("batch", [1, 3, 16])
def test_gemv_matches_oracle(ec, shape, t, single, batch):
    w = synth.llama_bf16(8700 + shape[0], *shape)
    x = synth.make_x(8701, batch, shape[1])
    W = ec.encode_bf16_exp(w, top_t=t, single=single)
    y = torch.full((batch, shape[0]), float("nan"), device="cuda")
    ec.gemv(W, torch.from_numpy(x.view(np.int16)).cuda(), y, batch=batch)
    assert ec.status() == 0
    y_ref, a_ref = O.gemv_bf16(w, x)
    check_gemv(y.cpu().numpy().astype(np.float64), y_ref, a_ref, f"exp gemv {shape} t={t} b={batch}")


def test_full_size_gemv_sampled(ec):
    """14336 x 4096 (the 8B gate shape), pair symbols, batch 1: rows sampled over the
    whole matrix against the oracle."""
    w = synth.llama_bf16(8800, 14336, 4096)
    x = synth.make_x(8801, 1, 4096)
    W = ec.encode_bf16_exp(w)
    y = torch.full((1, 14336), float("nan"), device="cuda")
    ec.gemv(W, torch.from_numpy(x.view(np.int16)).cuda(), y)
    assert ec.status() == 0
    rows = np.arange(0, 14336, 37, dtype=np.int64)
    y_ref, a_ref = O.gemv_bf16(w, x, rows=rows)
    check_gemv(y.cpu().numpy()[:, rows].astype(np.float64), y_ref, a_ref, "exp 14336x4096")


def test_group_and_gemm_routes(ec):
    """gemv_group over three matrices of one width, and the prefill route (ec_gemm)."""
    ws = [synth.llama_bf16(8900 + i, n, 1024) for i, n in enumerate((100, 256, 37))]
    Ws = [ec.encode_bf16_exp(w, top_t=(0, 4, 0)[i]) for i, w in enumerate(ws)]
    x = synth.make_x(8903, 5, 1024)
    xd = torch.from_numpy(x.view(np.int16)).cuda()
    ys = [torch.full((5, w.shape[0]), float("nan"), device="cuda") for w in ws]
    ec.gemv_group(Ws, xd, ys, batch=5)
    assert ec.status() == 0
    for w, y in zip(ws, ys):
        y_ref, a_ref = O.gemv_bf16(w, x)
        check_gemv(y.cpu().numpy().astype(np.float64), y_ref, a_ref, "exp group")
    xg = synth.make_x(8904, 64, 1024)
    for w, W in zip(ws, Ws):
        y = torch.full((64, w.shape[0]), float("nan"), device="cuda")
        ec.gemm(W, torch.from_numpy(xg.view(np.int16)).cuda(), y, 64)
        assert ec.status() == 0
        y_ref, a_ref = O.gemv_bf16(w, xg)
        check_gemv(y.cpu().numpy().astype(np.float64), y_ref, a_ref, "exp gemm")


def test_payload_corruption_is_reported(ec):
    """A flipped payload word breaks the tiles' final-state check: EC_ERR_CORRUPT from
    the decode and from the GEMV."""
    from test_abi import parse
    w = synth.llama_bf16(9000, 64, 4096)
    W = ec.encode_bf16_exp(w)
    blob = bytearray(W.serialize())
    h, dev = parse(bytes(blob))
    meta = len(blob) - len(dev)
    toff = np.frombuffer(dev, np.uint32, h["n_tiles"] + 1, h["tile_off_off"])
    at = meta + h["records_off"] + 16 * int(toff[3]) + 128 + 10  # a word of tile 3
    blob[at] ^= 0x5A
    Wc = ec.deserialize(bytes(blob), device=0)
    out = torch.zeros((64, 4096), dtype=torch.int16, device="cuda")
    assert ec.status() == 0
    ec.decode(Wc, out)
    assert ec.status() == -5
    y = torch.zeros((1, 64), device="cuda")
    ec.gemv(Wc, torch.zeros((1, 4096), dtype=torch.int16, device="cuda"), y)
    assert ec.status() == -5
