"""GPU parity of the FP8 path (MINE section 4, "Escapes": a top-t decoding table
with 0 always kept and per-tile correction records) against the oracle, through
the C ABI.  Decode: bf16(value * r_i) bit-exact with the oracle's dequantisation.
GEMV: within relative L2 <= 1e-3 and |err| <= 2e-3 * sum|w x| of the oracle's FP64
GEMV."""
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


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("t", [0, 2, 16, 64])
@pytest.mark.parametrize("shape,tile", [((1, 1), 4096), ((7, 300), 128), ((64, 1000), 4096), ((40, 4096), 1024),
                                        ((17, 14336), 4096)])
def test_decode(ec, shape, tile, t):
    codes, r = synth.make_fp8_case(8100 + shape[0], *shape)
    W = ec.encode_fp8(codes, r, top_t=t, tile_syms=tile)
    out = torch.full(shape, -1, dtype=torch.int16, device="cuda")
    ec.decode(W, out)
    assert ec.status() == 0
    assert np.array_equal(out.cpu().numpy().view(np.uint16), O.fp8_dequant_bf16(codes, r))


@pytest.mark.parametrize("t", [0, 32])
@pytest.mark.parametrize("shape", [(7, 300), (64, 1000), (256, 4096), (64, 14336)])
@pytest.mark.parametrize("batch", [1, 4, 16, 24])
def test_gemv_parity(ec, shape, batch, t):
    codes, r = synth.make_fp8_case(8200 + shape[1], *shape)
    x = synth.make_x(8300, batch, shape[1])
    W = ec.encode_fp8(codes, r, top_t=t)
    y = torch.full((batch, shape[0]), float("nan"), device="cuda")
    ec.gemv(W, dev(x.view(np.int16)), y, batch=batch)
    assert ec.status() == 0
    y_ref, a_ref = O.gemv_fp8(codes, r, x)
    check_gemv(y.cpu().numpy(), y_ref, a_ref, f"{shape} b={batch} t={t}")


def test_escape_heavy(ec):
    """t = 1: only code 0 in the table, every other weight is a correction record."""
    codes, r = synth.make_fp8_case(8400, 32, 4096)
    W = ec.encode_fp8(codes, r, top_t=1)
    out = torch.zeros((32, 4096), dtype=torch.int16, device="cuda")
    ec.decode(W, out)
    assert ec.status() == 0
    assert np.array_equal(out.cpu().numpy().view(np.uint16), O.fp8_dequant_bf16(codes, r))
    x = synth.make_x(8401, 2, 4096)
    y = torch.zeros((2, 32), device="cuda")
    ec.gemv(W, dev(x.view(np.int16)), y, batch=2)
    assert ec.status() == 0
    y_ref, a_ref = O.gemv_fp8(codes, r, x)
    check_gemv(y.cpu().numpy(), y_ref, a_ref, "t=1")


@pytest.mark.parametrize("shape", [(14336, 4096), (4096, 14336)])
def test_full_size_config(ec, shape):
    """Llama-3.1-8B gate/up and down shapes with a 32-code table: decode bit-exact
    on every weight and the batch-1 GEMV on every row."""
    codes, r = synth.make_fp8_case(8500 + shape[1], *shape)
    W = ec.encode_fp8(codes, r, top_t=32)
    out = torch.empty(shape, dtype=torch.int16, device="cuda")
    ec.decode(W, out)
    assert ec.status() == 0
    assert np.array_equal(out.cpu().numpy().view(np.uint16), O.fp8_dequant_bf16(codes, r))
    x = synth.make_x(8501, 1, shape[1])
    y = torch.empty((1, shape[0]), device="cuda")
    ec.gemv(W, dev(x.view(np.int16)), y, batch=1)
    assert ec.status() == 0
    y_ref, a_ref = O.gemv_fp8(codes, r, x)
    check_gemv(y.cpu().numpy(), y_ref, a_ref, f"{shape}")


def test_mixed_kind_decode_batch(ec):
    codes, r = synth.make_fp8_case(8600, 48, 1000)
    c4, s4 = synth.make_rans_case(0, 40, 1000)
    Ws = [ec.encode_fp8(codes, r, top_t=8), ec.encode_rans(c4, s4)]
    outs = [torch.zeros(W.shape, dtype=torch.int16, device="cuda") for W in Ws]
    ec.decode_batch(Ws, outs)
    assert ec.status() == 0
    assert np.array_equal(outs[0].cpu().numpy().view(np.uint16), O.fp8_dequant_bf16(codes, r))
    assert np.array_equal(outs[1].cpu().numpy().view(np.uint16), O.rans_dequant_bf16(c4, s4))
    assert ec.gemv_path(Ws[0], 16) == "cuda_cores"


def test_payload_corruption_is_reported(ec):
    codes, r = synth.make_fp8_case(8700, 32, 4096)
    W = ec.encode_fp8(codes, r, top_t=16)
    blob = bytearray(W.serialize())
    from test_abi import parse
    h, devb = parse(bytes(blob))
    meta = len(blob) - len(devb)
    blob[meta + h["records_off"] + 128 + 10] ^= 0x81  # a payload word of tile 0
    Wc = ec.deserialize(bytes(blob), device=0)
    out = torch.zeros((32, 4096), dtype=torch.int16, device="cuda")
    ec.decode(Wc, out)
    # the rANS tile's final states no longer return to 2^16: reported
    assert ec.status() == -5
