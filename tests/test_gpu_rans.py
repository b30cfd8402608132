"""GPU parity of the rANS tile path against the oracle, through the C ABI.

Decode: BF16(code * scale) bit-exact with the oracle's dequantisation (the oracle
also decodes its own tiles back to the codes).  GEMV: within relative L2 <= 1e-3
and |err| <= 2e-3 * sum|w x| of the oracle's FP64 GEMV."""
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


@pytest.mark.parametrize("tuple_", [1, 2])
@pytest.mark.parametrize("shape", [(1, 1), (7, 13), (3, 300), (64, 1000), (40, 4096), (17, 14336)])
def test_decode_ragged(ec, shape, tuple_):
    codes, scales = synth.make_rans_case(0, *shape)
    W = ec.encode_rans(codes, scales, codes_per_symbol=tuple_)
    out = torch.zeros(shape, dtype=torch.int16, device="cuda")
    ec.decode(W, out)
    assert ec.status() == 0
    assert np.array_equal(out.cpu().numpy().view(np.uint16), O.rans_dequant_bf16(codes, scales))


@pytest.mark.parametrize("tuple_", [1, 2])
@pytest.mark.parametrize("shape", [(7, 13), (64, 1000), (256, 4096), (64, 14336)])
@pytest.mark.parametrize("batch", [1, 4, 16])
def test_gemv_parity(ec, shape, batch, tuple_):
    codes, scales = synth.make_rans_case(1, *shape)
    x = synth.make_x(4100, batch, shape[1])
    W = ec.encode_rans(codes, scales, codes_per_symbol=tuple_)
    y = torch.full((batch, shape[0]), float("nan"), device="cuda")
    ec.gemv(W, dev(x.view(np.int16)), y, batch=batch)
    assert ec.status() == 0
    y_ref, a_ref = O.gemv_rans(codes, scales, x)
    check_gemv(y.cpu().numpy(), y_ref, a_ref, f"{shape} b={batch}")


@pytest.mark.parametrize("tuple_", [1, 2])
@pytest.mark.parametrize("idx", [0, 1])
def test_full_size_config(ec, idx, tuple_):
    """14336x4096 and 4096x14336 at full size, single and pair symbols: bit-exact
    dequantised decode against the oracle and the oracle's own tile codec round
    trip; GEMV on all rows."""
    codes, scales = synth.make_rans_case(idx)
    n, k = codes.shape
    r = O.Rans(codes, k=tuple_)
    dec, fin, rc = r.decode()
    assert rc == 0 and np.array_equal(dec, codes.ravel())
    W = ec.encode_rans(codes, scales, codes_per_symbol=tuple_)
    out = torch.zeros((n, k), dtype=torch.int16, device="cuda")
    ec.decode(W, out)
    assert ec.status() == 0
    assert np.array_equal(out.cpu().numpy().view(np.uint16), O.rans_dequant_bf16(codes, scales))
    x = synth.make_x(4000 + idx, 1, k)
    y = torch.zeros((1, n), device="cuda")
    ec.gemv(W, dev(x.view(np.int16)), y, batch=1)
    assert ec.status() == 0
    y_ref, a_ref = O.gemv_rans(codes, scales, x)
    check_gemv(y.cpu().numpy(), y_ref, a_ref, f"rans full {idx}")
    s = W.stats()
    assert s["bits_per_weight"] < 2.9


def test_mixed_tuple_group(ec):
    """One grouped launch over a single-symbol and a pair-symbol matrix of the same K."""
    k = 4096
    c0, s0 = synth.make_rans_case(5, 96, k)
    c1, s1 = synth.make_rans_case(6, 160, k)
    W0 = ec.encode_rans(c0, s0)
    W1 = ec.encode_rans(c1, s1, codes_per_symbol=2)
    x = synth.make_x(4200, 1, k)
    y0 = torch.full((1, 96), float("nan"), device="cuda")
    y1 = torch.full((1, 160), float("nan"), device="cuda")
    ec.gemv_group([W0, W1], dev(x.view(np.int16)), [y0, y1], batch=1)
    assert ec.status() == 0
    for y, c, s in ((y0, c0, s0), (y1, c1, s1)):
        y_ref, a_ref = O.gemv_rans(c, s, x)
        check_gemv(y.cpu().numpy(), y_ref, a_ref, "mixed tuple group")


@pytest.mark.parametrize("tuple_", [1, 2])
def test_payload_corruption_is_reported(ec, tuple_):
    codes, scales = synth.make_rans_case(0, 32, 4096)
    W = ec.encode_rans(codes, scales, codes_per_symbol=tuple_)
    blob = bytearray(W.serialize())
    from test_abi import parse
    h, devb = parse(bytes(blob))
    meta = len(blob) - len(devb)
    rec = meta + h["records_off"]
    blob[rec + 128 + 10] ^= 0x81  # a payload word of tile 0
    Wc = ec.deserialize(bytes(blob), device=0)
    out = torch.zeros((32, 4096), dtype=torch.int16, device="cuda")
    ec.decode(Wc, out)
    # the flipped word changes every later state of its lane: the final states (2^16 each)
    # and the count of words used no longer match, which the decoder reports
    assert ec.status() == -5


@pytest.mark.parametrize("tuple_", [1, 2])
def test_automatic_table_size_decodes(ec, tuple_):
    """A matrix whose automatic table is small (uniform codes: 2^9 slots) decodes
    bit-exactly and multiplies within tolerance."""
    rng = np.random.default_rng(9 + tuple_)
    codes = rng.integers(-8, 8, size=(64, 4096)).astype(np.int8)
    scales = synth.make_rans_case(0, 64, 4096)[1]
    W = ec.encode_rans(codes, scales, prob_bits=0, codes_per_symbol=tuple_)
    assert W.stats()["max_code_len"] == 9
    out = torch.zeros((64, 4096), dtype=torch.int16, device="cuda")
    ec.decode(W, out)
    assert ec.status() == 0
    assert np.array_equal(out.cpu().numpy().view(np.uint16), O.rans_dequant_bf16(codes, scales))
    x = synth.make_x(4300, 4, 4096)
    y = torch.zeros((4, 64), device="cuda")
    ec.gemv(W, dev(x.view(np.int16)), y, batch=4)
    assert ec.status() == 0
    y_ref, a_ref = O.gemv_rans(codes, scales, x)
    check_gemv(y.cpu().numpy(), y_ref, a_ref, "automatic table")


@pytest.mark.parametrize("tuple_", [1, 2])
@pytest.mark.parametrize("shape", [(7, 13), (64, 1000), (256, 4096), (33, 14336)])
def test_fp4_decode_and_gemv(ec, shape, tuple_):
    """FP4 E2M1 codes (values="fp4"): decode bit-exact with the oracle's BF16 of
    e2m1(code) * scale; GEMV at batch 1 and 4 within the GEMV tolerance."""
    codes, scales = synth.make_fp4_case(4400 + shape[0], *shape)
    W = ec.encode_rans(codes, scales, codes_per_symbol=tuple_, values="fp4")
    out = torch.zeros(shape, dtype=torch.int16, device="cuda")
    ec.decode(W, out)
    assert ec.status() == 0
    assert np.array_equal(out.cpu().numpy().view(np.uint16), O.rans_dequant_bf16(codes, scales, values="fp4"))
    for batch in (1, 4):
        x = synth.make_x(4401, batch, shape[1])
        y = torch.full((batch, shape[0]), float("nan"), device="cuda")
        ec.gemv(W, dev(x.view(np.int16)), y, batch=batch)
        assert ec.status() == 0
        y_ref, a_ref = O.gemv_rans(codes, scales, x, values="fp4")
        check_gemv(y.cpu().numpy(), y_ref, a_ref, f"fp4 {shape} k={tuple_} b={batch}")


@pytest.mark.parametrize("lo,hi", [(-2, 1), (-4, 3)])
def test_int2_and_int3_codes_through_pairs(ec, lo, hi):
    """int2 and int3 codes are subranges of the 4-bit codec: pair symbols over them
    decode bit-exact and multiply within tolerance."""
    shape = (96, 4096)
    codes = synth.codes_i8(4500 + hi, shape, std=1.0, lo=lo, hi=hi)
    scales = synth.scales_f16(4501, (shape[0], shape[1] // 128))
    W = ec.encode_rans(codes, scales, codes_per_symbol=2)
    out = torch.zeros(shape, dtype=torch.int16, device="cuda")
    ec.decode(W, out)
    assert ec.status() == 0
    assert np.array_equal(out.cpu().numpy().view(np.uint16), O.rans_dequant_bf16(codes, scales))
    x = synth.make_x(4502, 1, shape[1])
    y = torch.full((1, shape[0]), float("nan"), device="cuda")
    ec.gemv(W, dev(x.view(np.int16)), y, batch=1)
    assert ec.status() == 0
    y_ref, a_ref = O.gemv_rans(codes, scales, x)
    check_gemv(y.cpu().numpy(), y_ref, a_ref, f"int{hi.bit_length() + 1}")
    assert W.stats()["bits_per_weight"] < (2.6 if hi == 1 else 3.5)
