"""GPU parity of the E8 lattice decode (EntroPack sections 3.6, 3.7) against the
oracle, through the C ABI: the BF16 weights bf16(fp32(q * fp32(s * r_i)) * 0.5)
bit-exact with the oracle's reconstruction of the same points (the oracle also
decodes its own tiles of the same stream back to the points)."""
import numpy as np
import pytest
import torch

import oracle as O
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ec():
    import lossless_entropy_coded_gb300 as ec
    return ec


def decode(ec, W, shape):
    out = torch.full(shape, -1, dtype=torch.int16, device="cuda")
    ec.decode(W, out)
    assert ec.status() == 0
    return out.cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("shape,tile,b", [((1, 8), 32, 11), ((3, 256), 32, 11), ((7, 264), 64, 9),
                                          ((40, 1024), 512, 11), ((33, 776), 96, 12), ((2, 4096), 1024, 10),
                                          ((64, 14336), 512, 11), ((300, 4096), 1024, 12)])
def test_decode_ragged(ec, shape, tile, b):
    q2, r, s = synth.make_e8_case(7000 + shape[0], *shape)
    W = ec.encode_e8(q2, r, s, prob_bits=b, tile_vectors=tile)
    got = decode(ec, W, shape)
    assert np.array_equal(got, O.e8_reconstruct_bf16(q2, s, r))


def test_decode_empty(ec):
    W = ec.encode_e8(np.zeros((0, 256), np.int8), np.zeros(0, np.float32), 1.0)
    out = torch.zeros((0, 256), dtype=torch.int16, device="cuda")
    ec.decode(W, out)
    assert ec.status() == 0


def test_one_coset_only(ec):
    """Every point in D8 (c = 0): the eight coset-1 tables are unused and empty."""
    q2, r, s = synth.make_e8_case(31, 48, 1024)
    q2 = (q2 - (q2 & 1)).astype(np.int8)  # drop the coset offset: 2 z stays in 2 D8
    W = ec.encode_e8(q2, r, s)
    assert np.array_equal(decode(ec, W, q2.shape), O.e8_reconstruct_bf16(q2, s, r))


def test_power_of_two_scales_are_exact(ec):
    """With s and r_i powers of two the decoded weights are exactly q / 2 * s * r_i."""
    q2, _, _ = synth.make_e8_case(37, 96, 2048)
    r = (2.0 ** (np.arange(96) % 9 - 6)).astype(np.float32)
    s = 2.0 ** -5
    W = ec.encode_e8(q2, r, s)
    got = decode(ec, W, q2.shape)
    want = q2.astype(np.float64) / 2 * s * r[:, None].astype(np.float64)
    assert np.array_equal(synth.bf16_to_f32(got).astype(np.float64), want)


def test_extreme_row_scales(ec):
    """Rows whose factor g_i = s r_i is subnormal, tiny, huge (q g overflows to
    infinity) or zero take the two-multiply reconstruction; the others the single
    multiply by g_i / 2.  Both agree with the oracle bit for bit."""
    q2, r, s = synth.make_e8_case(47, 12, 512)
    r = r.copy()
    r[0], r[1], r[2], r[3] = 1e-38, 3e-37, 3e38, 0.0
    r[4], r[5] = 2.0 ** -125, 2.0 ** 120  # g on both edges of the single-multiply range
    r[6], r[7] = -0.03, -1e-39
    W = ec.encode_e8(q2, r, 1.0)
    got = decode(ec, W, q2.shape)
    assert np.array_equal(got, O.e8_reconstruct_bf16(q2, 1.0, r))


@pytest.mark.parametrize("dtype", ["e4m3", "int8", "bf16"])
@pytest.mark.parametrize("shape,tile,scale", [((7, 264), 64, 0.125), ((40, 1024), 512, 64.0), ((33, 776), 96, 2000.0),
                                              ((300, 4096), 1024, 400.0)])
def test_decode_as_dtype(ec, dtype, shape, tile, scale):
    """FP8 E4M3 and INT8 output (and BF16 through the same entry point), bit-exact
    with the oracle: scales from E4M3 subnormals up to saturation, INT8 up to its
    clamp."""
    q2, r, _ = synth.make_e8_case(7300 + shape[0], *shape)
    W = ec.encode_e8(q2, r, scale, tile_vectors=tile)
    tdt = torch.int16 if dtype == "bf16" else torch.uint8 if dtype == "e4m3" else torch.int8
    out = torch.full(shape, 0x55, dtype=tdt, device="cuda")
    ec.decode_as(W, out, dtype)
    assert ec.status() == 0
    got = out.cpu().numpy()
    want = O.e8_reconstruct(q2, scale, r, dtype)
    assert np.array_equal(got.view(want.dtype), want)


def test_decode_as_refusals(ec):
    w = synth.llama_bf16(7400, 16, 512)
    H = ec.encode_bf16(w)
    out8 = torch.zeros((16, 512), dtype=torch.uint8, device="cuda")
    with pytest.raises(ec.EcError) as e:
        ec.decode_as(H, out8, "e4m3")
    assert e.value.code == -4
    out16 = torch.zeros((16, 512), dtype=torch.int16, device="cuda")
    ec.decode_as(H, out16, "bf16")
    assert ec.status() == 0 and np.array_equal(out16.cpu().numpy().view(np.uint16), w)
    q2, r, s = synth.make_e8_case(7401, 16, 512)
    E = ec.encode_e8(q2, r, s)
    big = torch.zeros(16 * 512 + 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(ec.EcError) as e:
        ec.decode_as(E, big[1:], "int8")  # not 16-byte aligned
    assert e.value.code == -1


@pytest.mark.parametrize("shape", [(14336, 4096), (4096, 14336)])
def test_full_size_config(ec, shape):
    """Llama-3.1-8B gate/up and down shapes at about 4 bits per weight: the whole
    decoded matrix bit-exact with the oracle's reconstruction, and the oracle's own
    17-table tile codec round trip of a 512-row slice of the same points."""
    q2, r, s = synth.make_e8_case(7100 + shape[1], *shape)
    W = ec.encode_e8(q2, r, s)
    st = W.stats()
    assert 3.0 < st["bits_per_weight"] < 5.0
    got = decode(ec, W, shape)
    assert np.array_equal(got, O.e8_reconstruct_bf16(q2, s, r))
    e = O.E8(q2[:512], prob_bits=11, tile=512)
    pts, _, rc = e.decode()
    assert rc == 0 and np.array_equal(pts.reshape(512, -1), q2[:512])


def test_mixed_kind_decode_batch(ec):
    """One decode_batch call over a Huffman, a rANS and an E8 matrix."""
    w = synth.llama_bf16(7200, 64, 1000)
    codes, scales = synth.make_rans_case(0, 48, 1000)
    q2, r, s = synth.make_e8_case(7201, 80, 1000)
    Ws = [ec.encode_bf16(w), ec.encode_rans(codes, scales), ec.encode_e8(q2, r, s)]
    outs = [torch.zeros(W.shape, dtype=torch.int16, device="cuda") for W in Ws]
    ec.decode_batch(Ws, outs)
    assert ec.status() == 0
    assert np.array_equal(outs[0].cpu().numpy().view(np.uint16), w)
    assert np.array_equal(outs[1].cpu().numpy().view(np.uint16), O.rans_dequant_bf16(codes, scales))
    assert np.array_equal(outs[2].cpu().numpy().view(np.uint16), O.e8_reconstruct_bf16(q2, s, r))


def test_gemv_is_refused(ec):
    q2, r, s = synth.make_e8_case(41, 8, 256)
    W = ec.encode_e8(q2, r, s)
    x = torch.zeros((1, 256), dtype=torch.int16, device="cuda")
    y = torch.zeros((1, 8), device="cuda")
    with pytest.raises(ec.EcError) as e:
        ec.gemv(W, x, y)
    assert e.value.code == -4


@pytest.mark.parametrize("word", [3, 500])
def test_payload_corruption_is_reported(ec, word):
    q2, r, s = synth.make_e8_case(43, 32, 4096)
    W = ec.encode_e8(q2, r, s)
    blob = bytearray(W.serialize())
    from test_abi import parse
    h, devb = parse(bytes(blob))
    meta = len(blob) - len(devb)
    rec = meta + h["records_off"]
    blob[rec + 128 + 2 * word] ^= 0x5A  # a payload word of tile 0
    Wc = ec.deserialize(bytes(blob), device=0)
    out = torch.zeros(q2.shape, dtype=torch.int16, device="cuda")
    ec.decode(Wc, out)
    # the rANS tile's final states no longer return to 2^16: reported
    assert ec.status() == -5
