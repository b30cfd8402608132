"""GPU parity of the tensor-core Huffman GEMV (tcgen05, batch >= 6 on matrices
whose tiles lie inside rows) against the oracle's FP64 GEMV, through the C ABI:
relative L2 <= 1e-3 and |err| <= 2e-3 * sum|w x| per output."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from parity import check_gemv
from test_abi import parse
from test_gpu_huffman import fib_weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ec():
    import lossless_entropy_coded_gb300 as ec
    return ec


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run(ec, Ws, x, batch):
    ys = [torch.full((batch, W.n_rows), float("nan"), device="cuda") for W in Ws]
    ec.gemv_group(Ws, dev(x.view(np.int16)), ys, batch=batch)
    assert ec.status() == 0
    return [y.cpu().numpy() for y in ys]


@pytest.mark.parametrize("shape", [(256, 4096), (96, 14336), (100, 1024), (7, 13), (33, 2049), (1, 512)])
@pytest.mark.parametrize("batch", [6, 8, 16, 24, 32, 33, 64])
def test_mma_gemv_parity(ec, shape, batch):
    w = synth.llama_bf16(2300 + shape[0], *shape)
    W = ec.encode_bf16(w)
    h, _ = parse(W.serialize())
    assert h["k_pad"] % (32 * h["steps"]) == 0  # tiles inside rows: the tensor-core layout
    assert ec.gemv_path(W, batch) == ("tensor_cores" if shape[1] % 8 == 0 else "cuda_cores")
    x = synth.make_x(2400 + batch, batch, shape[1])
    (y,) = run(ec, [W], x, batch)
    y_ref, a_ref = O.gemv_bf16(w, x)
    check_gemv(y, y_ref, a_ref, f"{shape} b={batch}")


@pytest.mark.parametrize("shape,batch", [((8192, 1024), 6), ((8192, 1024), 17), ((14336, 4096), 8)])
def test_mma_several_items_per_cta(ec, shape, batch):
    """More work items than SMs: CTAs move from item to item (code-area prefetch, x
    of the next item's first chunk, the previous item's accumulators read one chunk
    late while the next item accumulates into the other TMEM half)."""
    w = synth.llama_bf16(3100 + shape[1], *shape)
    W = ec.encode_bf16(w)
    x = synth.make_x(3110 + batch, batch, shape[1])
    (y,) = run(ec, [W], x, batch)
    y_ref, a_ref = O.gemv_bf16(w, x)
    check_gemv(y, y_ref, a_ref, f"{shape} b={batch}")


@pytest.mark.parametrize("batch", [6, 16, 32])
def test_mma_group_of_three(ec, batch):
    """q/k/v-shaped group (different row counts, one K) in one launch."""
    ws = [synth.llama_bf16(2500 + i, n, 4096) for i, n in enumerate((512, 128, 136))]
    Ws = [ec.encode_bf16(w) for w in ws]
    x = synth.make_x(2510, batch, 4096)
    for y, w in zip(run(ec, Ws, x, batch), ws):
        y_ref, a_ref = O.gemv_bf16(w, x)
        check_gemv(y, y_ref, a_ref, f"group b={batch}")


@pytest.mark.parametrize("max_len", [24, 16])
def test_mma_long_codes(ec, max_len):
    """Codewords longer than the pair-table window walk the hierarchical table."""
    w = fib_weights()
    W = ec.encode_bf16(w, max_code_len=max_len)
    assert W.code_lengths().max() == max_len
    x = synth.make_x(2600, 16, w.shape[1])
    (y,) = run(ec, [W], x, 16)
    y_ref, a_ref = O.gemv_bf16(w, x)
    check_gemv(y, y_ref, a_ref, f"long codes {max_len}")


@pytest.mark.parametrize("batch", [16, 40])
def test_tiles_crossing_rows_stay_on_cuda_cores(ec, batch):
    """128-step tiles over K = 14336 cross rows: the CUDA-core kernel, in passes of 16."""
    w = synth.llama_bf16(2700, 64, 14336)
    W = ec.encode_bf16(w, tile_steps=128)
    assert W.stats()["k_pad"] % (32 * 128) != 0
    x = synth.make_x(2710, batch, 14336)
    (y,) = run(ec, [W], x, batch)
    y_ref, a_ref = O.gemv_bf16(w, x)
    check_gemv(y, y_ref, a_ref, f"crossing b={batch}")


def test_mma_repeated_calls_identical(ec):
    """Row sums are stored (one 128-step tile per row at K = 4096) and the eight
    partial accumulator tiles are added in a fixed order: repeated calls give
    identical y."""
    w = synth.llama_bf16(2800, 1024, 4096)
    W = ec.encode_bf16(w)
    h, _ = parse(W.serialize())
    assert h["steps"] == 128
    x = synth.make_x(2810, 16, 4096)
    a = run(ec, [W], x, 16)[0]
    b = run(ec, [W], x, 16)[0]
    assert np.array_equal(a, b)
    y_ref, a_ref = O.gemv_bf16(w, x)
    check_gemv(a, y_ref, a_ref, "repeat")


def test_mma_payload_corruption_is_reported_not_faulted(ec):
    """Lane 3 of tile 0 overwritten with ones (every lookup then decodes the 12-bit
    all-ones codeword): the tensor-core kernel's end-of-tile check must report it."""
    from test_abi import tile_layout, lane_starts
    w = synth.llama_bf16(2900, 64, 4096)
    W = ec.encode_bf16(w)
    blob = bytearray(W.serialize())
    h, devb = parse(bytes(blob))
    meta = len(blob) - len(devb)
    rec, S, _, _, area_off, _ = tile_layout(h, devb, 0)
    st = lane_starts(devb, rec)
    for b in range(area_off + st[3], area_off + st[4]):
        blob[meta + b] = 0xFF
    Wc = ec.deserialize(bytes(blob), device=0)
    x = synth.make_x(2910, 16, 4096)
    y = torch.zeros((16, 64), device="cuda")
    assert ec.gemv_path([Wc], 16) == "tensor_cores"
    ec.gemv(Wc, dev(x.view(np.int16)), y, batch=16)
    assert ec.status() == -5
    # the context is still healthy: the clean matrix gives the right product
    y_ref, a_ref = O.gemv_bf16(w, x)
    (y2,) = run(ec, [W], x, 16)
    check_gemv(y2, y_ref, a_ref, "clean after corrupt")
