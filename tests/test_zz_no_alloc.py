"""GPU test of ec_gemv_static, the GEMV entry point that allocates nothing.

It is compared, through the C ABI, with the regular ec_gemv on the same encoded
matrices and inputs, within the GEMV tolerance the other tests use (relative L2
<= 1e-3 and |err| <= 2e-3 * sum|w x| against the FP64 oracle, and the two GPU
results against each other), on two calls in a row: the second call reuses the
built-in scratch the first one left behind.  This file is collected last so a run
that stops at the first failure has already run every other test."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from parity import check_gemv

pytestmark = pytest.mark.gpu


# (max code length, hierarchical decode): window records with the default limit; with
# codewords up to 24 bits coded as records; and through DFloat11's sub-tables
CODES = [(12, False), (24, False), (24, True)]


@pytest.mark.parametrize("code", CODES)
@pytest.mark.parametrize("shape", [(256, 4096), (96, 14336), (7, 13), (300, 1000)])
@pytest.mark.parametrize("batch", [1, 3, 16])
def test_static_gemv_matches_ec_gemv_twice(shape, batch, code):
    """Batch 16 over 14336 columns takes several passes (x of 16 rows of 14336 BF16 values
    does not fit next to the tile buffers), each writing its own batch rows."""
    import lossless_entropy_coded_gb300 as ec
    w = synth.llama_bf16(2700 + shape[0], *shape)
    x = synth.make_x(2700, batch, shape[1])
    W = ec.encode_bf16(w, max_code_len=code[0], hierarchical=code[1])
    if code[0] == 24 and shape[0] * shape[1] >= 256 * 1000:
        assert W.code_lengths().max() > 12  # codewords longer than the pair window
    xd = torch.from_numpy(x.view(np.int16)).cuda()
    y_ref_gpu = torch.full((batch, shape[0]), float("nan"), device="cuda")
    ec.gemv(W, xd, y_ref_gpu, batch=batch)
    assert ec.status() == 0
    y_ref, a_ref = O.gemv_bf16(w, x)
    y_ref_gpu = y_ref_gpu.cpu().numpy().astype(np.float64)
    for call in range(2):
        y = torch.full((batch, shape[0]), float("nan"), device="cuda")
        ec.gemv_static(W, xd, y, batch=batch)
        torch.cuda.synchronize()
        ys = y.cpu().numpy().astype(np.float64)
        check_gemv(ys, y_ref, a_ref, f"static call {call} {shape} b={batch}")
        assert (np.abs(ys - y_ref_gpu) <= 2e-3 * a_ref + 1e-30).all()
        assert np.linalg.norm(ys - y_ref_gpu) <= 1e-3 * np.linalg.norm(y_ref)


def test_static_gemv_rejects_oversized_requests():
    import lossless_entropy_coded_gb300 as ec
    # 8192 rows x 28672 columns at batch 16 needs 8192 * 16 * 8 partial sums: more than the 4 MiB scratch
    w = np.zeros((8192, 28672), np.uint16)
    W = ec.encode_bf16(w)
    x = torch.zeros((16, 28672), dtype=torch.int16, device="cuda")
    y = torch.zeros((16, 8192), device="cuda")
    with pytest.raises(ec.EcError) as e:
        ec.gemv_static(W, x, y, batch=16)
    assert e.value.code == -4
    ec.gemv_static(W, x[:1], y[:1], batch=1)  # a size that fits still runs
    torch.cuda.synchronize()
    assert (y[:1] == 0).all()


@pytest.mark.parametrize("hier", [False, True])
def test_static_gemv_reports_corruption(hier):
    """A payload the walker must reject (lane 3 of tile 0 overwritten with ones, see
    test_gpu_huffman) is reported through ec_status after a static call, and the
    report survives until ec_status reads it."""
    import lossless_entropy_coded_gb300 as ec
    from test_abi import parse, tile_layout, lane_starts
    w = synth.llama_bf16(2500, 64, 4096)
    W = ec.encode_bf16(w, hierarchical=hier)
    blob = bytearray(W.serialize())
    h, devb = parse(bytes(blob))
    meta = len(blob) - len(devb)
    rec, S, _, _, area_off, _ = tile_layout(h, devb, 0)
    st = lane_starts(devb, rec)
    for b in range(area_off + st[3], area_off + st[4]):
        blob[meta + b] = 0xFF
    Wc = ec.deserialize(bytes(blob), device=0)
    x = torch.from_numpy(synth.make_x(2500, 1, 4096).view(np.int16)).cuda()
    y = torch.zeros((1, 64), device="cuda")
    assert ec.status() == 0
    ec.gemv_static(Wc, x, y, batch=1)
    ec.gemv_static(W, x, y, batch=1)  # a clean call after it does not clear the report
    assert ec.status() == -5
    assert ec.status() == 0
