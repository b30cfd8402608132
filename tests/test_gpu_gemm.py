"""GPU parity of the prefill route (ec_gemm): chunked decode into the work buffer,
then the tensor-core GEMM, against the FP64 oracle.

The route materialises the layer before a GEMM, as MINE does at batch > 1 (section
4, "Prefill") and DFloat11 does per transformer block ("Transformer-block-level
decompression").  The oracle is therefore the plain definition: the matrix the
decoder must write (the original BF16 patterns for Huffman matrices; the BF16
dequantisation of the other codecs), multiplied by x in FP64.  Every output element
is checked at the GEMV tolerance (relative L2 <= 1e-3 and |err| <= 2e-3 * sum|w x|);
repeated calls must agree bit for bit (K splits are added in a fixed order)."""
from concurrent.futures import ThreadPoolExecutor
import os

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


def oracle_gemm(w, x):
    """FP64 y and sum|w x| over row blocks on the host cores (the C oracle releases the GIL)."""
    n = w.shape[0]
    blocks = [(r0, min(n, r0 + 256)) for r0 in range(0, n, 256)]
    with ThreadPoolExecutor(os.cpu_count() or 1) as ex:
        parts = list(ex.map(lambda b: O.gemv_bf16(w, x, rows=np.arange(b[0], b[1], dtype=np.int64)), blocks))
    return np.concatenate([p[0] for p in parts], axis=1), np.concatenate([p[1] for p in parts], axis=1)


def run_gemm(ec, W, x, batch, work=None):
    xd = torch.from_numpy(x.view(np.int16)).cuda()
    y = torch.full((batch, W.n_rows), float("nan"), device="cuda")
    ec.gemm(W, xd, y, batch, work=work)
    assert ec.status() == 0
    return y


# (rows, cols, batch): ragged rows and columns (K % 8 != 0 re-strides x), several
# 128-row tiles and batch tiles, K splits over 4096 and 14336 columns, batch > 256
CASES = [(7, 13, 64), (300, 1000, 65), (1024, 4096, 64), (4096, 4096, 256), (96, 14336, 64), (520, 14336, 300),
         (1000, 512, 16), (129, 4096, 2)]


@pytest.mark.parametrize("rows,cols,batch", CASES)
def test_gemm_matches_oracle(ec, rows, cols, batch):
    w = synth.llama_bf16(3100 + rows, rows, cols)
    x = synth.make_x(3100 + cols, batch, cols)
    W = ec.encode_bf16(w)
    y = run_gemm(ec, W, x, batch)
    y_ref, a_ref = oracle_gemm(w, x)
    check_gemv(y.cpu().numpy().astype(np.float64), y_ref, a_ref, f"gemm {rows}x{cols} b={batch}")
    y2 = run_gemm(ec, W, x, batch)
    assert torch.equal(y, y2), "repeated ec_gemm calls differ"


@pytest.mark.parametrize("code", [(24, False), (24, True), (12, True)])
def test_gemm_long_codes_and_hierarchical(ec, code):
    w = synth.llama_bf16(3300, 640, 4096)
    x = synth.make_x(3301, 96, 4096)
    W = ec.encode_bf16(w, max_code_len=code[0], hierarchical=code[1])
    y = run_gemm(ec, W, x, 96)
    y_ref, a_ref = oracle_gemm(w, x)
    check_gemv(y.cpu().numpy().astype(np.float64), y_ref, a_ref, f"gemm code {code}")


@pytest.mark.parametrize("fraction", [2, 7])
def test_gemm_small_work_buffer_takes_more_chunks(ec, fraction):
    """A work buffer below the full-size request makes the chunks smaller: the same
    result from many decode + GEMM rounds (each chunk a row range of whole tiles)."""
    rows, cols, batch = 2304, 14336, 64
    w = synth.llama_bf16(3400, rows, cols)
    x = synth.make_x(3401, batch, cols)
    W = ec.encode_bf16(w)
    full = ec.gemm_work_bytes(W, batch)
    work = torch.empty(full // fraction, dtype=torch.uint8, device="cuda")
    y = run_gemm(ec, W, x, batch, work=work)
    y_ref, a_ref = oracle_gemm(w, x)
    check_gemv(y.cpu().numpy().astype(np.float64), y_ref, a_ref, f"gemm work/{fraction}")


def test_gemm_rejects_a_work_buffer_below_one_chunk(ec):
    w = synth.llama_bf16(3500, 512, 4096)
    W = ec.encode_bf16(w)
    x = torch.zeros((64, 4096), dtype=torch.int16, device="cuda")
    y = torch.zeros((64, 512), device="cuda")
    work = torch.empty(4096, dtype=torch.uint8, device="cuda")
    with pytest.raises(ec.EcError) as e:
        ec.gemm(W, x, y, 64, work=work)
    assert e.value.code == -1


def test_full_size_layer_matrices_sampled(ec):
    """Layer 0 of the 8B stack at batch 128 through ec_gemm: every matrix, rows sampled
    across all chunks (the oracle computes them one by one)."""
    for spec in synth.layer_8b(0):
        w = synth.make_weights(spec)
        W = ec.encode_bf16(w)
        x = synth.make_x(spec.seed, 128, spec.k_cols)
        y = run_gemm(ec, W, x, 128).cpu().numpy().astype(np.float64)
        rows = np.unique(np.concatenate([np.arange(0, spec.n_rows, 97), [spec.n_rows - 1]])).astype(np.int64)
        y_ref, a_ref = O.gemv_bf16(w, x, rows=rows)
        check_gemv(y[:, rows], y_ref, a_ref, f"{spec.name} b=128")


def test_bf16_gemm_matches_oracle(ec):
    rows, cols, batch = 1536, 4096, 128
    w = synth.llama_bf16(3600, rows, cols)
    x = synth.make_x(3601, batch, cols)
    wd = torch.from_numpy(w.view(np.int16)).cuda()
    xd = torch.from_numpy(x.view(np.int16)).cuda()
    y_ref, a_ref = oracle_gemm(w, x)
    for work in (None, torch.empty(64 << 20, dtype=torch.uint8, device="cuda")):
        y = torch.full((batch, rows), float("nan"), device="cuda")
        ec.bf16_gemm(wd, xd, y, batch, work=work)
        torch.cuda.synchronize()
        check_gemv(y.cpu().numpy().astype(np.float64), y_ref, a_ref, f"bf16_gemm work={work is not None}")


def test_gemm_other_codecs(ec):
    """rANS 4-bit, FP8 and E8 matrices decode whole into the work buffer: the oracle is
    their BF16 dequantisation times x."""
    batch = 80
    codes, scales = synth.make_rans_case(0, 384, 4096)
    cases = [(ec.encode_rans(codes, scales), O.rans_dequant_bf16(codes, scales))]
    fc, fr = synth.make_fp8_case(3700, 256, 2048)
    cases.append((ec.encode_fp8(fc, fr), O.fp8_dequant_bf16(fc, fr)))
    q2, rs, s = synth.make_e8_case(3701, 200, 1024)
    cases.append((ec.encode_e8(q2, rs, s), O.e8_reconstruct_bf16(q2, s, rs)))
    for W, wb in cases:
        x = synth.make_x(3702, batch, W.k_cols)
        y = run_gemm(ec, W, x, batch)
        y_ref, a_ref = oracle_gemm(wb, x)
        check_gemv(y.cpu().numpy().astype(np.float64), y_ref, a_ref, f"gemm kind {W.kind}")


def test_gemm_reports_corruption(ec):
    """Lane 3 of tile 0 overwritten with ones (as in test_gpu_huffman): the chunk decode
    reports it through ec_status."""
    from test_abi import parse, tile_layout, lane_starts
    w = synth.llama_bf16(3800, 256, 4096)
    W = ec.encode_bf16(w)
    blob = bytearray(W.serialize())
    h, devb = parse(bytes(blob))
    meta = len(blob) - len(devb)
    rec, S, _, _, area_off, _ = tile_layout(h, devb, 0)
    st = lane_starts(devb, rec)
    for b in range(area_off + st[3], area_off + st[4]):
        blob[meta + b] = 0xFF
    Wc = ec.deserialize(bytes(blob), device=0)
    x = torch.zeros((64, 4096), dtype=torch.int16, device="cuda")
    y = torch.zeros((64, 256), device="cuda")
    assert ec.status() == 0
    ec.gemm(Wc, x, y, 64)
    assert ec.status() == -5


def test_gemm_group_matches_oracle(ec):
    """ec_gemm_group over matrices with their own x: Huffman matrices decoded together,
    one with K % 8 != 0 and an exponent-codec matrix taken alone; with the full work
    buffer (one decode launch for the packable ones), then with 1.5 MB, where the pack
    splits over several decode launches and the largest matrix, bigger than the area
    left beside the partial sums, goes alone in row chunks."""
    batch = 48
    specs = [(256, 1024), (96, 1024), (300, 1000), (128, 13), (1100, 1024), (200, 1024)]
    ws = [synth.llama_bf16(3900 + i, n, k) for i, (n, k) in enumerate(specs)]
    Ws = [ec.encode_bf16(w) for w in ws[:5]] + [ec.encode_bf16_exp(ws[5])]
    xs = [synth.make_x(3950 + i, batch, k) for i, (_, k) in enumerate(specs)]
    xd = [torch.from_numpy(x.view(np.int16)).cuda() for x in xs]
    refs = [oracle_gemm(w, x) for w, x in zip(ws, xs)]
    full = ec.gemm_group_work_bytes(Ws, batch)
    for work_bytes in (full, 1536 * 1024):
        work = torch.empty(work_bytes, dtype=torch.uint8, device="cuda")
        ys = [torch.full((batch, n), float("nan"), device="cuda") for n, _ in specs]
        ec.gemm_group(Ws, xd, ys, batch, work=work)
        assert ec.status() == 0
        for i, (y, (y_ref, a_ref)) in enumerate(zip(ys, refs)):
            check_gemv(y.cpu().numpy().astype(np.float64), y_ref, a_ref, f"group {i} work={work_bytes}")
