"""GPU parity of the Huffman-exponent path against the oracle, through the C ABI.

Decoded weights must be bit-exact with the input (the oracle's DFloat11 decode
returns the input too, checked alongside); GEMV outputs must match the oracle's
FP64 GEMV within relative L2 <= 1e-3 and |err| <= 2e-3 * sum|w x| per element."""
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


def decode_gpu(ec, W, n, k):
    out = torch.full((n, k), -1, dtype=torch.int16, device="cuda")
    ec.decode(W, out)
    assert ec.status() == 0
    return out.cpu().numpy().view(np.uint16)


def gemv_gpu(ec, W, x, n):
    b = x.shape[0]
    y = torch.full((b, n), float("nan"), dtype=torch.float32, device="cuda")
    ec.gemv(W, dev(x.view(np.int16)), y, batch=b)
    assert ec.status() == 0
    return y.cpu().numpy()


def fib_weights(n_sym=30, rows=None):
    """A histogram with Fibonacci counts: the unconstrained code is 29 deep, so the
    24-bit limit binds and sub-table walks are exercised."""
    fib = [1, 1]
    while len(fib) < n_sym:
        fib.append(fib[-1] + fib[-2])
    e = np.concatenate([np.full(f, 100 + i) for i, f in enumerate(fib)])
    rng = np.random.default_rng(0)
    rng.shuffle(e)
    m = (rng.integers(0, 256, e.size)).astype(np.uint16)
    w = (e.astype(np.uint16) << 7) | (m & 0x7F) | ((m & 0x80) << 8)
    k = 4096
    r = w.size // k
    return w[: r * k].reshape(r, k)


def test_all_65536_patterns_round_trip(ec):
    w = np.arange(65536, dtype=np.uint16).reshape(256, 256)
    W = ec.encode_bf16(w)
    assert np.array_equal(decode_gpu(ec, W, 256, 256), w)


@pytest.mark.parametrize("shape", [(1, 1), (7, 13), (1, 4096), (4096, 1), (3, 300), (5, 1000), (33, 2049)])
@pytest.mark.parametrize("steps", [32, 128, 256])
def test_round_trip_ragged_shapes(ec, shape, steps):
    w = synth.llama_bf16(2100 + shape[0], *shape)
    W = ec.encode_bf16(w, tile_steps=steps)
    assert np.array_equal(decode_gpu(ec, W, *shape), w)


def test_round_trip_config1_and_oracle_agrees(ec):
    spec = synth.single_1024()
    w = synth.make_weights(spec)
    W = ec.encode_bf16(w)
    got = decode_gpu(ec, W, 1024, 1024)
    assert np.array_equal(got, w)
    assert np.array_equal(O.DF11(w).decode(), w.ravel())
    assert W.stats()["max_code_len"] == int(O.DF11(w, max_len=12).lengths.max())


@pytest.mark.parametrize("max_len", [24, 16, 12, 9])
def test_long_codes_and_length_limit(ec, max_len):
    w = fib_weights()
    W = ec.encode_bf16(w, max_code_len=max_len)
    assert W.code_lengths().max() == min(max_len, 24)
    assert np.array_equal(decode_gpu(ec, W, *w.shape), w)
    x = synth.make_x(77, 2, w.shape[1])
    y_ref, a_ref = O.gemv_bf16(w, x)
    check_gemv(gemv_gpu(ec, W, x, w.shape[0]), y_ref, a_ref, f"fib L={max_len}")


@pytest.mark.parametrize("shape", [(1024, 1024), (256, 4096), (96, 14336), (7, 13), (1, 1), (300, 1000)])
@pytest.mark.parametrize("batch", [1, 3, 16])
def test_gemv_parity(ec, shape, batch):
    w = synth.llama_bf16(2200 + shape[1], *shape)
    x = synth.make_x(2200, batch, shape[1])
    W = ec.encode_bf16(w)
    y_ref, a_ref = O.gemv_bf16(w, x)
    check_gemv(gemv_gpu(ec, W, x, shape[0]), y_ref, a_ref, f"{shape} b={batch}")


@pytest.mark.parametrize("shape,steps", [((48, 8192), 256), ((40, 14336), 224), ((33, 4096), 256), ((17, 5000), 240)])
@pytest.mark.parametrize("batch", [1, 3, 16])
def test_gemv_parity_large_tiles(ec, shape, steps, batch):
    """Tiles of up to 8192 weights: inside rows (x from tensor memory at batch 1), two
    rows per tile, and tiles that cross rows anywhere; window records past position
    4095 fold into their rows."""
    w = synth.llama_bf16(2250 + steps, *shape)
    x = synth.make_x(2250, batch, shape[1])
    W = ec.encode_bf16(w, tile_steps=steps, max_code_len=10)  # a short window: many records
    assert W.stats()["n_records"] > 0
    y_ref, a_ref = O.gemv_bf16(w, x)
    check_gemv(gemv_gpu(ec, W, x, shape[0]), y_ref, a_ref, f"{shape} steps={steps} b={batch}")
    assert np.array_equal(decode_gpu(ec, W, *shape), w)


def test_gemv_group_matches_individual(ec):
    shapes = [(512, 1024), (128, 1024), (128, 1024)]
    ws = [synth.llama_bf16(2300 + i, *s) for i, s in enumerate(shapes)]
    Ws = [ec.encode_bf16(w) for w in ws]
    x = synth.make_x(2300, 2, 1024)
    ys = [torch.full((2, s[0]), float("nan"), dtype=torch.float32, device="cuda") for s in shapes]
    ec.gemv_group(Ws, dev(x.view(np.int16)), ys, batch=2)
    assert ec.status() == 0
    for w, y in zip(ws, ys):
        y_ref, a_ref = O.gemv_bf16(w, x)
        check_gemv(y.cpu().numpy(), y_ref, a_ref, "group")


def test_decode_batch(ec):
    shapes = [(256, 1024), (64, 1024), (100, 700), (256, 3584)]
    ws = [synth.llama_bf16(2400 + i, *s) for i, s in enumerate(shapes)]
    Ws = [ec.encode_bf16(w) for w in ws]
    outs = [torch.zeros(s, dtype=torch.int16, device="cuda") for s in shapes]
    ec.decode_batch(Ws, outs)
    assert ec.status() == 0
    for w, o in zip(ws, outs):
        assert np.array_equal(o.cpu().numpy().view(np.uint16), w)


def test_full_size_8b_layer(ec):
    """All seven Llama-3.1-8B layer matrices at full size: bit-exact decode and the
    batch-1 GEMV against the oracle's FP64 GEMV (all rows)."""
    for spec in synth.layer_8b():
        w = synth.make_weights(spec)
        W = ec.encode_bf16(w)
        out = torch.empty((spec.n_rows, spec.k_cols), dtype=torch.int16, device="cuda")
        ec.decode(W, out)
        assert ec.status() == 0
        assert torch.equal(out, torch.from_numpy(w.view(np.int16)).cuda()), spec.name
        del out
        x = synth.make_x(spec.seed, 1, spec.k_cols)
        y_ref, a_ref = O.gemv_bf16(w, x)
        check_gemv(gemv_gpu(ec, W, x, spec.n_rows), y_ref, a_ref, spec.name)
        s = W.stats()
        # lane starts, alignment and offsets; window records (4 bytes each) besides
        assert (s["aux_bytes"] - 4 * s["n_records"]) * 8 / w.size < 0.25
        assert 4 * s["n_records"] * 8 / w.size < 0.2
        W.free()


@pytest.mark.parametrize("hier", [False, True])
def test_payload_corruption_is_reported_not_faulted(ec, hier):
    """Lane 3's codewords of tile 0 overwritten with ones: every lookup then decodes
    the all-ones codeword (the longest, 12 bits; the code is complete), so the lane
    runs far past the next lane's start and the walker must report EC_ERR_CORRUPT,
    for the decode and for the GEMV, without a fault."""
    w = synth.llama_bf16(2500, 64, 4096)
    W = ec.encode_bf16(w, hierarchical=hier)
    assert W.code_lengths().max() == 12
    blob = bytearray(W.serialize())
    from test_abi import parse, tile_layout, lane_starts
    h, devb = parse(bytes(blob))
    meta = len(blob) - len(devb)
    rec, S, _, _, area_off, _ = tile_layout(h, devb, 0)
    st = lane_starts(devb, rec)
    assert 8 * (st[4] - st[3]) < 12 * S  # the lane's true code is shorter than S ones-codewords
    for b in range(area_off + st[3], area_off + st[4]):
        blob[meta + b] = 0xFF
    Wc = ec.deserialize(bytes(blob), device=0)
    out = torch.zeros((64, 4096), dtype=torch.int16, device="cuda")
    ec.decode(Wc, out)
    assert ec.status() == -5
    x = synth.make_x(2500, 1, 4096)
    y = torch.zeros((1, 64), dtype=torch.float32, device="cuda")
    ec.gemv(Wc, dev(x.view(np.int16)), y, batch=1)
    assert ec.status() == -5
    # the context is still healthy and the clean matrix still decodes exactly
    assert np.array_equal(decode_gpu(ec, W, 64, 4096), w)


def test_empty_and_zero_k(ec):
    W = ec.encode_bf16(np.zeros((5, 0), np.uint16))
    y = torch.full((1, 5), 7.0, device="cuda")
    ec.gemv(W, torch.zeros(8, dtype=torch.int16, device="cuda"), y, batch=1)
    assert ec.status() == 0
    assert (y == 0).all()
    W0 = ec.encode_bf16(np.zeros((0, 64), np.uint16))
    ec.decode(W0, torch.zeros(8, dtype=torch.int16, device="cuda"))
    assert ec.status() == 0


def test_block_70b_decode_batch_is_bit_exact(ec):
    """One 70B-shaped decoder block (q, o 8192^2; k, v 1024x8192; gate, up
    28672x8192; down 8192x28672; 855.6 M weights) decoded to BF16 by a single
    ec_decode_batch launch, as timed by the bench: every weight equals the input."""
    Ws, outs, refs = [], [], []
    for s in synth.block_70b():
        w = synth.make_weights(s)
        Ws.append(ec.encode_bf16(w))
        refs.append(torch.from_numpy(w.view(np.int16)).cuda())
        outs.append(torch.empty((s.n_rows, s.k_cols), dtype=torch.int16, device="cuda"))
        del w
    ec.decode_batch(Ws, outs)
    assert ec.status() == 0
    for s, o, r in zip(synth.block_70b(), outs, refs):
        assert torch.equal(o, r), s.name


def test_full_size_layer_grouped_batch16_sampled_rows(ec):
    """The 8B layer set at batch 16 through the grouped launches the bench times
    (q/k/v, o, gate/up, down); 96 sampled rows of every matrix against the oracle's
    FP64 GEMV of those rows."""
    specs = {s.name.split(".")[-1]: s for s in synth.layer_8b()}
    groups = [["q", "k", "v"], ["o"], ["gate", "up"], ["down"]]
    rng = np.random.default_rng(7)
    for names in groups:
        ws = [synth.make_weights(specs[n]) for n in names]
        Ws = [ec.encode_bf16(w) for w in ws]
        x = synth.make_x(specs[names[0]].seed, 16, specs[names[0]].k_cols)
        ys = [torch.full((16, specs[n].n_rows), float("nan"), device="cuda") for n in names]
        ec.gemv_group(Ws, dev(x.view(np.int16)), ys, batch=16)
        assert ec.status() == 0
        for n, w, y in zip(names, ws, ys):
            rows = np.sort(rng.choice(w.shape[0], 96, replace=False))
            y_ref, a_ref = O.gemv_bf16(np.ascontiguousarray(w[rows]), x)
            check_gemv(y.cpu().numpy()[:, rows], y_ref, a_ref, f"{n} batch 16")
        for W in Ws:
            W.free()


def test_group_mixing_code_limits_uses_the_long_code_kernel(ec):
    """A group whose matrices have different length limits (24 with codewords
    longer than the pair window, and 12) runs as one launch of the kernel that
    walks the hierarchical table, with every matrix's result exact."""
    w_long = fib_weights()[:, :2048]
    w_a = synth.llama_bf16(2600, w_long.shape[0], 2048)
    Ws = [ec.encode_bf16(w_long, max_code_len=24), ec.encode_bf16(w_a)]
    assert Ws[0].code_lengths().max() > 12 and Ws[1].code_lengths().max() <= 12
    x = synth.make_x(2600, 3, 2048)
    ys = [torch.full((3, w_long.shape[0]), float("nan"), device="cuda") for _ in Ws]
    ec.gemv_group(Ws, dev(x.view(np.int16)), ys, batch=3)
    assert ec.status() == 0
    for w, y in zip((w_long, w_a), ys):
        y_ref, a_ref = O.gemv_bf16(w, x)
        check_gemv(y.cpu().numpy(), y_ref, a_ref, "mixed limits")


def test_decode_batch_mixes_rans_and_huffman(ec):
    w = synth.llama_bf16(2601, 96, 1536)
    codes, scales = synth.make_rans_case(0, 40, 1024)
    Ws = [ec.encode_bf16(w), ec.encode_rans(codes, scales)]
    outs = [torch.zeros((96, 1536), dtype=torch.int16, device="cuda"),
            torch.zeros((40, 1024), dtype=torch.int16, device="cuda")]
    ec.decode_batch(Ws, outs)
    assert ec.status() == 0
    assert np.array_equal(outs[0].cpu().numpy().view(np.uint16), w)
    assert np.array_equal(outs[1].cpu().numpy().view(np.uint16), O.rans_dequant_bf16(codes, scales))


def test_misaligned_device_pointers_are_rejected(ec):
    from lossless_entropy_coded_gb300 import _ec
    w = synth.llama_bf16(2602, 32, 1024)
    W = ec.encode_bf16(w)
    x = torch.zeros(1024 + 8, dtype=torch.int16, device="cuda")
    y = torch.zeros(32 + 4, dtype=torch.float32, device="cuda")
    lib = ec.lib
    assert lib.ec_gemv(W.handle, x.data_ptr() + 2, y.data_ptr(), 1, None) == _ec.EC_ERR_INVALID_ARG
    assert lib.ec_gemv(W.handle, x.data_ptr(), y.data_ptr() + 4, 1, None) == _ec.EC_ERR_INVALID_ARG
    out = torch.zeros(32 * 1024 + 8, dtype=torch.int16, device="cuda")
    assert lib.ec_decode(W.handle, out.data_ptr() + 2, None) == _ec.EC_ERR_INVALID_ARG
    assert ec.status() == 0


@pytest.mark.parametrize("batch", [1, 3])
def test_gemv_group_of_seven_matrices(ec, batch):
    """A group of seven matrices of one width in one launch (seven pair tables in
    shared memory): every output against the oracle."""
    shapes = [(256, 1024), (64, 1024), (96, 1024), (128, 1024), (33, 1024), (300, 1024), (7, 1024)]
    ws = [synth.llama_bf16(2350 + i, *sh) for i, sh in enumerate(shapes)]
    Ws = [ec.encode_bf16(w) for w in ws]
    x = synth.make_x(2350, batch, 1024)
    ys = [torch.full((batch, sh[0]), float("nan"), dtype=torch.float32, device="cuda") for sh in shapes]
    ec.gemv_group(Ws, torch.from_numpy(x.view(np.int16)).cuda(), ys, batch=batch)
    assert ec.status() == 0
    for i, (w, y) in enumerate(zip(ws, ys)):
        y_ref, a_ref = O.gemv_bf16(w, x)
        check_gemv(y.cpu().numpy().astype(np.float64), y_ref, a_ref, f"group member {i} b={batch}")
