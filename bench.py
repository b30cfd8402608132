"""Benchmark: fused entropy decode + GEMV per token on the Llama-3.1-8B-shaped linear stack.

One step = one token of single-stream decoding through all 224 linear layers of a
32-layer Llama-3.1-8B-shaped stack (q, k, v, o, gate, up, down per layer), batch 1,
Huffman-exponent coded weights, four grouped launches per layer (q/k/v, o,
gate/up, down) captured in one CUDA graph.  Weights are synthetic (seeded,
Llama-shaped distributions); the compressed stack (~9.4 GB) is far larger than L2,
so every step streams it from HBM.

Printed: one JSON line (rank 0).  `value` is microseconds per token (lower is
better); `roofline` is the fused GEMV kernel's achieved compressed-stream GB/s
against the measured HBM copy peak; `e2e` adds the host<->device copies of the
step's activations and outputs; `cpu_baseline` is the CPU oracle on a bounded
sample.  `--impl reference` times the CPU oracle instead (the reference arm).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--no-extras]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused decode+GEMV us/token & compressed-stream HBM GB/s (% of GB300 peak)"
WORKLOAD = "llama-3.1-8b linear stack, 32 layers x (q,k,v,o,gate,up,down), batch 1, Huffman-exponent BF16"
KERNEL_SRC = os.path.join(ROOT, "lossless_entropy_coded_gb300", "csrc", "ec_kernels.cu")
PROFILE = os.path.join(ROOT, "profiles", "huff_gemv_8b_stack.md")


# ------------------------------------------------------------------ helpers
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_hash() -> str:
    """First 16 hex digits of the SHA-256 of the kernel source without the sections
    that the batch-1 Huffman GEMV never runs (the text between each "<tag>: begin" /
    "<tag>: end" marker pair: the E8, rANS, FP8, exponent-codec, tensor-core and
    prefill code): the fused GEMV's counters stay valid while only that code changes."""
    with open(KERNEL_SRC, "rb") as f:
        src = f.read()
    src = re.sub(rb"/\* ---- ([A-Za-z0-9 ]+): begin ---- \*/.*?/\* ---- \1: end ---- \*/\n", b"", src, flags=re.S)
    return hashlib.sha256(src).hexdigest()[:16]


def profiled_traffic():
    """Per-launch DRAM bytes of the fused GEMV kernel from the committed ncu summary,
    only if it was taken on the current kernel source."""
    if not os.path.exists(PROFILE):
        return None
    txt = open(PROFILE).read()
    m = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", txt)
    t = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if not m or not t or m.group(1) != kernel_hash():
        return None
    return float(t.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu, self.rows, self.proc = gpu, [], None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([c.strip() for c in line.split(",")])

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in self.rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


# ------------------------------------------------------------------ the stack
class Stack:
    """Per-layer compressed matrices, activations and outputs of the 8B stack."""

    GROUPS = [("qkv", ["q", "k", "v"]), ("o", ["o"]), ("gu", ["gate", "up"]), ("down", ["down"])]

    def __init__(self, n_layers: int, keep_bf16: bool, device: int):
        import torch

        import lossless_entropy_coded_gb300 as ec
        import synth
        self.ec, self.torch = ec, torch
        self.n_layers = n_layers
        self.mats, self.bf16, self.specs = [], [], []
        self.x_host, self.y_dev = [], []
        x_parts, y_sizes = [], []
        self.compressed_bytes = 0
        self.weights = 0
        t0 = time.time()
        for l in range(n_layers):
            specs = {s.name.split(".")[1]: s for s in synth.layer_8b(l)}
            layer, layer_bf16 = {}, {}
            for nm, s in specs.items():
                w = synth.make_weights(s)
                W = ec.encode_bf16(w, device=device)
                layer[nm] = W
                self.compressed_bytes += W.stats()["device_bytes"]
                self.weights += w.size
                if keep_bf16:
                    layer_bf16[nm] = torch.from_numpy(w.view(np.int16)).to(f"cuda:{device}")
                del w
            self.mats.append(layer)
            self.bf16.append(layer_bf16)
            self.specs.append(specs)
            for g, names in self.GROUPS:
                k = specs[names[0]].k_cols
                x_parts.append(synth.make_x(specs[names[0]].seed, 1, k).ravel())
                y_sizes.extend(specs[n].n_rows for n in names)
        self.encode_s = time.time() - t0
        # one contiguous activation buffer and one output buffer (for the e2e copies)
        xs = np.concatenate(x_parts)
        self.x_pinned = torch.from_numpy(xs.view(np.int16)).pin_memory()
        self.x_dev = self.x_pinned.to(f"cuda:{device}")
        self.y_total = int(sum(y_sizes))
        self.y_dev_all = torch.zeros(self.y_total, dtype=torch.float32, device=f"cuda:{device}")
        self.y_pinned = torch.zeros(self.y_total, dtype=torch.float32).pin_memory()
        # views per launch
        self.calls = []
        xo = yo = 0
        for l in range(n_layers):
            for g, names in self.GROUPS:
                k = self.specs[l][names[0]].k_cols
                xv = self.x_dev[xo:xo + k]
                xo += k
                ys = []
                for n in names:
                    r = self.specs[l][n].n_rows
                    ys.append(self.y_dev_all[yo:yo + r])
                    yo += r
                self.calls.append(([self.mats[l][n] for n in names], xv, ys, [self.bf16[l].get(n) for n in names]))
        self.algo_bytes = self.compressed_bytes + 2 * xs.size + 4 * self.y_total

    def run_ec(self, batch_x=None):
        for Ws, x, ys, _ in self.calls:
            self.ec.gemv_group(Ws, x, ys, batch=1)

    def run_bf16_own(self):
        for Ws, x, ys, ws in self.calls:
            for w, y in zip(ws, ys):
                self.ec.bf16_gemv(w, x, y, batch=1)

    def run_cublas(self):
        F = self.torch.nn.functional
        bf = self.torch.bfloat16
        for Ws, x, ys, ws in self.calls:
            xb = x.view(bf).view(1, -1)
            for w, y in zip(ws, ys):
                y.copy_(F.linear(xb, w.view(bf)).view(-1))


def capture(torch, fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()  # first call outside capture: one-time attribute setup
    stream.synchronize()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
        fn()
    return g


def time_graph(torch, g, stream, steps, warmup, pre=None, post=None):
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            if pre:
                pre()
            g.replay()
            if post:
                post()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            if pre:
                pre()
            g.replay()
            if post:
                post()
        e1.record(stream)
        stream.synchronize()
    return e0.elapsed_time(e1) / steps * 1e3  # us per step


def group_us(torch, stack, stream, steps, warmup):
    """Microseconds per launch of each launch group (q/k/v, o, gate/up, down): the
    group's launches of every layer captured as one CUDA graph and replayed, so that
    consecutive launches overlap as they do in the token's graph."""
    out = {}
    for gi, (gname, _) in enumerate(Stack.GROUPS):
        calls = stack.calls[gi::len(Stack.GROUPS)]

        def run(calls=calls):
            for Ws, x, ys, _ in calls:
                stack.ec.gemv_group(Ws, x, ys, batch=1)
        g = capture(torch, run, stream)
        out[gname] = time_graph(torch, g, stream, steps, warmup) / len(calls)
    return out


# ------------------------------------------------------------------ CPU oracle sample
class OracleSample:
    """CPU oracle (DFloat11 two-phase decode + FP64 GEMV) on all seven matrices of
    layer 0 of the stack, cut into independent blocks of 1024 rows (each encoded on
    its own, outside the timed part) that a thread pool runs on every host core (the
    oracle's C calls release the GIL).  One pass is 1/32 of a token's weights; its
    time is scaled to one token (224 matrices)."""

    def __init__(self):
        import oracle as O
        import synth
        self.O = O
        self.cores = os.cpu_count() or 1
        self.jobs = []
        self.weights = 0
        specs = synth.layer_8b(0)
        for s in specs:
            w = synth.make_weights(s)
            x = synth.make_x(s.seed, 1, s.k_cols)
            for r0 in range(0, s.n_rows, 1024):
                wb = np.ascontiguousarray(w[r0:r0 + 1024])
                self.jobs.append((O.DF11(wb), wb.shape, x))
                self.weights += wb.size
        self.token_weights = sum(s.n_rows * s.k_cols for s in specs) * synth.N_LAYERS_8B

    def run(self, pool):
        """One timed pass on the pool; returns (us_per_token, seconds)."""
        t0 = time.perf_counter()
        list(pool.map(lambda j: self.O.gemv_bf16(j[0].decode().reshape(j[1]), j[2]), self.jobs))
        dt = time.perf_counter() - t0
        return dt / self.weights * self.token_weights * 1e6, dt

    def describe(self, dt):
        return (f"oracle on {self.cores} host cores: DF11 decode + FP64 GEMV of all 7 layer-0 matrices "
                f"({self.weights} weights in {len(self.jobs)} blocks of 1024 rows, {dt:.2f} s a pass), "
                f"scaled x{self.token_weights / self.weights:.1f} to the {self.token_weights} weights of one token")


def oracle_timings():
    """The oracle on configs 1, 2 and 4 (the 1024x1024 matrix, the 8B layer set, one
    rANS shape): decode + FP64 GEMV, timed single-threaded and on all host cores.
    The work is cut into independent row blocks of 1024 rows, each encoded on its
    own outside the timed part; all cores run the blocks in a thread pool (the
    oracle's C calls release the GIL), single-threaded runs them in order."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle as O
    import synth
    cores = os.cpu_count() or 1

    def blocks_bf16(specs):
        jobs = []
        for s in specs:
            w = synth.make_weights(s)
            x = synth.make_x(s.seed, 1, s.k_cols)
            for r0 in range(0, s.n_rows, 1024):
                wb = np.ascontiguousarray(w[r0:r0 + 1024])
                d = O.DF11(wb)
                jobs.append(lambda d=d, shape=wb.shape, x=x: O.gemv_bf16(d.decode().reshape(shape), x))
        return jobs

    def blocks_rans(idx):
        codes, scales = synth.make_rans_case(idx)
        n, k = codes.shape
        x = synth.make_x(4000 + idx, 1, k)
        jobs = []
        for r0 in range(0, n, 1024):
            cb, sb = np.ascontiguousarray(codes[r0:r0 + 1024]), np.ascontiguousarray(scales[r0:r0 + 1024])
            rc = O.Rans(cb)
            jobs.append(lambda rc=rc, cb=cb, sb=sb, x=x: (rc.decode(), O.gemv_rans(cb, sb, x)))
        return jobs

    out = {"cores": cores, "unit": "s", "blocks": "1024 rows, encoded outside the timed part"}
    for name, make in (("config1_1024x1024", lambda: blocks_bf16([synth.single_1024()])),
                       ("config2_8b_layer_set", lambda: blocks_bf16(synth.layer_8b())),
                       ("config4_rans_14336x4096", lambda: blocks_rans(0))):
        jobs = make()
        t0 = time.perf_counter()
        for j in jobs:
            j()
        single = time.perf_counter() - t0
        t0 = time.perf_counter()
        with ThreadPoolExecutor(cores) as ex:
            list(ex.map(lambda j: j(), jobs))
        allc = time.perf_counter() - t0
        out[name] = {"single_thread_s": round(single, 3), "all_cores_s": round(allc, 3)}
    return out


def run_reference(args):
    """The reference arm: the oracle, as it stands, on the host cores.  A step is one
    pass over the layer-0 sample (1/32 of a token); `value` is that pass scaled to one
    token, so it is extrapolated, and ms_per_step is the measured pass."""
    from concurrent.futures import ThreadPoolExecutor
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    t0 = time.time()
    sample = OracleSample()
    with ThreadPoolExecutor(sample.cores) as pool:
        for _ in range(args.warmup):
            sample.run(pool)
        dts = [sample.run(pool)[1] for _ in range(args.steps)]
    dt = float(np.mean(dts))
    value = dt / sample.weights * sample.token_weights * 1e6
    desc = sample.describe(dt)
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "us/token", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "value_extrapolated": f"a step is one pass over 1/{sample.token_weights / sample.weights:.0f} of a token's "
                                  "weights; value scales the mean pass to one token",
            "config": {"workload": WORKLOAD, "global_batch": 1, "matrices": 224},
            "cpu_baseline": {"value": round(value, 1), "unit": "us/token", "cores": sample.cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 1), "unit": "us/token", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": round(time.time() - t0, 1)}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ extras
def extras(torch, ec, stream, device):
    """Secondary measurements: config 1 latency, rANS shapes, E8 decode, 70B-block decode."""
    import synth
    out = {}
    dev = f"cuda:{device}"

    def t_loop(fn, iters=50, warm=5):
        with torch.cuda.stream(stream):
            for _ in range(warm):
                fn()
            stream.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(iters):
                fn()
            b.record(stream)
            stream.synchronize()
        return a.elapsed_time(b) / iters * 1e3

    # config 1: 1024x1024, latency-bound
    spec = synth.single_1024()
    w = synth.make_weights(spec)
    W = ec.encode_bf16(w, device=device)
    x = torch.from_numpy(synth.make_x(spec.seed, 1, 1024).view(np.int16)).to(dev)
    y = torch.empty((1, 1024), device=dev)
    g = capture(torch, lambda: ec.gemv(W, x, y), stream)
    out["w1024_gemv_us"] = round(t_loop(g.replay, 200), 2)
    dw = torch.empty((1024, 1024), dtype=torch.int16, device=dev)
    g2 = capture(torch, lambda: ec.decode(W, dw), stream)
    out["w1024_decode_us"] = round(t_loop(g2.replay, 200), 2)
    out["w1024_bpw"] = round(W.stats()["bits_per_weight"], 3)
    # the same matrix with codewords up to 24 bits (the limit the workload states):
    # window records carry what the 12-bit pair window cannot
    W24 = ec.encode_bf16(w, max_code_len=24, device=device)
    g3 = capture(torch, lambda: ec.gemv(W24, x, y), stream)
    out["w1024_maxlen24_gemv_us"] = round(t_loop(g3.replay, 200), 2)
    g4 = capture(torch, lambda: ec.decode(W24, dw), stream)
    out["w1024_maxlen24_decode_us"] = round(t_loop(g4.replay, 200), 2)
    out["w1024_maxlen24_bpw"] = round(W24.stats()["bits_per_weight"], 3)
    out["w1024_maxlen24_longest_code"] = int(W24.code_lengths().max())

    # rANS 4-bit tiles, both shapes, one code per symbol and pair symbols (rotate 8
    # copies to stay out of L2)
    for idx, (n, k) in enumerate(synth.RANS_SHAPES):
        codes, scales = synth.make_rans_case(idx)
        xr = torch.from_numpy(synth.make_x(4000 + idx, 1, k).view(np.int16)).to(dev)
        yr = torch.empty((1, n), device=dev)
        for tup, tag in ((1, ""), (2, "_pair")):
            blob = ec.encode_rans(codes, scales, device=-1, codes_per_symbol=tup).serialize()
            Rs = [ec.deserialize(blob, device=device) for _ in range(8)]
            st = Rs[0].stats()

            def rg():
                for R in Rs:
                    ec.gemv(R, xr, yr)
            gr = capture(torch, rg, stream)
            us = t_loop(gr.replay, 20) / len(Rs)
            out[f"rans{tag}_{n}x{k}_gemv_us"] = round(us, 2)
            out[f"rans{tag}_{n}x{k}_bpw"] = round(st["bits_per_weight"], 3)
            out[f"rans{tag}_{n}x{k}_gbs"] = round(st["device_bytes"] / us / 1e3, 1)
            del Rs, gr

    # E8 lattice points at about 4 bits per weight, 14336 x 4096: decode (17-table
    # rANS tiles + reconstruction) to BF16, four copies rotated to stay out of L2
    n8, k8 = 14336, 4096
    q2, r8, s8 = synth.make_e8_case(7500, n8, k8)
    blob = ec.encode_e8(q2, r8, s8, device=-1).serialize()
    Es = [ec.deserialize(blob, device=device) for _ in range(4)]
    de = torch.empty((n8, k8), dtype=torch.int16, device=dev)

    def e8d():
        for E in Es:
            ec.decode(E, de)
    ge = capture(torch, e8d, stream)
    us = t_loop(ge.replay, 20) / len(Es)
    st = Es[0].stats()
    out["e8_14336x4096_decode_us"] = round(us, 2)
    out["e8_14336x4096_bpw"] = round(st["bits_per_weight"], 3)
    out["e8_14336x4096_decode_in_gbs"] = round(st["device_bytes"] / us / 1e3, 1)
    out["e8_14336x4096_decode_hbm_gbs"] = round((st["device_bytes"] + 2 * n8 * k8) / us / 1e3, 1)
    out["e8_14336x4096_weights_per_s"] = float(f"{n8 * k8 / us * 1e6:.4g}")
    d8 = torch.empty((n8, k8), dtype=torch.uint8, device=dev)

    def e8f():
        for E in Es:
            ec.decode_as(E, d8, "e4m3")
    gf = capture(torch, e8f, stream)
    out["e8_14336x4096_decode_e4m3_us"] = round(t_loop(gf.replay, 20) / len(Es), 2)
    del Es, ge, gf, de, d8, q2

    # FP8 E4M3 weights, 14336 x 4096, batch-1 GEMV with every code in the table and
    # with a 32-code table plus correction records (8 copies rotated)
    cf, rf = synth.make_fp8_case(7600, 14336, 4096)
    xf = torch.from_numpy(synth.make_x(7601, 1, 4096).view(np.int16)).to(dev)
    yf = torch.empty((1, 14336), device=dev)
    for t, tag in ((0, "all"), (32, "t32")):
        blob = ec.encode_fp8(cf, rf, top_t=t, device=-1).serialize()
        Fs = [ec.deserialize(blob, device=device) for _ in range(8)]
        st = Fs[0].stats()

        def fg():
            for F in Fs:
                ec.gemv(F, xf, yf)
        gg = capture(torch, fg, stream)
        us = t_loop(gg.replay, 20) / len(Fs)
        out[f"fp8_{tag}_14336x4096_gemv_us"] = round(us, 2)
        out[f"fp8_{tag}_14336x4096_bpw"] = round(st["bits_per_weight"], 3)
        out[f"fp8_{tag}_14336x4096_gbs"] = round(st["device_bytes"] / us / 1e3, 1)
        del Fs, gg
    del cf

    # 70B-shaped block: one batched decode of all seven matrices to BF16
    Ws, outs, comp, nw = [], [], 0, 0
    for s in synth.block_70b():
        w = synth.make_weights(s)
        Wm = ec.encode_bf16(w, device=device)
        Ws.append(Wm)
        comp += Wm.stats()["device_bytes"]
        nw += w.size
        outs.append(torch.empty((s.n_rows, s.k_cols), dtype=torch.int16, device=dev))
        del w
    gd = capture(torch, lambda: ec.decode_batch(Ws, outs), stream)
    us = t_loop(gd.replay, 10, 2)
    out["block70b_decode_us"] = round(us, 1)
    out["block70b_decode_in_gbs"] = round(comp / us / 1e3, 1)
    out["block70b_decode_weights_per_s"] = float(f"{nw / us * 1e6:.4g}")
    out["block70b_decode_hbm_gbs"] = round((comp + 2 * nw) / us / 1e3, 1)
    assert ec.status() == 0
    return out


def batch_sweep(torch, ec, stack, stream, device):
    """Fused GEMV over the 8B layer set at batch 1 .. 64 (layers 0 and 1 of the stack
    alternately, 600 MB, so repeated replays do not run from L2), with the kernel
    family the library picks at each batch (CUDA cores, or from batch 6 the tensor
    cores), the same layer set coded with the 24-bit length limit at batch 1, and
    the same layer set through the rANS exponent codec at batch 1."""
    import synth
    dev = f"cuda:{device}"
    n_l = min(2, stack.n_layers)
    out = {}

    def t_graph(fn, iters=20, warm=3):
        g = capture(torch, fn, stream)
        return time_graph(torch, g, stream, iters, warm)

    sweep, paths = {}, {}
    for b in (1, 2, 4, 8, 16, 32, 64):
        paths[str(b)] = ec.gemv_path([stack.mats[0][n] for n in Stack.GROUPS[0][1]], b)
        bufs = []
        for l in range(n_l):
            for gname, names in Stack.GROUPS:
                Ws = [stack.mats[l][n] for n in names]
                k = stack.specs[l][names[0]].k_cols
                x = torch.from_numpy(synth.make_x(stack.specs[l][names[0]].seed, b, k).view(np.int16)).to(dev)
                ys = [torch.empty((b, stack.specs[l][n].n_rows), device=dev) for n in names]
                bufs.append((Ws, x, ys))

        def run(bufs=bufs, b=b):
            for Ws, x, ys in bufs:
                ec.gemv_group(Ws, x, ys, batch=b)
        sweep[str(b)] = round(t_graph(run) / n_l, 1)
    out["batch_sweep_us_per_layer_set"] = sweep
    out["batch_sweep_kernels"] = paths

    # materialisation for larger batches: decode each layer's matrices to BF16
    # (one ec_decode_batch launch per layer) and multiply with cuBLAS, against
    # cuBLAS on the uncompressed BF16 weights; per layer set
    F, bf = torch.nn.functional, torch.bfloat16
    dec = [{n: torch.empty((s.n_rows, s.k_cols), dtype=torch.int16, device=dev) for n, s in stack.specs[l].items()}
           for l in range(n_l)]
    mat, ref, gem, own = {}, {}, {}, {}
    for b in (16, 64, 256):
        xs = {}
        for l in range(n_l):
            for gname, names in Stack.GROUPS:
                k = stack.specs[l][names[0]].k_cols
                xs[(l, gname)] = torch.randn((b, k), device=dev).to(bf)

        def run_mat(b=b, xs=xs):
            for l in range(n_l):
                names = list(stack.specs[l])
                ec.decode_batch([stack.mats[l][n] for n in names], [dec[l][n] for n in names])
                for gname, gn in Stack.GROUPS:
                    for n in gn:
                        F.linear(xs[(l, gname)], dec[l][n].view(bf))

        def run_ref(b=b, xs=xs):
            for l in range(n_l):
                for gname, gn in Stack.GROUPS:
                    for n in gn:
                        F.linear(xs[(l, gname)], stack.bf16[l][n].view(bf))
        # the library's prefill route (ec_gemm_group per layer: the layer decoded into
        # the work buffer in one launch, then the tcgen05 GEMMs) and that GEMM alone on
        # the uncompressed weights
        ys = {(l, n): torch.empty((b, s.n_rows), device=dev) for l in range(n_l) for n, s in stack.specs[l].items()}
        order = [(gname, n) for gname, gn in Stack.GROUPS for n in gn]
        wb = max(ec.gemm_group_work_bytes([stack.mats[l][n] for _, n in order], b) for l in range(n_l))
        work = torch.empty(wb, dtype=torch.uint8, device=dev)

        def run_gemm(b=b, xs=xs, ys=ys, work=work, order=order):
            for l in range(n_l):  # one ec_gemm_group per layer: the block decoded in one launch
                ec.gemm_group([stack.mats[l][n] for _, n in order],
                              [xs[(l, g)].view(torch.int16) for g, _ in order], [ys[(l, n)] for _, n in order], b,
                              work=work)

        def run_own(b=b, xs=xs, ys=ys, work=work):
            for l in range(n_l):
                for gname, gn in Stack.GROUPS:
                    for n in gn:
                        ec.bf16_gemm(stack.bf16[l][n], xs[(l, gname)].view(torch.int16), ys[(l, n)], b, work=work)
        mat[str(b)] = round(t_graph(run_mat) / n_l, 1)
        ref[str(b)] = round(t_graph(run_ref) / n_l, 1)
        gem[str(b)] = round(t_graph(run_gemm) / n_l, 1)
        own[str(b)] = round(t_graph(run_own) / n_l, 1)
        del work
    out["materialize_gemm_us_per_layer_set"] = mat
    out["bf16_cublas_gemm_us_per_layer_set"] = ref
    out["ec_gemm_us_per_layer_set"] = gem
    out["own_tcgen05_bf16_gemm_us_per_layer_set"] = own
    # the 24-bit limit (hierarchical-table kernel) on layer 0..n_l-1 at batch 1
    mats24, bufs = [], []
    for l in range(n_l):
        specs = stack.specs[l]
        m = {nm: ec.encode_bf16(synth.make_weights(s), max_code_len=24, device=device) for nm, s in specs.items()}
        mats24.append(m)
        for gname, names in Stack.GROUPS:
            k = specs[names[0]].k_cols
            x = torch.from_numpy(synth.make_x(specs[names[0]].seed, 1, k).view(np.int16)).to(dev)
            ys = [torch.empty((1, specs[n].n_rows), device=dev) for n in names]
            bufs.append(([m[n] for n in names], x, ys))

    def run24():
        for Ws, x, ys in bufs:
            ec.gemv_group(Ws, x, ys, batch=1)
    out["layer_set_us_maxlen24"] = round(t_graph(run24) / n_l, 1)
    out["layer_set_bpw_maxlen24"] = round(8 * sum(W.stats()["device_bytes"] for m in mats24 for W in m.values())
                                          / sum(s.n_rows * s.k_cols for l in range(n_l)
                                                for s in stack.specs[l].values()), 4)
    # the same layer set through the rANS exponent codec (pair symbols, table size by
    # the size bound) at batch 1, beside the Huffman walker
    mats_x, bufs = [], []
    for l in range(n_l):
        specs = stack.specs[l]
        m = {nm: ec.encode_bf16_exp(synth.make_weights(s), device=device) for nm, s in specs.items()}
        mats_x.append(m)
        for gname, names in Stack.GROUPS:
            k = specs[names[0]].k_cols
            x = torch.from_numpy(synth.make_x(specs[names[0]].seed, 1, k).view(np.int16)).to(dev)
            ys = [torch.empty((1, specs[n].n_rows), device=dev) for n in names]
            bufs.append(([m[n] for n in names], x, ys))

    def run_exp():
        for Ws, x, ys in bufs:
            ec.gemv_group(Ws, x, ys, batch=1)
    out["layer_set_us_rans_exponents"] = round(t_graph(run_exp) / n_l, 1)
    out["layer_set_bpw_rans_exponents"] = round(8 * sum(W.stats()["device_bytes"] for m in mats_x for W in m.values())
                                                / sum(s.n_rows * s.k_cols for l in range(n_l)
                                                      for s in stack.specs[l].values()), 4)
    assert ec.status(stream) == 0
    return out


def aggregate_ranks(torch, dist, us_local: float, world: int, device: str):
    """Replicas: every rank decodes its own token per step.  The step time is the
    slowest rank's (max over ranks); the whole job makes `world` tokens per step,
    so microseconds per token = step time / world."""
    t = torch.tensor([us_local], dtype=torch.float64, device=device)
    if dist is not None and world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    us_step = float(t.item())
    return us_step, us_step / world


# ------------------------------------------------------------------ main
PROFILE_CASES = ("gemm", "bf16_gemm", "exp", "rans_pair", "decode", "fp8_t32", "e8", "mma")


def profile_case(name: str, batch: int) -> None:
    """One library call on a named workload, three times, untimed: the command that
    the ncu summaries in profiles/ capture.  gemm: ec_gemm_group over layer 0 of the
    8B stack at `batch`; bf16_gemm: the tcgen05 GEMM on layer 0's gate matrix
    uncompressed; exp: the rANS exponent codec's GEMV on layer 0's gate matrix; rans_pair:
    the 4-bit pair-symbol GEMV on 14336 x 4096; decode: ec_decode_batch of layer 0;
    fp8_t32: the FP8 GEMV with a 32-code table on 14336 x 4096; e8: the E8 decode to
    BF16 of 14336 x 4096; mma: the tensor-core GEMV of layer 0's gate/up group at
    `batch` (6..64)."""
    import torch
    import lossless_entropy_coded_gb300 as ec
    import synth
    dev = "cuda:0"
    specs = synth.layer_8b(0)
    gate = [s for s in specs if s.name.endswith("gate")][0]

    def xs_of(k, b=batch):
        return torch.from_numpy(synth.make_x(k, b, k).view(np.int16)).to(dev)
    if name == "gemm":
        Ws = [ec.encode_bf16(synth.make_weights(s), device=0) for s in specs]
        xs = [xs_of(s.k_cols) for s in specs]
        ys = [torch.empty((batch, s.n_rows), device=dev) for s in specs]
        work = torch.empty(ec.gemm_group_work_bytes(Ws, batch), dtype=torch.uint8, device=dev)
        run = lambda: ec.gemm_group(Ws, xs, ys, batch, work=work)
    elif name == "bf16_gemm":
        w = torch.from_numpy(synth.make_weights(gate).view(np.int16)).to(dev)
        x, y = xs_of(gate.k_cols), torch.empty((batch, gate.n_rows), device=dev)
        work = torch.empty(64 << 20, dtype=torch.uint8, device=dev)
        run = lambda: ec.bf16_gemm(w, x, y, batch, work=work)
    elif name == "exp":
        W = ec.encode_bf16_exp(synth.make_weights(gate), device=0)
        x, y = xs_of(gate.k_cols, 1), torch.empty((1, gate.n_rows), device=dev)
        run = lambda: ec.gemv(W, x, y)
    elif name == "rans_pair":
        codes, scales = synth.make_rans_case(0)
        W = ec.encode_rans(codes, scales, codes_per_symbol=2, device=0)
        x, y = xs_of(codes.shape[1], 1), torch.empty((1, codes.shape[0]), device=dev)
        run = lambda: ec.gemv(W, x, y)
    elif name == "decode":
        Ws = [ec.encode_bf16(synth.make_weights(s), device=0) for s in specs]
        outs = [torch.empty((s.n_rows, s.k_cols), dtype=torch.int16, device=dev) for s in specs]
        run = lambda: ec.decode_batch(Ws, outs)
    elif name == "e8":
        q2, r8, s8 = synth.make_e8_case(7500, 14336, 4096)
        W = ec.encode_e8(q2, r8, s8, device=0)
        out = torch.empty((14336, 4096), dtype=torch.int16, device=dev)
        run = lambda: ec.decode_as(W, out, "bf16")
    elif name == "mma":
        gu = [s for s in specs if s.name.split(".")[1] in ("gate", "up")]
        Ws = [ec.encode_bf16(synth.make_weights(s), device=0) for s in gu]
        x = xs_of(gu[0].k_cols)
        ys = [torch.empty((batch, s.n_rows), device=dev) for s in gu]
        assert ec.gemv_path(Ws, batch) == "tensor_cores"
        run = lambda: ec.gemv_group(Ws, x, ys, batch=batch)
    else:
        codes, r = synth.make_fp8_case(8000, 14336, 4096)
        W = ec.encode_fp8(codes, r, top_t=32, device=0)
        x, y = xs_of(4096, 1), torch.empty((1, 14336), device=dev)
        run = lambda: ec.gemv(W, x, y)
    for _ in range(3):
        run()
    torch.cuda.synchronize()
    assert ec.status() == 0
    print(json.dumps({"case": name, "batch": batch, "status": "ok"}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=32)
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", choices=PROFILE_CASES, help="run one named workload untimed (for ncu) and exit")
    ap.add_argument("--batch", type=int, default=256, help="batch rows of --case gemm / bf16_gemm / mma")
    args = ap.parse_args()
    if args.case:
        return profile_case(args.case, args.batch)
    args.warmup = max(3, args.warmup)
    args.warmup_ref = 0
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    import lossless_entropy_coded_gb300 as ec

    t_setup = time.time()
    stack = Stack(args.layers, keep_bf16=True, device=local)
    stream = torch.cuda.Stream()
    g_ec = capture(torch, stack.run_ec, stream)
    g_bf = capture(torch, stack.run_bf16_own, stream)
    g_cb = capture(torch, stack.run_cublas, stream)
    assert ec.status(stream) == 0
    setup_s = time.time() - t_setup

    # correctness guard on a few outputs of the timed graph (against the BF16 path)
    g_ec.replay()
    stream.synchronize()
    y_ec = stack.y_dev_all.clone()
    g_bf.replay()
    stream.synchronize()
    rel = float(torch.linalg.norm(y_ec - stack.y_dev_all) / torch.linalg.norm(stack.y_dev_all))
    assert rel < 1e-4, f"fused GEMV disagrees with the BF16 GEMV (rel {rel})"

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        us_ec = time_graph(torch, g_ec, stream, args.steps, args.warmup)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
    clocks = clk.summary()
    us_bf = time_graph(torch, g_bf, stream, max(20, args.steps // 4), args.warmup)
    us_cb = time_graph(torch, g_cb, stream, max(20, args.steps // 4), args.warmup)
    # end to end: pinned host activations in, outputs back to pinned host memory
    us_e2e = time_graph(torch, g_ec, stream, max(20, args.steps // 4), args.warmup,
                        pre=lambda: stack.x_dev.copy_(stack.x_pinned, non_blocking=True),
                        post=lambda: stack.y_pinned.copy_(stack.y_dev_all, non_blocking=True))
    g_us = group_us(torch, stack, stream, max(10, args.steps // 10), args.warmup)
    assert ec.status(stream) == 0
    groups = {}
    for gname, names in Stack.GROUPS:
        us_g = g_us[gname]
        nbytes = sum(stack.mats[0][n].stats()["device_bytes"] for n in names)
        groups[gname] = {"us": round(us_g, 2), "compressed_gbs": round(nbytes / us_g / 1e3, 1)}

    us_step, value = aggregate_ranks(torch, dist if world > 1 else None, us_ec, world, "cuda")

    peak, peak_kind = peaks()
    # the timed graph holds only the fused GEMV kernel, len(stack.calls) launches a step:
    # its mean launch duration is the step time over the launches (consecutive launches
    # overlap their prologues, so a launch timed alone would take longer)
    per_launch_bytes = stack.algo_bytes / len(stack.calls)
    launch_us = us_ec / len(stack.calls)
    achieved = per_launch_bytes / (launch_us * 1e-6) / 1e9
    traffic = profiled_traffic()
    ex = {}
    if rank == 0 and not args.no_extras:
        ex = extras(torch, ec, stream, local)
        ex.update(batch_sweep(torch, ec, stack, stream, local))
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        from concurrent.futures import ThreadPoolExecutor
        sample = OracleSample()
        with ThreadPoolExecutor(sample.cores) as pool:
            sample.run(pool)
            runs = [sample.run(pool) for _ in range(3)]
        v, dt = float(np.median([r[0] for r in runs])), float(np.median([r[1] for r in runs]))
        cpu = {"value": round(v, 1), "unit": "us/token", "cores": sample.cores, "kind": "oracle",
               "sample": sample.describe(dt)}
        ex["oracle_timings"] = oracle_timings()

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "us/token", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us_step / 1e3, 4),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "global_batch": 1, "matrices": 224, "weights": stack.weights,
                       "compressed_bytes": stack.compressed_bytes,
                       "l2": "inputs larger than L2 (compressed stack >> 129 MB), no flush",
                       "launches_per_step": len(stack.calls), "cuda_graph": True},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic,
                         "kernel": "huff_gemv_kernel<1>", "peak_kind": peak_kind,
                         "bytes_per_launch": round(per_launch_bytes), "launch_us_mean": round(launch_us, 3),
                         "launch_us_from": "timed step / launches per step (the step's graph holds only this kernel)"},
            "cpu_baseline": cpu,
            "e2e": {"value": round(us_e2e / world, 2), "unit": "us/token",
                    "h2d_bytes_per_step": int(stack.x_pinned.numel() * 2),
                    "d2h_bytes_per_step": int(stack.y_total * 4)},
            "gpu_launches": len(stack.calls) * args.steps,
            "clocks": clocks,
            "detail": {
                "bf16_gemv_own_us_per_token": round(us_bf, 2),
                "bf16_cublas_us_per_token": round(us_cb, 2),
                "speedup_vs_own_bf16": round(us_bf / us_step, 3),
                "speedup_vs_cublas": round(us_cb / us_step, 3),
                "step_compressed_gbs": round(stack.compressed_bytes / us_step / 1e3, 1),
                "step_frac_of_peak": round(stack.compressed_bytes / us_step / 1e3 / peak, 4),
                "step_frac_of_8tbs": round(stack.compressed_bytes / us_step / 1e3 / 8000.0, 4),
                "bits_per_weight": round(8 * stack.compressed_bytes / stack.weights, 3),
                "effective_weights_per_s": float(f"{stack.weights / us_step * 1e6:.4g}"),
                "launch_groups": groups,
                "setup_s": round(setup_s, 1), "encode_s": round(stack.encode_s, 1),
                **ex,
            },
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
