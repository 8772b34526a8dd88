"""Benchmark: Llama-3.2-3B quantized linears on one GB300 (or N replicas).

One step = one pass of the hot path over one batch of seeded synthetic inputs:
  * prefill at M = 1024 tokens: fused gate/up + SwiGLU (Q4_K, K 3072, N_ff 8192),
    the Q6_K down projection (K 8192 -> 3072) and the Q6_K attn_v (3072 -> 1024);
  * decode at M = 1: the seven linears of one layer (q, k, o, gate, up in Q4_K;
    v, down in Q6_K).
Reported metric (``value``): prefill GEMM TFLOP/s at M = 1024 (2*M*N*K per
linear, dequant arithmetic not counted), with the decode GEMV HBM GB/s (packed
weight + activation + output bytes) alongside.  Inputs rotate over enough
copies that every step reads more than the 129 MB L2 from HBM.

--impl reference times the CPU oracle (the only reference implementation:
the pages publish no code) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from tests import synth  # noqa: E402

METRIC = "prefill GEMM TFLOP/s (% FP16 tensor peak) at M=1024; decode GEMV HBM GB/s"
PREFILL_M = 1024
N_COPIES = 3  # rotating input copies: ~3 x 230 MB per cycle, well above L2
CLOCK_SOAK_S = 0.5  # untimed replay of the step after the timed region, for the clock samples


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def prefill_linears():
    gate = synth.Linear("ffn_gate", synth.Q4K, synth.FFN, synth.HIDDEN)
    up = synth.Linear("ffn_up", synth.Q4K, synth.FFN, synth.HIDDEN)
    down = synth.Linear("ffn_down", synth.Q6K, synth.HIDDEN, synth.FFN)
    v = synth.Linear("attn_v", synth.Q6K, synth.KV_DIM, synth.HIDDEN)
    return gate, up, down, v


def prefill_flops():
    gate, up, down, v = prefill_linears()
    return 2.0 * PREFILL_M * (gate.N * gate.K + up.N * up.K + down.N * down.K + v.N * v.K)


def step_config(world):
    """The workload one step runs (the same for both arms)."""
    return {"workload": "llama-3.2-3b linears: prefill M=1024 (gate/up+SwiGLU Q4_K, down Q6_K, attn_v Q6_K)"
                        " + decode M=1 (one layer's 7 linears)",
            "prefill_tokens": PREFILL_M, "decode_tokens": 1, "replicas": world,
            "l2": "%d rotating input copies, %.0f MB read per step (> 129 MB L2)"
                  % (N_COPIES, (decode_bytes() + 51.5e6 + 28e6) / 1e6)}


def kernel_sources_sha(names):
    """Hash of the CUDA source files a kernel's device code is built from, to
    tell whether stored ncu counters of that kernel are current."""
    import hashlib
    h = hashlib.sha256()
    d = os.path.join(ROOT, "quantized_q4_matmul_gb300", "csrc")
    for name in sorted(names):
        with open(os.path.join(d, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def measured_traffic(key):
    """DRAM bytes per launch from an ncu capture (profiles/traffic.json), or None
    if there is none or the kernel's sources have changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(key)
    if not e or e.get("sources_sha256") != kernel_sources_sha(e.get("sources", [])):
        return None
    return e.get("bytes_per_launch")


def decode_linears():
    return synth.layer_linears(0)  # layer 0: down is Q6_K


def decode_bytes():
    tot = 0
    for lin in decode_linears():
        tot += synth.weight_bytes(lin.qtype, lin.N, lin.K) + 2 * lin.K + 4 * lin.N
    return tot


# ----------------------------------------------------------------------------
# Clock sampling during the timed region
# ----------------------------------------------------------------------------
class Clocks:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        # Raw samples (the bench line carries their summary); QK_CLOCKS_DIR
        # keeps them somewhere else than the temporary directory.
        import tempfile
        self.path = os.path.join(os.environ.get("QK_CLOCKS_DIR", tempfile.gettempdir()),
                                 "clocks_bench_%d.csv" % os.getpid())

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.QUERY,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm),
                "window": "every 100 ms over the timed steps and %.1f s of untimed replays of the same step "
                          "graphs right after them" % CLOCK_SOAK_S}


# ----------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample
# ----------------------------------------------------------------------------
_CPU_INPUTS = []


def _cpu_inputs():
    """The prefill step's inputs for the oracle (generated once per process)."""
    if not _CPU_INPUTS:
        rng = synth.rng_for(7, 1)
        gate, up, down, v = prefill_linears()
        _CPU_INPUTS.extend([synth.q4k_weights(rng, gate.N, gate.K), synth.q4k_weights(rng, up.N, up.K),
                            synth.q6k_weights(rng, down.N, down.K), synth.q6k_weights(rng, v.N, v.K),
                            synth.activations(rng, PREFILL_M, gate.K),
                            synth.swiglu_activations(rng, PREFILL_M, down.K)])
    return _CPU_INPUTS


def cpu_single_thread():
    """The oracle on one host thread over configs 0 and 1 in full: the attn_q
    matmul at M = 16 (0.30 GFLOP) and the decode layer's seven linears at M = 1
    (63.9 MB of weights), each timed once after a warm-up call."""
    import oracle
    rng = synth.rng_for(7, 2)
    n0 = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        q = synth.Linear("attn_q", synth.Q4K, synth.HIDDEN, synth.HIDDEN)
        W = synth.q4k_weights(rng, q.N, q.K)
        x = synth.activations(rng, 16, q.K)
        oracle.matmul(oracle.Q4K, W, x[:1], q.N, q.K, rows=np.arange(64))
        t0 = time.perf_counter()
        oracle.matmul(oracle.Q4K, W, x, q.N, q.K)
        t_q = time.perf_counter() - t0
        lins = synth.layer_linears(0)
        data = [(l, synth.weights(rng, l.qtype, l.N, l.K), synth.activations(rng, 1, l.K)) for l in lins]
        t0 = time.perf_counter()
        for l, W, x in data:
            oracle.matmul(oracle.Q4K if l.qtype == "q4k" else oracle.Q6K, W, x, l.N, l.K)
        t_d = time.perf_counter() - t0
    finally:
        oracle.set_num_threads(n0)
    dbytes = sum(synth.weight_bytes(l.qtype, l.N, l.K) + 2 * l.K + 4 * l.N for l in lins)
    return {"attn_q_m16": {"ms": 1e3 * t_q, "tflops": 2.0 * 16 * q.N * q.K / t_q / 1e12, "cores": 1,
                           "sample": "full problem (M=16, N=K=3072), fp64 oracle, 1 thread"},
            "decode_layer_m1": {"ms": 1e3 * t_d, "gbs": dbytes / t_d / 1e9, "cores": 1,
                                "sample": "one layer's 7 linears at M=1 in full, fp64 oracle, 1 thread"}}


def cpu_baseline(target_s: float = 12.0):
    """The oracle on host cores over a bounded sample of the prefill step: the
    same fraction f of the output features of each of its problems (gate/up +
    SwiGLU, down, attn_v at M=1024), f grown until one run takes at least half
    of `target_s` (a short run overestimates the time per feature: fixed costs
    dominate it)."""
    import oracle
    gate, up, down, v = prefill_linears()
    Wg, Wu, Wd, Wv, xg, xd = _cpu_inputs()

    def run(f):
        rg, rd, rv = (max(1, min(n, int(round(f * n)))) for n in (gate.N, down.N, v.N))
        t0 = time.perf_counter()
        oracle.gateup_swiglu(Wg, Wu, xg, gate.N, gate.K, rows=np.arange(rg))
        oracle.matmul(oracle.Q6K, Wd, xd, down.N, down.K, rows=np.arange(rd))
        oracle.matmul(oracle.Q6K, Wv, xg, v.N, v.K, rows=np.arange(rv))
        dt = max(time.perf_counter() - t0, 1e-3)
        flops = 2.0 * PREFILL_M * (2 * gate.K * rg + down.K * rd + v.K * rv)
        return dt, flops, (rg, rd, rv)

    f = 8.0 * oracle.num_threads() / gate.N
    while True:
        dt, flops, rows = run(f)
        if dt >= 0.5 * target_s or f >= 1.0:
            break
        f = min(1.0, max(2.0 * f, f * target_s / dt))
    reps = 1
    if dt < 0.5 * target_s:  # the whole step is shorter than the target: repeat it
        reps = max(1, int(round(target_s / dt)))
        dt, flops = 0.0, 0.0
        for _ in range(reps):
            d, fl, rows = run(f)
            dt += d
            flops += fl
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": "prefill step at M=1024, fraction %.3f of the output features of each problem "
                      "(gate/up+SwiGLU %d of %d, down %d of %d, attn_v %d of %d; fp64 oracle, %d threads), "
                      "%d run(s), %.1f s" % (f, rows[0], gate.N, rows[1], down.N, rows[2], v.N, oracle.num_threads(),
                                           reps, dt)}


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------
class Workload:
    """Device-resident inputs (N_COPIES rotating copies) and outputs of one step."""

    def __init__(self, torch, dev, seed=0):
        self.torch = torch
        self.dev = dev
        gate, up, down, v = prefill_linears()
        self.copies = []
        for c in range(N_COPIES):
            rng = synth.rng_for(seed, 100 + c)
            d = {}
            d["gate"] = torch.from_numpy(synth.q4k_weights(rng, gate.N, gate.K)).to(dev)
            d["up"] = torch.from_numpy(synth.q4k_weights(rng, up.N, up.K)).to(dev)
            d["down"] = torch.from_numpy(synth.q6k_weights(rng, down.N, down.K)).to(dev)
            d["v"] = torch.from_numpy(synth.q6k_weights(rng, v.N, v.K)).to(dev)
            d["x_gu"] = torch.from_numpy(synth.activations(rng, PREFILL_M, gate.K).view(np.uint16)).to(dev)
            d["x_down"] = torch.from_numpy(synth.swiglu_activations(rng, PREFILL_M, down.K).view(np.uint16)).to(dev)
            d["x_v"] = torch.from_numpy(synth.swiglu_activations(rng, PREFILL_M, v.K).view(np.uint16)).to(dev)
            dec = []
            for lin in decode_linears():
                Wd = torch.from_numpy(synth.weights(rng, lin.qtype, lin.N, lin.K)).to(dev)
                xd = torch.from_numpy(synth.activations(rng, 1, lin.K).view(np.uint16)).to(dev)
                dec.append((lin, Wd, xd))
            d["decode"] = dec
            self.copies.append(d)
        self.y_gu = torch.empty(PREFILL_M, gate.N, dtype=torch.float16, device=dev)
        self.y_down = torch.empty(PREFILL_M, down.N, dtype=torch.float32, device=dev)
        self.y_v = torch.empty(PREFILL_M, v.N, dtype=torch.float32, device=dev)
        self.y_dec = [torch.empty(1, lin.N, dtype=torch.float32, device=dev) for lin in decode_linears()]
        self.y_dec_gu = torch.empty(1, synth.FFN, dtype=torch.float16, device=dev)

    def prefill(self, qk, c, stream, part=None):
        """The prefill step's three GEMMs; `part` "gu" = the fused gate/up alone,
        "rest" = down and attn_v."""
        d = self.copies[c]
        gate, up, down, v = prefill_linears()
        if part in (None, "gu"):
            qk.qk_gateup_swiglu_q4k(d["gate"], d["up"], d["x_gu"], self.y_gu, PREFILL_M, gate.N, gate.K, stream)
        if part in (None, "rest"):
            qk.qk_matmul_q6k(d["down"], d["x_down"], self.y_down, PREFILL_M, down.N, down.K, stream)
            qk.qk_matmul_q6k(d["v"], d["x_v"], self.y_v, PREFILL_M, v.N, v.K, stream)
        return 3

    def decode(self, qk, c, stream, chain=False):
        """The seven M = 1 linears of one layer.  Default: as independent problems
        in one grouped launch (qk_matmul_batch).  With `chain`: with the layer's
        dependencies -- {q, k, v} (one grouped launch), then o, then the fused
        gate/up + SwiGLU, then down (four launches)."""
        d = self.copies[c]
        dec = d["decode"]
        probs = [dict(qtype=lin.qtype, blocks=Wd, x_f16=xd, y=y, M=1, N=lin.N, K=lin.K)
                 for (lin, Wd, xd), y in zip(dec, self.y_dec)]
        if not chain:
            qk.qk_matmul_batch(probs, stream)
            return 1
        qk.qk_matmul_batch(probs[0:3], stream)
        qk.qk_matmul_batch(probs[3:4], stream)
        (lg, Wg, xg), (lu, Wu, _) = dec[4], dec[5]
        qk.qk_gateup_swiglu_q4k(Wg, Wu, xg, self.y_dec_gu, 1, lg.N, lg.K, stream)
        qk.qk_matmul_batch(probs[6:7], stream)
        return 4


def chain_bytes():
    """Bytes moved by the chained decode layer (fused gate/up writes fp16)."""
    tot = 0
    for lin in decode_linears():
        tot += synth.weight_bytes(lin.qtype, lin.N, lin.K)
        if lin.name == "ffn_up":
            continue
        tot += 2 * lin.K + (2 if lin.name == "ffn_gate" else 4) * lin.N
    return tot


def dequant_bytes():
    """Bytes the dequant export moves for one layer's seven weight tensors:
    the packed blocks in, 4 bytes per weight out."""
    return sum(synth.weight_bytes(l.qtype, l.N, l.K) + 4 * l.N * l.K for l in decode_linears())


def measure_dequant(torch, qk, wl, stream, dev, reps):
    """The dequant export (bit-exact fp32 weights) of one layer's seven weight
    tensors, captured as one CUDA graph per rotating copy and timed with CUDA
    events around each replay (weights ~64 MB in, ~403 MB out: beyond L2)."""
    s = stream.cuda_stream
    lins = decode_linears()
    outs = [torch.empty(l.N * l.K, dtype=torch.float32, device=dev) for l in lins]
    fns = {"q4k": qk.qk_dequant_q4k, "q6k": qk.qk_dequant_q6k}

    def one(c):
        for (lin, Wd, _), out in zip(wl.copies[c]["decode"], outs):
            fns[lin.qtype](Wd, lin.N * lin.K // 256, out, s)
        return len(lins)

    with torch.cuda.stream(stream):
        for i in range(3):
            one(i % N_COPIES)
    qk.qk_get_device_status(s)
    torch.cuda.synchronize()
    graphs = []
    for c in range(N_COPIES):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
            one(c)
        graphs.append(g)
    ms = []
    with torch.cuda.stream(stream):
        for i in range(3 + reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graphs[i % N_COPIES].replay()
            e1.record(stream)
            e1.synchronize()
            if i >= 3:
                ms.append(e0.elapsed_time(e1))
    qk.qk_get_device_status(s)
    med = statistics.median(ms)
    nbytes = dequant_bytes()
    pk = peaks()
    gbs = nbytes / (med * 1e-3) / 1e9
    del graphs, outs
    return {"metric": "dequant export HBM GB/s", "value": gbs, "unit": "GB/s", "frac_of_hbm": gbs / pk["hbm_gbs"],
            "ms_per_layer": med, "bytes_per_layer": nbytes, "launches_per_layer": len(lins),
            "note": "qk_dequant_q4k/q6k over one layer's 7 weight tensors (packed in, fp32 out), "
                    "one CUDA graph per rotating copy, %d replays" % reps}


# ----------------------------------------------------------------------------
# Per-configuration measurements (each kernel timed alone, L2 flushed first)
# ----------------------------------------------------------------------------
L2_FLUSH_BYTES = 512 << 20  # written before every timed launch: more than the 129 MB L2


def stats(ms):
    """Median, p95 and spread of per-run times (ms)."""
    a = np.asarray(ms, dtype=np.float64)
    return {"median": float(np.median(a)), "p95": float(np.percentile(a, 95)), "min": float(a.min()),
            "max": float(a.max()), "runs": int(a.size)}


def roof(flops, nbytes, ms, pk):
    """Achieved rates and the fraction of the attainable rate min(peak, AI x BW)."""
    s = ms * 1e-3
    tflops, gbs = flops / s / 1e12, nbytes / s / 1e9
    ai = flops / nbytes
    att = min(pk["bf16_tflops"], ai * pk["hbm_gbs"] / 1e3)
    bound = "tensor" if att >= pk["bf16_tflops"] else "hbm"
    return {"tflops": tflops, "gbs": gbs, "intensity_flop_per_byte": ai, "bound": bound,
            "attainable_tflops": att, "frac_of_attainable": tflops / att}


def timed(torch, stream, fn, reps, flush):
    """CUDA-event time of fn() on `stream`, each run after an L2 flush: a write
    of the whole flush buffer, then a read of its first half, so that L2 holds
    clean lines (write-backs of a dirty L2 would otherwise load the timed
    kernel's first microseconds)."""
    ms = []
    half = flush[: flush.numel() // 2].view(torch.int32)
    with torch.cuda.stream(stream):
        for i in range(reps + 2):
            flush.fill_(i & 0xFF)
            half.sum()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            if i >= 2:
                ms.append(e0.elapsed_time(e1))
    return ms


L2_BYTES = 129 << 20


def graph_steady(torch, stream, fns, R, reps):
    """Per-call time of R calls (cycling over fns) captured in one CUDA graph,
    one sample per replay: launch gaps as a captured decode loop sees them."""
    with torch.cuda.stream(stream):
        for f in fns:
            f()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
        for i in range(R):
            fns[i % len(fns)]()
    ms = []
    with torch.cuda.stream(stream):
        for i in range(reps + 1):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            e1.synchronize()
            if i:
                ms.append(e0.elapsed_time(e1) / R)
    del g
    return ms


def lin_bytes(lin, M, gateup=False):
    """Packed weight bytes + fp16 x + output bytes of one linear at M tokens."""
    w = synth.weight_bytes(lin.qtype, lin.N, lin.K) * (2 if gateup else 1)
    return w + 2 * M * lin.K + (2 if gateup else 4) * M * lin.N


def device_weights(torch, gen, qtype, N, K, dev):
    """Seeded random blocks drawn on the device with the recipe of tests/synth.py
    (uniform quant and scale bytes, fp16 |N(0,1)|*1e-4 scales; Q6_K int8 scales
    uniform on -32..63), for the sweep's 1.9 GiB of weights."""
    nb = N * (K // 256)
    bb = 144 if qtype == "q4k" else 210
    blk = torch.randint(0, 256, (nb, bb), dtype=torch.uint8, device=dev, generator=gen)

    def f16(n):
        return (torch.randn(n, device=dev, generator=gen).abs() * 1e-4).half().view(torch.uint8).view(n, 2)

    if qtype == "q4k":
        blk[:, 0:2] = f16(nb)
        blk[:, 2:4] = f16(nb)
    else:
        blk[:, 192:208] = torch.randint(-32, 64, (nb, 16), dtype=torch.int8, device=dev, generator=gen).view(
            torch.uint8)
        blk[:, 208:210] = f16(nb)
    return blk.view(-1)


ATTN_L = 4096  # cached positions of the decode-step attention


def attention_inputs(torch, dev, M, pos0, L, seed):
    """q [M][24][128] and caches [8][L][128], fp16 N(0, 1), seeded."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    H, Hkv, Dh = synth.N_HEADS, synth.N_KV_HEADS, synth.HEAD_DIM
    q = torch.randn(M, H, Dh, device=dev, generator=gen).half()
    k = torch.randn(Hkv, L, Dh, device=dev, generator=gen).half()
    v = torch.randn(Hkv, L, Dh, device=dev, generator=gen).half()
    return q, k, v


def measure_attention(torch, qk, dev, stream, reps, entry):
    """GQA attention of the 3B model (24 query / 8 key-value heads, head dim
    128, scale 1/sqrt(128)): one decode step over ATTN_L cached positions
    (rotating caches larger than L2, CUDA graph) and a causal prefill of
    PREFILL_M tokens (CUDA graph)."""
    H, Hkv, Dh = synth.N_HEADS, synth.N_KV_HEADS, synth.HEAD_DIM
    s = stream.cuda_stream
    scale = 1.0 / np.sqrt(Dh)
    res = {}
    L = ATTN_L
    kvb = 2 * Hkv * L * Dh * 2
    nc = max(2, int(np.ceil(3 * L2_BYTES / kvb)))
    sets = [attention_inputs(torch, dev, 1, L - 1, L, 90 + i) for i in range(nc)]
    o = torch.empty(1, H, Dh, device=dev)
    ms = graph_steady(torch, stream, [lambda q=q, k=k, v=v: qk.qk_gqa_attention(q, k, v, o, 1, H, Hkv, Dh, L - 1, L, scale, s)
                                      for q, k, v in sets], 4 * nc, reps)
    res["decode_L%d" % L] = entry("attention decode L=%d" % L, 4.0 * H * Dh * L, kvb + H * Dh * 6, ms,
                                  "attn_decode_kernel (cluster split of the cache, tensor-core scores), "
                                  "%d steps per CUDA graph over %d caches" % (4 * nc, nc))
    del sets
    M = PREFILL_M
    q, k, v = attention_inputs(torch, dev, M, 0, M, 99)
    o = torch.empty(M, H, Dh, device=dev)
    ms = graph_steady(torch, stream, [lambda: qk.qk_gqa_attention(q, k, v, o, M, H, Hkv, Dh, 0, M, scale, s)], 8, reps)
    res["prefill_M%d" % M] = entry("attention prefill M=%d" % M, 4.0 * H * Dh * M * (M + 1) / 2,
                                   2 * M * H * Dh + 2 * 2 * Hkv * M * Dh + 4 * M * H * Dh, ms,
                                   "attn_prefill_tc_kernel (tcgen05: S, P and O in tensor memory; causal 128-query "
                                   "blocks), 8 per CUDA graph")
    res["note"] = ("flops count the causal dot products (4 * H * D per visible query-key pair); decode bytes = "
                   "the key and value cache read once")
    return res


def measure_configs(torch, qk, dev, stream, reps, pk, log=print):
    """Every workload configuration with its own roofline fraction:
    config 0 (attn_q M=16), config 1 (the decode layer: grouped, chained and per
    linear), config 2 (gate/up + SwiGLU M=1024), config 3 (down and attn_v
    M=1024, separately) and config 4 (every linear of the model plus the LM head
    at M in 1..2048)."""
    s = stream.cuda_stream
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    out = {}
    rng = synth.rng_for(0, 900)

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    def x16(M, K, swiglu=False):
        x = synth.swiglu_activations(rng, M, K) if swiglu else synth.activations(rng, M, K)
        return up(x.view(np.uint16))

    def entry(name, flops, nbytes, ms, kernel, extra=None):
        st = stats(ms)
        r = {"kernel": kernel, "ms": st, "flops": flops, "bytes": nbytes}
        r.update(roof(flops, nbytes, st["median"], pk))
        if extra:
            r.update(extra)
        log("  %-28s %8.4f ms  %8.1f GB/s  %7.1f TFLOP/s  %5.1f%% of attainable (%s)" % (
            name, st["median"], r["gbs"], r["tflops"], 100 * r["frac_of_attainable"], r["bound"]))
        return r

    fns = {"q4k": qk.qk_matmul_q4k, "q6k": qk.qk_matmul_q6k}

    def kernel_of(qtype, M, K, gateup=False):
        if qk.qk_uses_gemv(qtype, M, K, gateup):
            return "gemv_decode_kernel (decode GEMV)" if M == 1 else "gemv_decode_kernel (2..8 tokens in the MMA columns)"
        return "gemm_tc_kernel (tcgen05 GEMM)"

    # config 0: attn_q, M = 16
    q = synth.Linear("attn_q", synth.Q4K, synth.HIDDEN, synth.HIDDEN)
    W = up(synth.q4k_weights(rng, q.N, q.K))
    x = x16(16, q.K)
    y = torch.empty(16, q.N, dtype=torch.float32, device=dev)
    ms = timed(torch, stream, lambda: qk.qk_matmul_q4k(W, x, y, 16, q.N, q.K, s), reps, flush)
    out["attn_q_m16"] = entry("attn_q M=16", 2.0 * 16 * q.N * q.K, lin_bytes(q, 16), ms, kernel_of("q4k", 16, q.K))
    del W, x, y

    # config 1: one layer's seven linears at M = 1
    lins = synth.layer_linears(0)
    Ws = [up(synth.weights(rng, l.qtype, l.N, l.K)) for l in lins]
    xs = [x16(1, l.K) for l in lins]
    ys = [torch.empty(1, l.N, dtype=torch.float32, device=dev) for l in lins]
    y_gu = torch.empty(1, synth.FFN, dtype=torch.float16, device=dev)
    per = {}
    for l, W, x, y in zip(lins, Ws, xs, ys):
        ms = timed(torch, stream, lambda: fns[l.qtype](W, x, y, 1, l.N, l.K, s), reps, flush)
        per[l.name] = entry("decode " + l.name, 2.0 * l.N * l.K, lin_bytes(l, 1), ms, kernel_of(l.qtype, 1, l.K))
    probs = [dict(qtype=l.qtype, blocks=W, x_f16=x, y=y, M=1, N=l.N, K=l.K) for l, W, x, y in zip(lins, Ws, xs, ys)]
    layer_bytes = sum(lin_bytes(l, 1) for l in lins)
    layer_flops = sum(2.0 * l.N * l.K for l in lins)
    ms = timed(torch, stream, lambda: qk.qk_matmul_batch(probs, s), reps, flush)
    grouped = entry("decode layer, grouped", layer_flops, layer_bytes, ms, "gemv_decode_kernel, one launch")

    def chain():
        qk.qk_matmul_batch(probs[0:3], s)
        qk.qk_matmul_batch(probs[3:4], s)
        qk.qk_gateup_swiglu_q4k(Ws[4], Ws[5], xs[4], y_gu, 1, lins[4].N, lins[4].K, s)
        qk.qk_matmul_batch(probs[6:7], s)

    cbytes = layer_bytes - lin_bytes(lins[5], 1) - lin_bytes(lins[4], 1) + lin_bytes(lins[4], 1, gateup=True)
    ms = timed(torch, stream, chain, reps, flush)
    chained = entry("decode layer, chained", layer_flops, cbytes, ms,
                    "gemv_decode_kernel, 4 launches: {q,k,v} -> o -> gate/up+SwiGLU -> down")
    # Steady state: R layers back to back in one CUDA graph over copies of the
    # layer's weights that together exceed L2 (each layer reads its own copy),
    # as a captured decode loop runs them.
    ncopy = max(2, int(-(-2.5 * L2_BYTES // layer_bytes)))
    gen = torch.Generator(device=dev)
    gen.manual_seed(901)
    sets = [[dict(p, blocks=device_weights(torch, gen, l.qtype, l.N, l.K, dev)) for p, l in zip(probs, lins)]
            for _ in range(ncopy - 1)] + [probs]
    ups = [device_weights(torch, gen, "q4k", lins[5].N, lins[5].K, dev) for _ in range(ncopy - 1)] + [Ws[5]]

    def grouped_of(ps):
        return lambda: qk.qk_matmul_batch(ps, s)

    def chain_of(ps, wu):
        gu = [dict(ps[4], up_blocks=wu, y=y_gu)]

        def f():
            qk.qk_matmul_batch(ps[0:3], s)
            qk.qk_matmul_batch(ps[3:4], s)
            qk.qk_matmul_batch(gu, s)
            qk.qk_matmul_batch(ps[6:7], s)
        return f

    steady = {}
    for name, mk, nbytes in (("grouped", lambda ps, wu: grouped_of(ps), layer_bytes), ("chained", chain_of, cbytes)):
        ms = graph_steady(torch, stream, [mk(ps, wu) for ps, wu in zip(sets, ups)], 4 * ncopy, reps)
        steady[name] = entry("decode layer, %s, steady" % name, layer_flops, nbytes, ms,
                             "gemv_decode_kernel, %d layers per CUDA graph over %d weight copies (%d MB > L2)" % (
                                 4 * ncopy, ncopy, ncopy * layer_bytes >> 20))
    out["decode_layer_m1"] = {"grouped": grouped, "chained": chained, "per_linear": per, "steady": steady}

    # int8 activations (qk_matmul_batch_q8x) beside the fp16 path: the grouped
    # layer and the tied LM head (323 MB, more than L2), both as steady state
    q8 = {}
    ms = graph_steady(torch, stream, [lambda ps=ps: qk.qk_matmul_batch_q8x(
        [dict(p) for p in ps if "up_blocks" not in p], s) for ps in sets], 4 * ncopy, reps)
    q8["layer_grouped_steady"] = entry("decode layer, grouped, int8 x", layer_flops, layer_bytes, ms,
                                       "gemv_decode_kernel (int8 activations), one launch per layer")
    lm = synth.LM_HEAD
    Wl = device_weights(torch, gen, lm.qtype, lm.N, lm.K, dev)
    xl = x16(1, lm.K)
    yl = torch.empty(1, lm.N, dtype=torch.float32, device=dev)
    for name, call in (("lm_head_fp16", lambda: qk.qk_matmul_q6k(Wl, xl, yl, 1, lm.N, lm.K, s)),
                       ("lm_head_int8x", lambda: qk.qk_matmul_q8x_q6k(Wl, xl, yl, 1, lm.N, lm.K, s))):
        ms = graph_steady(torch, stream, [call], 8, reps)
        q8[name + "_steady"] = entry("LM head, %s, steady" % name.split("_")[-1], 2.0 * lm.N * lm.K,
                                     lin_bytes(lm, 1), ms, "gemv_decode_kernel, 8 launches per CUDA graph")
    out["decode_int8_activations"] = q8
    del Ws, xs, ys, probs, sets, ups, Wl

    out["attention"] = measure_attention(torch, qk, dev, stream, reps, entry)

    # config 2: fused gate/up + SwiGLU at M = 1024
    g = synth.Linear("ffn_gate", synth.Q4K, synth.FFN, synth.HIDDEN)
    Wg, Wu = up(synth.q4k_weights(rng, g.N, g.K)), up(synth.q4k_weights(rng, g.N, g.K))
    x = x16(PREFILL_M, g.K)
    y = torch.empty(PREFILL_M, g.N, dtype=torch.float16, device=dev)
    ms = timed(torch, stream, lambda: qk.qk_gateup_swiglu_q4k(Wg, Wu, x, y, PREFILL_M, g.N, g.K, s), reps, flush)
    out["prefill_gateup_swiglu_m1024"] = entry("gate/up+SwiGLU M=1024", 2.0 * 2 * PREFILL_M * g.N * g.K,
                                               lin_bytes(g, PREFILL_M, gateup=True), ms,
                                               kernel_of("q4k", PREFILL_M, g.K, True))
    del Wg, Wu, x, y

    # config 3: down (Q6_K, K 8192) and attn_v (Q6_K, 3072 -> 1024) at M = 1024, x = silu(z1) z2
    c3 = {}
    for l in (synth.Linear("ffn_down", synth.Q6K, synth.HIDDEN, synth.FFN),
              synth.Linear("attn_v", synth.Q6K, synth.KV_DIM, synth.HIDDEN)):
        W = up(synth.q6k_weights(rng, l.N, l.K))
        x = x16(PREFILL_M, l.K, swiglu=True)
        y = torch.empty(PREFILL_M, l.N, dtype=torch.float32, device=dev)
        ms = timed(torch, stream, lambda: qk.qk_matmul_q6k(W, x, y, PREFILL_M, l.N, l.K, s), reps, flush)
        c3[l.name] = entry(l.name + " M=1024", 2.0 * PREFILL_M * l.N * l.K, lin_bytes(l, PREFILL_M), ms,
                           kernel_of("q6k", PREFILL_M, l.K))
        del W, x, y
    out["prefill_down_v_m1024"] = c3
    del flush
    torch.cuda.empty_cache()

    # config 4: every linear of the 28 layers plus the LM head, one call each, at each M
    gen = torch.Generator(device=dev)
    gen.manual_seed(4)
    model = synth.model_linears()
    Wm = [device_weights(torch, gen, l.qtype, l.N, l.K, dev) for _, l in model]
    wbytes = sum(synth.weight_bytes(l.qtype, l.N, l.K) for _, l in model)
    sweep = {}
    for M in synth.SWEEP_M:
        xk = {K: x16(M, K) for K in sorted({l.K for _, l in model})}
        yn = {N: torch.empty(M, N, dtype=torch.float32, device=dev) for N in sorted({l.N for _, l in model})}

        def one_pass():
            for (_, l), W in zip(model, Wm):
                fns[l.qtype](W, xk[l.K], yn[l.N], M, l.N, l.K, s)

        # one pass = 197 launches captured in a CUDA graph (2 GB of weights, far
        # more than L2, so no flush is needed); the host's per-call cost would
        # otherwise set the time at small M
        ms = graph_steady(torch, stream, [one_pass], 1, max(3, reps // 2))
        flops = sum(2.0 * M * l.N * l.K for _, l in model)
        nbytes = sum(lin_bytes(l, M) for _, l in model)
        sweep[str(M)] = entry("model sweep M=%d" % M, flops, nbytes, ms,
                              "%s, %d launches per pass, one CUDA graph" % (kernel_of("q4k", M, 3072), len(model)),
                              {"weight_bytes": wbytes})
        if M == 1:
            # the decode step as an engine runs it: each layer's linears in one
            # grouped launch (qk_matmul_batch), the LM head on its own
            by_layer = {}
            ysl = {}  # one output per position in a layer: a grouped launch's outputs must not overlap
            for ((li, l), W) in zip(model, Wm):
                pos = len(by_layer.setdefault(li, []))
                y = ysl.setdefault((pos, l.N), torch.empty(1, l.N, dtype=torch.float32, device=dev))
                by_layer[li].append(dict(qtype=l.qtype, blocks=W, x_f16=xk[l.K], y=y, M=1, N=l.N, K=l.K))
            groups = [probs for _, probs in sorted(by_layer.items(), key=lambda kv: str(kv[0]))]

            def grouped_pass():
                for probs in groups:
                    qk.qk_matmul_batch(probs, s)

            ms = graph_steady(torch, stream, [grouped_pass], 1, max(3, reps // 2))
            sweep["1_grouped"] = entry("model sweep M=1, grouped", flops, nbytes, ms,
                                       "gemv_decode_kernel, %d grouped launches per pass, one CUDA graph" % len(groups),
                                       {"weight_bytes": wbytes})
        del xk, yn
    out["model_sweep"] = sweep
    out["note"] = ("each kernel timed alone with CUDA events; before every run L2 is flushed by a %d MB write "
                   "followed by a %d MB read (so it holds clean lines); the sweep's 1.9 GiB of weights exceed L2 "
                   "(one pass per run, 197 launches); attainable = min(bf16 peak, intensity x HBM)"
                   % (L2_FLUSH_BYTES >> 20, L2_FLUSH_BYTES >> 21))
    del Wm
    torch.cuda.empty_cache()
    return out


def run_gpu(args, rank, world, dist):
    import torch
    import quantized_q4_matmul_gb300 as qk

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    qk.lib()
    wl = Workload(torch, dev, seed=rank)
    stream = torch.cuda.Stream(device=dev)
    s = stream.cuda_stream
    pk = peaks()

    # Warm-up, then capture each part of each rotating copy as a CUDA graph so
    # the timed region measures the kernels, not host launch overhead.  The
    # prefill is two graphs (the fused gate/up, then down + attn_v) with an
    # event between them, which times the dominant kernel inside the step.
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            wl.prefill(qk, i % N_COPIES, s)
            wl.decode(qk, i % N_COPIES, s)
    qk.qk_get_device_status(s)
    torch.cuda.synchronize()
    g_gu, g_rest, g_dec, g_chain = [], [], [], []
    for c in range(N_COPIES):
        for graphs, fn in ((g_gu, lambda: wl.prefill(qk, c, s, "gu")), (g_rest, lambda: wl.prefill(qk, c, s, "rest")),
                           (g_dec, lambda: wl.decode(qk, c, s)),
                           (g_chain, lambda: wl.decode(qk, c, s, chain=True))):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
                fn()
            graphs.append(g)
    n_pre, n_dec = 3, 1
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            g_gu[i % N_COPIES].replay()
            g_rest[i % N_COPIES].replay()
            g_dec[i % N_COPIES].replay()
    torch.cuda.synchronize()

    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches = 0
    with Clocks(local) as clk:
        with torch.cuda.stream(stream):
            t_start.record(stream)
            for i in range(args.steps):
                evs[i][0].record(stream)
                g_gu[i % N_COPIES].replay()
                evs[i][3].record(stream)
                g_rest[i % N_COPIES].replay()
                evs[i][1].record(stream)
                g_dec[i % N_COPIES].replay()
                evs[i][2].record(stream)
                launches += n_pre + n_dec
            t_end.record(stream)
        t_end.synchronize()
        # nvidia-smi samples every 100 ms, far longer than the timed steps: the
        # same step graphs keep replaying (untimed, after t_end) for ~0.5 s so
        # that the samples see the GPU under this load.
        soak_end = time.perf_counter() + CLOCK_SOAK_S
        with torch.cuda.stream(stream):
            i = 0
            while time.perf_counter() < soak_end:
                for _ in range(16):
                    g_gu[i % N_COPIES].replay()
                    g_rest[i % N_COPIES].replay()
                    g_dec[i % N_COPIES].replay()
                    i += 1
                stream.synchronize()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    qk.qk_get_device_status(s)
    total_ms = t_start.elapsed_time(t_end)
    pre_ms = [e[0].elapsed_time(e[1]) for e in evs]
    gu_ms = [e[0].elapsed_time(e[3]) for e in evs]  # the fused gate/up launch inside the step
    dec_ms = [e[1].elapsed_time(e[2]) for e in evs]
    # The same seven GEMVs with the layer's dependency chain (reported alongside).
    chain_ms = []
    for i in range(args.steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            g_chain[i % N_COPIES].replay()
            e1.record(stream)
        e1.synchronize()
        chain_ms.append(e0.elapsed_time(e1))

    # End to end through the public API with host buffers: every step, the
    # prefill's inputs are copied in from pinned host memory and its outputs
    # copied back, inside the timed region.  Copies run on two copy streams and
    # overlap the GEMMs: each GEMM waits only for its own input's upload, and
    # each output's download starts when its GEMM is done.
    gate, up, down, v = prefill_linears()
    c0 = wl.copies[0]
    d_x = (c0["x_gu"], c0["x_down"], c0["x_v"])
    d_y = (wl.y_gu, wl.y_down, wl.y_v)
    h_x = [t.cpu().pin_memory() for t in d_x]
    h_y = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in d_y]
    h2d = sum(t.numel() * t.element_size() for t in h_x)
    d2h = sum(t.numel() * t.element_size() for t in h_y)
    calls = (lambda: qk.qk_gateup_swiglu_q4k(c0["gate"], c0["up"], c0["x_gu"], wl.y_gu, PREFILL_M, gate.N, gate.K, s),
             lambda: qk.qk_matmul_q6k(c0["down"], c0["x_down"], wl.y_down, PREFILL_M, down.N, down.K, s),
             lambda: qk.qk_matmul_q6k(c0["v"], c0["x_v"], wl.y_v, PREFILL_M, v.N, v.K, s))
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    e2e_pre = []
    torch.cuda.synchronize()
    for i in range(args.steps):
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev_x = [torch.cuda.Event() for _ in d_x]
        ev_y = [torch.cuda.Event() for _ in d_y]
        t0.record(stream)
        s_in.wait_event(t0)
        s_out.wait_event(t0)
        with torch.cuda.stream(s_in):
            for hx, dx, ev in zip(h_x, d_x, ev_x):
                dx.copy_(hx, non_blocking=True)
                ev.record(s_in)
        for call, evx, evy in zip(calls, ev_x, ev_y):
            stream.wait_event(evx)
            call()
            evy.record(stream)
        with torch.cuda.stream(s_out):
            for hy, dy, ev in zip(h_y, d_y, ev_y):
                s_out.wait_event(ev)
                hy.copy_(dy, non_blocking=True)
        stream.wait_stream(s_out)
        t1.record(stream)
        t1.synchronize()
        e2e_pre.append(t0.elapsed_time(t1))
    torch.cuda.synchronize()

    flops = prefill_flops()
    dbytes = decode_bytes()
    pre_med = statistics.median(pre_ms)
    dec_med = statistics.median(dec_ms)
    local_res = {
        "total_ms": total_ms, "pre_ms": pre_med, "dec_ms": dec_med, "gu_ms": statistics.median(gu_ms),
        "e2e_pre_ms": statistics.median(e2e_pre), "launches": launches, "clocks": clk.summary(),
        "chain_ms": statistics.median(chain_ms),
    }
    if dist is not None:
        allr = [None] * world
        dist.all_gather_object(allr, local_res)
    else:
        allr = [local_res]
    if rank != 0:
        return None
    max_total = max(r["total_ms"] for r in allr)
    max_pre = max(r["pre_ms"] for r in allr)
    max_dec = max(r["dec_ms"] for r in allr)
    tflops = world * flops / (max_pre * 1e-3) / 1e12
    dec_gbs = world * dbytes / (max_dec * 1e-3) / 1e9
    gu_flops = 2.0 * 2 * PREFILL_M * gate.N * gate.K
    gu_ms_med = local_res["gu_ms"]
    gu_ach = gu_flops / (gu_ms_med * 1e-3) / 1e12
    traffic = measured_traffic("gateup_swiglu_m1024")
    res = {
        "metric": METRIC,
        "value": tflops,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": max_total / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16 (q4_k/q6_k weights, fp32 accumulate)",
        "data": "synthetic (seeded Llama-3.2-3B-shaped Q4_K/Q6_K weights, fp16 N(0,1) activations)",
        "config": step_config(world),
        "frac_of_fp16_peak": tflops / world / pk["bf16_tflops"],
        "decode": {"metric": "decode GEMV HBM GB/s", "value": dec_gbs, "unit": "GB/s",
                   "frac_of_hbm": dec_gbs / world / pk["hbm_gbs"], "ms_per_layer": max_dec,
                   "bytes_per_layer": dbytes,
                   "note": "one layer's 7 GEMVs (M=1) as independent problems in one grouped launch",
                   "chained": {"value": chain_bytes() / (max(r["chain_ms"] for r in allr) * 1e-3) / 1e9,
                               "unit": "GB/s", "ms_per_layer": max(r["chain_ms"] for r in allr),
                               "note": "with the layer's dependencies: {q,k,v} -> o -> fused gate/up+SwiGLU -> down"}},
        "roofline": {"bound": "tensor", "kernel": "gemm_tc_kernel<Q4_K, gate/up+SwiGLU> M=1024 N=2x8192 K=3072",
                     "achieved": gu_ach, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": gu_ach / pk["bf16_tflops"], "traffic": traffic,
                     "peak_source": pk["source"] + " (cuBLAS bf16 burst; fp16 dense rate equals bf16)",
                     "timing": "median over the timed steps of CUDA events on the step's stream around the "
                               "gate/up launch (its own graph, between the step's other graphs)"},
        "e2e": {"value": flops / (statistics.median([r["e2e_pre_ms"] for r in allr]) * 1e-3) / 1e12,
                "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": sum(r["launches"] for r in allr),
        "clocks": local_res["clocks"],
    }
    # Every workload configuration timed alone (rank 0), after the step's
    # numbers are final.
    if not args.no_configs:
        res["configs"] = measure_configs(torch, qk, dev, stream, max(10, args.steps), pk,
                                         log=lambda m: print(m, file=sys.stderr))
    # The dequant export (not part of the step) last, on rank 0, after every
    # number above is final: whatever happens here only affects this field.
    try:
        res["dequant"] = measure_dequant(torch, qk, wl, stream, dev, max(5, args.steps))
    except Exception as e:  # noqa: BLE001 -- reported in the line, not fatal
        res["dequant"] = {"error": ("%s: %s" % (type(e).__name__, e))[:300]}
    return res


def run_reference(args, rank):
    if rank != 0:
        return None
    import oracle
    oracle.build()
    for _ in range(args.warmup):
        cpu_baseline(target_s=1.0)
    vals, ts = [], []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        r = cpu_baseline(target_s=float(os.environ.get("QK_REF_STEP_S", "10")))
        ts.append(time.perf_counter() - t0)
        vals.append(r["value"])
    v = statistics.median(vals)
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": 0, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(ts), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
        "config": step_config(1),
        "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": r["cores"], "kind": "oracle",
                         "sample": r["sample"]},
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_profile(args):
    """Run one call of the step five times on cuda:0 (a target for ncu -k ... -s 4 -c 1)."""
    import torch
    import quantized_q4_matmul_gb300 as qk
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    wl = Workload(torch, dev)
    stream = torch.cuda.Stream(device=dev)
    s = stream.cuda_stream
    gate, _, down, v = prefill_linears()
    d = wl.copies[0]
    calls = {
        "gateup": lambda: qk.qk_gateup_swiglu_q4k(d["gate"], d["up"], d["x_gu"], wl.y_gu, PREFILL_M, gate.N, gate.K, s),
        "down": lambda: qk.qk_matmul_q6k(d["down"], d["x_down"], wl.y_down, PREFILL_M, down.N, down.K, s),
        "v": lambda: qk.qk_matmul_q6k(d["v"], d["x_v"], wl.y_v, PREFILL_M, v.N, v.K, s),
        "decode": lambda: wl.decode(qk, 0, s),
    }
    if args.profile == "lmhead":
        gen = torch.Generator(device=dev)
        gen.manual_seed(5)
        lm = synth.LM_HEAD
        Wl = device_weights(torch, gen, lm.qtype, lm.N, lm.K, dev)
        xl = torch.from_numpy(synth.activations(synth.rng_for(5, 5), 1, lm.K).view(np.uint16)).to(dev)
        yl = torch.empty(1, lm.N, dtype=torch.float32, device=dev)
        calls["lmhead"] = lambda: qk.qk_matmul_q6k(Wl, xl, yl, 1, lm.N, lm.K, s)
    if args.profile == "dequant":
        g = decode_linears()[4]  # ffn_gate, Q4_K 8192 x 3072: 14 MB in, 100 MB out
        nbk = g.N * g.K // 256
        gen = torch.Generator(device=dev)
        gen.manual_seed(6)
        Wq = device_weights(torch, gen, g.qtype, g.N, g.K, dev)
        dq_out = torch.empty(nbk * 256, dtype=torch.float32, device=dev)
        calls["dequant"] = lambda: qk.qk_dequant_q4k(Wq, nbk, dq_out, s)
    if args.profile in ("attn_decode", "attn_prefill"):
        H, Hkv, Dh = synth.N_HEADS, synth.N_KV_HEADS, synth.HEAD_DIM
        M, L = (1, ATTN_L) if args.profile == "attn_decode" else (PREFILL_M, PREFILL_M)
        qa, ka, va = attention_inputs(torch, dev, M, L - M, L, 7)
        oa = torch.empty(M, H, Dh, device=dev)
        calls[args.profile] = lambda: qk.qk_gqa_attention(qa, ka, va, oa, M, H, Hkv, Dh, L - M, L, 1 / np.sqrt(Dh), s)
    with torch.cuda.stream(stream):
        for _ in range(5):
            calls[args.profile]()
    qk.qk_get_device_status(s)
    torch.cuda.synchronize()
    print("profiled %s: 5 calls" % args.profile)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-configuration measurements")
    ap.add_argument("--profile", choices=["gateup", "down", "v", "decode", "lmhead", "dequant", "attn_decode",
                                          "attn_prefill"],
                    help="run one call of the step 5 times on one GPU and exit (for ncu)")
    args = ap.parse_args()
    if args.profile:
        run_profile(args)
        return
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.gpus != world:
        sys.exit("bench.py: --gpus %d but WORLD_SIZE is %d: launch N > 1 ranks with torchrun "
                 "(python -m torch.distributed.run --nproc-per-node N bench.py --gpus N ...)" % (args.gpus, world))
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        backend = "gloo" if args.impl == "reference" else "nccl"
        dist_mod.init_process_group(backend=backend)
        dist = dist_mod

    if args.impl == "reference":
        res = run_reference(args, rank)
    else:
        res = run_gpu(args, rank, world, dist)
        if res is not None and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline()
            res["cpu_baseline"]["single_thread"] = cpu_single_thread()
    if res is not None:
        print(json.dumps(res), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
