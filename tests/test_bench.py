"""bench.py's host-side contract, checked on CPU: the algorithmic work units of a
step, the JSON line of the reference arm (the fp64 oracle on host cores), and
the multi-process launch (torchrun, gloo, world size 2: rank 0 alone prints)."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

ENV = dict(os.environ, QK_REF_STEP_S="0.3", OMP_NUM_THREADS=os.environ.get("OMP_NUM_THREADS", "4"))


def test_step_work_units():
    """Prefill flops of the step (gate/up, down, attn_v at M=1024), the decode
    layer's algorithmic bytes (packed weights of one layer's 7 linears, x, y)
    and the dequant export's (packed weights in, fp32 weights out)."""
    assert bench.prefill_flops() == 2.0 * 1024 * (2 * 8192 * 3072 + 3072 * 8192 + 1024 * 3072)
    weights = sum(bench.synth.weight_bytes(l.qtype, l.N, l.K) for l in bench.decode_linears())
    assert weights == 63_922_176
    x = sum(2 * l.K for l in bench.decode_linears())
    y = sum(4 * l.N for l in bench.decode_linears())
    assert bench.decode_bytes() == weights + x + y == 64_086_016
    # dequant export of the same seven tensors: packed in, fp32 out (100,663,296 weights)
    assert sum(l.N * l.K for l in bench.decode_linears()) == 100_663_296
    assert bench.dequant_bytes() == weights + 4 * 100_663_296 == 466_575_360


def _json_lines(out):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def _check_reference_line(d):
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["steps"] == 1 and d["warmup"] >= 3
    assert d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["data"] == "synthetic" and "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=ENV, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_reference_line(lines[0])


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_reference_arm_two_ranks_gloo():
    """Launched like the multi-GPU bench (torchrun, one process per rank): the
    ranks join a gloo group, rank 0 alone runs the oracle and prints one line,
    and every rank exits 0."""
    pytest.importorskip("torch.distributed")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, env=ENV, capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_reference_line(lines[0])


def test_clock_summary_parsing(tmp_path, monkeypatch):
    """The clocks object of the bench line: median SM clock, max clock and the
    throttle reasons seen active, from nvidia-smi's CSV samples."""
    monkeypatch.setenv("QK_CLOCKS_DIR", str(tmp_path))
    c = bench.Clocks(0)
    c.proc = object()  # as if the sampler had run
    with open(c.path, "w") as f:
        f.write("0, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active\n"
                "0, 1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active\n"
                "0, 2070, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active\n"
                "garbage line\n")
    d = c.summary()
    assert d["sm_mhz"] == 2070.0 and d["sm_max_mhz"] == 2070.0 and d["samples"] == 3
    assert d["reasons"] == ["sw_power_cap"]
    assert "untimed replays" in d["window"]
    c.proc = None
    assert c.summary()["reasons"] == ["nvidia-smi unavailable"]


def test_roofline_fraction_uses_the_attainable_rate():
    """Each configuration reports its fraction of min(peak, intensity x HBM):
    an HBM-bound decode GEMV against the copy bandwidth, a tensor-bound GEMM
    against the tensor peak."""
    pk = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}
    # decode: 64 MB moved for 63 MFLOP in 0.016 ms -> 4 TB/s, HBM-bound
    r = bench.roof(63e6, 64e6, 0.016, pk)
    assert r["bound"] == "hbm"
    assert abs(r["gbs"] - 4000.0) < 1e-6
    assert abs(r["frac_of_attainable"] - 4000.0 / 6800.0) < 1e-9
    # prefill: 103 GFLOP over 35 MB in 0.1 ms -> 1030 TFLOP/s, tensor-bound
    r = bench.roof(103e9, 35e6, 0.1, pk)
    assert r["bound"] == "tensor" and abs(r["frac_of_attainable"] - 1030.0 / 1900.0) < 1e-9
    s = bench.stats([1.0, 2.0, 3.0, 4.0, 100.0])
    assert s["median"] == 3.0 and s["min"] == 1.0 and s["max"] == 100.0 and s["runs"] == 5
    assert 4.0 < s["p95"] <= 100.0


def test_lin_bytes_and_sweep_totals():
    """Config 4's weights: the 28 layers' linears under the Q4_K_M mix plus the
    tied LM head, 2,022,193,152 bytes (1.883 GiB, the pages' 1.9 GiB)."""
    model = bench.synth.model_linears()
    assert sum(bench.synth.weight_bytes(l.qtype, l.N, l.K) for _, l in model) == 2_022_193_152
    q = bench.synth.Linear("attn_q", "q4k", 3072, 3072)
    assert bench.lin_bytes(q, 16) == 3072 * 12 * 144 + 2 * 16 * 3072 + 4 * 16 * 3072
    g = bench.synth.Linear("ffn_gate", "q4k", 8192, 3072)
    assert bench.lin_bytes(g, 1, gateup=True) == 2 * 8192 * 12 * 144 + 2 * 3072 + 2 * 8192


def test_gpus_flag_must_match_the_launcher():
    """--gpus N without a launcher that starts N ranks is an error, not a
    silent single replica."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--steps", "1"],
                       env={k: v for k, v in ENV.items() if k not in ("WORLD_SIZE", "RANK")}, capture_output=True,
                       text=True, timeout=300, cwd=ROOT)
    assert r.returncode != 0 and "torchrun" in r.stderr
