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
