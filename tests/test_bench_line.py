"""The JSON line contract of bench.py: the reference arm (the fp64 oracle on
the host cores, runs on the CPU) and the library arm (one small workload on
the GPU), each as the user runs it, in a child process."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BASE_KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
             "scaling", "vs_baseline", "dtype", "data", "config", "e2e")


def _run(args, env=None, timeout=600):
    e = dict(os.environ)
    e.update(env or {})
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT, env=e,
                       capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    return r.stdout


def test_reference_arm_prints_one_line():
    out = _run(["--impl", "reference", "--workload", "full_b1_h2_s512_d64", "--steps", "2", "--warmup", "1"])
    lines = [l for l in out.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for k in BASE_KEYS + ("impl", "cpu_baseline"):
        assert k in line, k
    assert line["impl"] == "reference"
    assert line["steps"] == 2 and line["warmup"] == 1 and line["n_gpus"] == 1
    assert line["config"]["workload"] == "full_b1_h2_s512_d64"
    assert line["value"] > 0 and line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_reference_arm_is_silent_on_other_ranks():
    out = _run(["--impl", "reference", "--workload", "full_b1_h2_s512_d64", "--steps", "1", "--warmup", "0"],
               env={"RANK": "1", "WORLD_SIZE": "2"})
    assert out.strip() == ""


@pytest.mark.gpu
def test_library_arm_line():
    out = _run(["--workload", "full_b1_h2_s512_d64", "--steps", "5", "--warmup", "3", "--no-cpu-baseline"])
    line = json.loads([l for l in out.splitlines() if l.strip()][-1])
    for k in BASE_KEYS + ("roofline", "clocks", "gpu_launches", "det_nondet_ratio", "ms_per_step_without_finalize"):
        assert k in line, k
    assert line["n_gpus"] == 1 and line["steps"] == 5 and line["warmup"] == 3
    assert line["dtype"] == "bf16" and line["higher_is_better"] is True and line["scaling"] == "weak"
    assert line["config"]["workload"] == "full_b1_h2_s512_d64"
    assert line["value"] > 0 and line["ms_per_step"] > 0
    rf = line["roofline"]
    assert rf["bound"] == "tensor" and rf["unit"] == "TFLOP/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    # delta, the persistent kernel and the finalize per timed step at least
    assert line["gpu_launches"] >= 3 * line["steps"]


def test_traffic_is_reported_only_for_the_kernel_source_it_was_taken_on(monkeypatch):
    # the roofline's DRAM traffic comes from an ncu capture keyed to the kernel
    # sources' hash: a figure is reported while the sources still have that
    # hash and withheld (null) once they change
    import sys
    sys.path.insert(0, ROOT)
    import bench
    h = bench.kernel_source_hash()
    assert len(h) == 16 and int(h, 16) >= 0
    assert bench.NCU_TRAFFIC, "no recorded captures"
    for (w, s), (nbytes, src) in bench.NCU_TRAFFIC.items():
        assert nbytes > 0
        assert bench.traffic_for(w, s) == (nbytes if src == h else None)
    w, s = next(iter(bench.NCU_TRAFFIC))
    monkeypatch.setitem(bench.NCU_TRAFFIC, (w, s), (123, h))
    assert bench.traffic_for(w, s) == 123
    monkeypatch.setitem(bench.NCU_TRAFFIC, (w, s), (123, "0" * 16))
    assert bench.traffic_for(w, s) is None
    assert bench.traffic_for("no_such_workload", "shift") is None
