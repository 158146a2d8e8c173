"""Host-side logic of bench.py (no GPU): clock-sample parsing, the stored
DRAM-traffic records and the workload descriptions in the JSON line."""

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from block_sparse_long_bigbird_gb300.workloads import WORKLOADS  # noqa: E402


def _sampler(lines):
    s = bench.ClockSampler(0)
    s.lines = lines
    return s.summary()


def test_clock_summary_median_and_reasons():
    # index, sm, max sm, power, active mask, hw_slowdown, hw_thermal, sw_thermal, sw_power_cap
    lines = [
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1395.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    s = _sampler(lines)
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_flags_thermal_and_skips_garbage():
    lines = [
        "garbage line",
        "0, 1500, 2070, 700.0, 0x40, Not Active, Active, Not Active, Not Active",
        "0, N/A, 2070, 700.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    s = _sampler(lines)
    assert s["samples"] == 1 and s["sm_mhz"] == 1500.0
    assert s["reasons"] == ["hw_thermal_slowdown"]


def test_clock_summary_without_samples():
    s = _sampler([])
    assert s["samples"] == 0 and s["reasons"] == ["unavailable"]


def test_traffic_records_follow_the_kernel_source(tmp_path, monkeypatch):
    # The DRAM traffic the bench reports comes from an ncu capture of one
    # kernel source: a record is used only while the source hash it was taken
    # with matches the current file, and is ignored (traffic: null) otherwise.
    src = tmp_path / "kernel.cuh"
    src.write_text("// kernel v1\n")
    rec = {"kernel": "k", "workload": "bigbird_bf16_n4096", "source_sha": bench.file_sha(str(src)),
           "dram_bytes_per_launch": 123, "source": "test"}
    tf = tmp_path / "traffic.json"
    tf.write_text(json.dumps([rec]))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tf))
    assert bench.read_traffic("k", "bigbird_bf16_n4096", str(src)) == 123
    assert bench.read_traffic("k", "longformer_bf16_n4096", str(src)) is None
    src.write_text("// kernel v2\n")
    assert bench.read_traffic("k", "bigbird_bf16_n4096", str(src)) is None


def test_traffic_records_are_well_formed():
    with open(bench.TRAFFIC_FILE) as f:
        entries = json.load(f)
    for e in entries:
        assert set(e) >= {"kernel", "workload", "source_sha", "dram_bytes_per_launch", "source"}
        assert e["workload"] in WORKLOADS
        assert isinstance(e["dram_bytes_per_launch"], int) and e["dram_bytes_per_launch"] > 0
        assert len(e["source_sha"]) == 16


def test_workload_configs_name_the_workload_and_no_model():
    for name, wl in WORKLOADS.items():
        cfg = bench.workload_config(wl)
        assert cfg["workload"].startswith(name)
        assert "model" not in cfg
        for key in ("B", "H", "n", "d", "dtype", "l2"):
            assert key in cfg, (name, key)


def test_reference_arm_times_the_oracle_without_the_library():
    # `bench.py --impl reference` times the float64 oracle on the host cores
    # and prints the contract's JSON line; it must not load the CUDA library
    # (a fresh interpreter, since other tests in this process load it).
    import subprocess

    code = (
        "import sys, runpy, io, contextlib\n"
        "sys.argv = ['bench.py', '--impl', 'reference', '--workload', 'bigbird_fp32_n1024',\n"
        "            '--steps', '1', '--warmup', '0', '--cpu-seconds', '1']\n"
        "buf = io.StringIO()\n"
        "with contextlib.redirect_stdout(buf):\n"
        "    try:\n"
        "        runpy.run_path('bench.py', run_name='__main__')\n"
        "    except SystemExit:\n"
        "        pass\n"
        "print(buf.getvalue().strip().splitlines()[-1])\n"
        "print('libsparse_attn' in open('/proc/self/maps').read())\n"
    )
    res = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    out = res.stdout.strip().splitlines()
    line, loaded = json.loads(out[-2]), out[-1]
    assert loaded == "False", "the reference arm loaded the CUDA library"
    assert line["impl"] == "reference" and line["dtype"] == "f64"
    assert line["value"] > 0 and line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    assert line["config"]["workload"].startswith("bigbird_fp32_n1024")
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
