"""The benchmark's one-line JSON contract, read back from a real run: the
reference arm (the float64 oracle on the host, no GPU) and, on a GPU, the
CUDA arm with its roofline, CPU baseline, end-to-end, launch count and clock
record.
"""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, timeout):
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, timeout=timeout)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, p.stdout[-2000:]
    return json.loads(lines[0])


def _common(d, workload):
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "e2e"):
        assert k in d, k
    assert d["unit"] == "Gelem/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["data"] == "synthetic"
    assert d["config"]["workload"] == workload
    assert d["vs_baseline"] is None  # the pages publish no number for this metric
    assert d["value"] > 0 and d["ms_per_step"] > 0


def test_default_workload_is_the_largest_single_gpu_configuration():
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench
    from mamba_selective_scan_gb300.inputs import WORKLOADS
    assert bench.DEFAULT_WORKLOAD == max(WORKLOADS, key=lambda k: WORKLOADS[k].elems)


def test_reference_arm_prints_the_contract_line():
    # a small workload keeps the CPU suite quick; the arm is the same code
    d = _run(["--impl", "reference", "--steps", "1", "--warmup", "3",
              "--workload", "trainer_b8_t128_d512"], timeout=600)
    _common(d, "trainer_b8_t128_d512")
    assert d["impl"] == "reference" and d["steps"] == 1 and d["warmup"] == 3
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"]
    assert cb["value"] == d["value"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


@pytest.mark.gpu
def test_cuda_arm_prints_the_contract_line():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = _run(["--steps", "20", "--warmup", "3", "--no-extras", "--cpu-seconds", "2"], timeout=900)
    _common(d, "longseq_b1_t65536_d2048")
    assert "impl" not in d or d["impl"] != "reference"
    assert d["scaling"] == "weak" and d["warmup"] >= 3
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    assert 0 < r["frac"] < 1.5
    # the achieved figure is the metric's minimum bytes over the backward's time
    bwd_s = d["config"]["batch"] * d["config"]["seq_len"] * d["config"]["d_inner"] / (
        d["hbm_roofline"]["bwd_gelem_s"] * 1e9)
    assert abs(r["algorithmic_bytes_per_launch"] / bwd_s / 1e9 - r["achieved"]) < 0.01 * r["achieved"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0
    assert cb["single_thread"]["cores"] == 1 and cb["model"]
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert e["value"] != d["value"]
    per_step = d["config"]["fwd_launches"] + d["config"]["bwd_launches"]
    assert per_step >= 2 and d["gpu_launches"] == 20 * per_step
    c = d["clocks"]
    assert c["sm_max_mhz"] > 0 and isinstance(c["reasons"], list)


def test_traffic_key_ignores_comments_but_not_code():
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench
    src = "int f(int a) {  // one\n  return a + 1; /* two\n lines */ }\n"
    assert bench.code_only(src) == bench.code_only("int f(int a) {\n return a + 1; }")
    assert bench.code_only(src) != bench.code_only("int f(int a) { return a + 2; }")
    assert len(bench.source_hash()) == 16


def test_traffic_record_from_a_launch_list(tmp_path):
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench
    hdr = '"ID","Kernel Name","Metric Name","Metric Unit","Metric Value"\n'
    rows = []
    for launch, (name, rd, wr) in enumerate([
            ("void m3_fwd2_kernel<float, 0, 16>(FwdArgs)", "1.5", "0.5"),
            ("void m3_fwd2_kernel<float, 1, 16>(FwdArgs)", "4", "2"),
            ("void m3_bwd2_kernel<float, 0, 0, 16, 0>(BwdArgs)", "10", "0"),
            ("void m3_fwd2_kernel<float, 0, 16>(FwdArgs)", "2.5", "0.5"),
            ("void other_kernel(int)", "99", "99")]):
        rows.append(f'"{launch}","{name}","gpu__time_duration.sum","ns","1,000"\n')
        rows.append(f'"{launch}","{name}","dram__bytes_read.sum","Mbyte","{rd}"\n')
        rows.append(f'"{launch}","{name}","dram__bytes_write.sum","Mbyte","{wr}"\n')
    p = tmp_path / "launches.csv"
    p.write_text("==PROF== a line before the table\n" + hdr + "".join(rows))
    rec = bench.traffic_from_launch_list(str(p), "w")
    per = rec["per_kernel_bytes_per_launch"]
    assert per == {"m3_fwd2_kernel<float, 0, 16>": 2_500_000, "m3_fwd2_kernel<float, 1, 16>": 6_000_000,
                   "m3_bwd2_kernel<float, 0, 0, 16, 0>": 10_000_000}
    assert rec["traffic"] == {"w": {"fwd": 8_500_000, "bwd": 10_000_000}}
    assert rec["source_sha256_16"] == bench.source_hash()
