"""The benchmark's JSON line contract, checked on the CPU through the
reference arm (the CPU oracle): one line with the metric, value, unit, rank
and step counts, the CPU-baseline block and an end-to-end block."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "1"], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1 and d["value"] > 0
    assert d["config"]["workload"] == "image_2048_bf16" and "sample" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def _bench_module():
    sys.path.insert(0, ROOT)
    import bench
    return bench


def test_clock_sampler_child_reports_samples_inside_the_region():
    # the NVML child run against a stand-in for the driver's library: it
    # prints "ready", keeps its samples and dumps them when terminated; the
    # parent parses them and decodes the clock-event reason bits
    import time
    bench = _bench_module()
    fake = '''
class _FakeNvml:
    def nvmlInit_v2(self): return 0
    def nvmlDeviceGetHandleByUUID(self, u, p): return 0
    def nvmlDeviceGetMaxClockInfo(self, h, k, p): p._obj.value = 2070; return 0
    def nvmlDeviceGetClockInfo(self, h, k, p): p._obj.value = 1980; return 0
    def nvmlDeviceGetCurrentClocksEventReasons(self, h, p): p._obj.value = 0x4 | 0x40; return 0
nv = _FakeNvml()'''
    code = bench.NVML_CHILD.replace('nv = ctypes.CDLL("libnvidia-ml.so.1")', fake)
    assert code != bench.NVML_CHILD
    saved = bench.NVML_CHILD
    bench.NVML_CHILD = code
    try:
        s = bench.NvmlSampler("GPU-test")
        s.wait_ready()
        t0 = time.time()
        time.sleep(0.03)
        t1 = time.time()
        rows = s.stop()
    finally:
        bench.NVML_CHILD = saved
    assert len(rows) >= 10
    c = bench.ClockSampler.summarise(rows, t0, t1, 0.0, "NVML")
    assert c["samples"] >= 5 and c["window"] == "timed region"
    assert c["sm_mhz"] == 1980 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


def test_clock_sampler_without_nvml_gives_no_rows():
    bench = _bench_module()
    assert bench.NvmlSampler(None).stop() == []
    saved = bench.NVML_CHILD
    bench.NVML_CHILD = "import sys; sys.exit(1)"
    try:
        s = bench.NvmlSampler("GPU-test")
        s.wait_ready(timeout=10)
        assert s.stop() == []
    finally:
        bench.NVML_CHILD = saved


def test_link_bound_is_the_slowest_leg():
    bench = _bench_module()
    rates = {"h2d_gbs": 200.0, "d2h_gbs": 100.0, "both_gbs": 250.0}
    # in-leg bound: 2e9 B at 200 GB/s = 10 ms; out: 0.5e9 at 100 = 5 ms; both: 2.5e9 at 250 = 10 ms
    assert abs(bench.link_bound_ms(rates, 2e9, 0.5e9) - 10.0) < 1e-9
    assert abs(bench.link_bound_ms(rates, 1e9, 1.5e9) - 15.0) < 1e-9
    assert abs(bench.link_bound_ms(rates, 1e9, 1e9) - 10.0) < 1e-9
