"""Host logic of the benchmark that needs no GPU: the roofline's DRAM traffic
is taken from a committed ncu capture only while the kernel's source is the
one that was captured."""
import hashlib
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _tree(tmp_path, src_text, rec_sha):
    csrc = tmp_path / "indexer_driven_top_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text(src_text)
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({
        "k_demo@decode b64 ctx8192": {"source": "k.cu", "source_sha": rec_sha,
                                      "dram_bytes_per_launch": 1234.0,
                                      "workload": "decode b64 ctx8192"}}))


def test_traffic_is_reported_for_the_captured_source(tmp_path, monkeypatch):
    text = "// kernel source\n"
    _tree(tmp_path, text, hashlib.sha256(text.encode()).hexdigest()[:16])
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # the configuration name maps to the workload the capture names
    assert bench._kernel_traffic("k_demo", "k.cu", "c1") == 1234.0
    assert bench._kernel_traffic("k_demo", "k.cu", "decode b64 ctx8192") == 1234.0


def test_traffic_is_null_once_the_source_changes(tmp_path, monkeypatch):
    _tree(tmp_path, "// kernel source, edited since the capture\n",
          hashlib.sha256(b"// kernel source\n").hexdigest()[:16])
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._kernel_traffic("k_demo", "k.cu", "c1") is None


def test_traffic_is_null_without_a_capture(tmp_path, monkeypatch):
    text = "// kernel source\n"
    _tree(tmp_path, text, hashlib.sha256(text.encode()).hexdigest()[:16])
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._kernel_traffic("k_other", "k.cu", "c1") is None
    assert bench._kernel_traffic("k_demo", "k.cu", "c3") is None
    assert bench._kernel_traffic("k_demo", "missing.cu", "c1") is None


def test_committed_captures_name_existing_sources():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        recs = json.load(f)
    assert recs
    for key, rec in recs.items():
        kernel, workload = key.split("@")
        assert rec["workload"] == workload and kernel.startswith("k_")
        assert os.path.exists(os.path.join(ROOT, "indexer_driven_top_gb300", "csrc",
                                           rec["source"]))
        assert rec["dram_bytes_per_launch"] > 0


def test_clock_sampler_reads_median_clock_and_active_reasons(tmp_path, monkeypatch):
    """A stand-in nvidia-smi prints three samples (power cap active in one)
    and then waits to be stopped, as the real one does under -lms."""
    fake = tmp_path / "bin" / "nvidia-smi"
    fake.parent.mkdir()
    fake.write_text(
        "#!/bin/sh\n"
        "printf '0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active\\n'\n"
        "printf '0, 1980, 2070, 1390.7, 0x4, Not Active, Not Active, Not Active, Active\\n'\n"
        "printf '0, 2055, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active\\n'\n"
        "exec sleep 30\n")
    fake.chmod(0o755)
    monkeypatch.setenv("PATH", f"{fake.parent}{os.pathsep}{os.environ['PATH']}")
    monkeypatch.setenv("SI_CLOCK_LOG_DIR", str(tmp_path / "clocks"))
    s = bench.ClockSampler(0)
    s.start()
    assert s.proc is not None and s.path.startswith(str(tmp_path / "clocks"))
    import time
    time.sleep(0.5)
    got = s.stop()
    assert got == {"sm_mhz": 2055.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
                   "samples": 3}


def test_clock_sampler_without_nvidia_smi(monkeypatch, tmp_path):
    monkeypatch.setenv("PATH", str(tmp_path))
    s = bench.ClockSampler(0)
    s.start()
    assert s.stop()["reasons"] == ["nvidia-smi unavailable"]
