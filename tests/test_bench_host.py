"""Host logic of the benchmark that needs no GPU: the roofline's DRAM traffic
is taken from a committed ncu capture only while the kernel's source is the
one that was captured; the roofline holds each kernel to the bound it is
closer to; the clock sampler's parsing."""
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


CODE = "// kernel\n__global__ void k(int *p) { p[0] = 1; }  // store\n"


def test_traffic_is_reported_for_the_captured_source(tmp_path, monkeypatch):
    _tree(tmp_path, CODE, bench.code_sha(CODE))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # the configuration name maps to the workload the capture names
    assert bench._kernel_traffic("k_demo", "k.cu", "c1") == 1234.0
    assert bench._kernel_traffic("k_demo", "k.cu", "decode b64 ctx8192") == 1234.0


def test_traffic_survives_a_comment_edit(tmp_path, monkeypatch):
    edited = "/* what k does,\n   reworded */\n\n__global__ void k(int *p) { p[0] = 1; }\n"
    _tree(tmp_path, edited, bench.code_sha(CODE))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._kernel_traffic("k_demo", "k.cu", "c1") == 1234.0


def test_traffic_is_null_once_the_code_changes(tmp_path, monkeypatch):
    _tree(tmp_path, CODE.replace("p[0] = 1", "p[0] = 2"), bench.code_sha(CODE))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._kernel_traffic("k_demo", "k.cu", "c1") is None


def test_code_sha_ignores_comments_only():
    assert bench.code_sha("a; // x\n") == bench.code_sha("a;\n")
    assert bench.code_sha("a; /* x */\n") == bench.code_sha("a;\n")
    assert bench.code_sha("a;\n") != bench.code_sha("b;\n")
    assert bench.code_sha("a;\n") == hashlib.sha256(b"a;").hexdigest()[:16]


def test_traffic_is_null_without_a_capture(tmp_path, monkeypatch):
    text = CODE
    _tree(tmp_path, text, bench.code_sha(text))
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


class _Wl:
    """Shapes of a workload as the roofline needs them (decode-like)."""
    name = "c1"
    Hi, Di, Hq, Dqk, Dv = 64, 128, 128, 576, 512
    q_idx_dtype, k_idx_dtype, kv_dtype = "bf16", "e4m3", "bf16"
    n_seq, n_q = 64, 64


def test_roofline_reports_the_closer_bound(monkeypatch):
    """A kernel is held to the roof it is closer to: bytes against the
    measured HBM copy bandwidth, FLOPs against the dense tensor peak of its
    operands (FP8 for the indexer, the sustained figure inside a long step)."""
    peaks = {"hbm_gbs": 1000.0, "bf16_tflops": 100.0, "bf16_tflops_sustained": 80.0,
             "src": "measured"}
    # 500 GB/s of bytes, 10 TFLOP/s of work: HBM-bound
    r = bench.roofline_of("attn", _Wl, {"attn": 5e11, "flops_attn": 1e13}, 1000.0, peaks, False)
    assert r["bound"] == "hbm" and abs(r["frac"] - 0.5) < 1e-12
    assert r["other_bound"]["bound"] == "tensor" and abs(r["other_bound"]["frac"] - 0.1) < 1e-12
    # 100 GB/s of bytes, 60 TFLOP/s of work inside a long step: tensor-bound,
    # against the sustained peak
    r = bench.roofline_of("attn", _Wl, {"attn": 1e11, "flops_attn": 6e13}, 1000.0, peaks, True)
    assert r["bound"] == "tensor" and r["peak"] == 80.0 and abs(r["frac"] - 0.75) < 1e-12
    assert r["traffic"] is None
    # the indexer multiplies FP8 operands: twice the bf16 peak
    r = bench.roofline_of("indexer", _Wl, {"indexer": 1e6, "flops_indexer": 1e16}, 1000.0, peaks,
                          False)
    assert r["bound"] == "tensor" and r["peak"] == 200.0


def test_algorithmic_bytes_count_each_sequences_rows_once():
    """A prefill's rows share their sequence's keys and latent rows: the
    bytes the method must move count them once per sequence; decode rows
    (one per request) count their own."""
    import synth
    wl = synth.make("c0")                         # one sequence, 256 causal rows, K = 32
    a = bench.algorithmic_bytes(wl, out_bytes=4)
    n = wl.n_q
    q_b = n * wl.Hq * wl.Dqk * 4 + n * wl.Hq * wl.Dv * 4 + n * wl.K * 4
    assert a["attn"] == 256 * wl.Dqk * 4 + q_b   # fp32 rows: each of the 256 positions once
    assert a["flops_attn"] == 2 * sum(min(32, p + 1) for p in range(256)) * wl.Hq * (wl.Dqk + wl.Dv)
    d = synth.make("c1", batch=3, ctx=100, K=64)  # three decode rows of 100 positions
    a = bench.algorithmic_bytes(d)
    row_b = d.Dqk * 2                            # bf16 latent row
    assert a["attn"] == 3 * 64 * row_b + 3 * (d.Hq * d.Dqk * 2 + d.Hq * d.Dv * 2 + 64 * 4)
