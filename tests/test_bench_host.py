"""Host logic of bench.py that needs no GPU: the profile hash ignores comments
but not code, both arms report the same config object, and a DRAM traffic
entry is only used while it matches the kernel source it was taken on."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synthetic  # noqa: E402


def test_code_hash_ignores_comments_not_code(tmp_path):
    a = tmp_path / "a.cu"
    a.write_text("int f(int x) {\n  return x + 1;  // one\n}\n")
    b = tmp_path / "b.cu"
    b.write_text("// header\nint f(int x) {\n\n  return x + 1;  // another comment\n}\n")
    c = tmp_path / "c.cu"
    c.write_text("int f(int x) {\n  return x + 2;\n}\n")
    d = tmp_path / "d.cu"
    d.write_text('const char* s = "a // b";\n')
    e = tmp_path / "e.cu"
    e.write_text('const char* s = "a // c";\n')
    assert bench.code_hash(str(a)) == bench.code_hash(str(b))
    assert bench.code_hash(str(a)) != bench.code_hash(str(c))
    assert bench.code_hash(str(d)) != bench.code_hash(str(e))      # "//" inside a string is code


def test_workload_config_is_shared_by_both_arms():
    wl = synthetic.WORKLOADS["mixtral"]
    cfg = bench.workload_config(wl, "mxfp8", 1)
    assert cfg["workload"].startswith("mixtral: Mixtral-8x7B MoE layer T=16384 H=4096 I=14336 E=8 top-2")
    assert cfg["gemm_flops_per_step"] == 18.0 * 16384 * 2 * 4096 * 14336
    assert cfg["parallelism"] == "single GPU"
    assert bench.workload_config(wl, "mxfp8", 4)["parallelism"] == "replicas"


def test_traffic_entry_tracks_the_kernel_source(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    src_dir = tmp_path / "mxfp8_grouped_gemm_gb300" / "csrc"
    src_dir.mkdir(parents=True)
    src = src_dir / "gemm.cu"
    src.write_text("int k() { return 1; }\n")
    entry = {"bytes_per_launch": 123, "source_sha": bench.code_hash(str(src))}
    (prof / "ncu_traffic.json").write_text(json.dumps({"source": "gemm.cu", "entries": {"mixtral/fwd.gate_up": entry}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_for("fwd.gate_up", "mixtral") == 123
    assert bench.traffic_for("fwd.down", "mixtral") is None
    src.write_text("// a comment edit\nint k() { return 1; }\n")
    assert bench.traffic_for("fwd.gate_up", "mixtral") == 123
    src.write_text("int k() { return 2; }\n")
    assert bench.traffic_for("fwd.gate_up", "mixtral") is None

