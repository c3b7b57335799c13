"""bench.py's contract pieces that run without a GPU: the reference arm's JSON line, the rank
handling, the recorded-traffic lookup and the peak per operand type."""
import json
import os
import subprocess
import sys


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _run(args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=240)


def test_reference_arm_json_line():
    r = _run(["--impl", "reference", "--workload", "ragged_200x136x72", "--steps", "2", "--warmup", "3"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 3 and d["value"] > 0
    assert d["config"]["workload"] == "ragged_200x136x72"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_print_nothing():
    r = _run(["--impl", "reference", "--workload", "ragged_200x136x72", "--steps", "1", "--warmup", "3"],
             {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [l for l in r.stdout.splitlines() if l.startswith("{")]


def test_recorded_traffic_needs_the_current_sources(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.json").write_text(json.dumps(
        {"square_4096": {"tc_gemm_kernel": {"dram_bytes_per_launch": 123, "source_hash": "abc"}}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel=None: "abc")
    assert bench.recorded_traffic("square_4096", "tc_gemm_kernel") == 123
    assert bench.recorded_traffic("square_4096", "skinny_kernel") is None
    assert bench.recorded_traffic("glu_gate_1024x21568x4096", "tc_gemm_kernel") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel=None: "changed")
    assert bench.recorded_traffic("square_4096", "tc_gemm_kernel") is None


def test_source_hash_covers_every_kernel_file():
    h = bench.kernel_source_hash()
    assert len(h) == 16 and int(h, 16) >= 0
    import os
    csrc = os.path.join(bench.ROOT, "gemm_epilogue_gb300", "csrc")
    for kernel, files in bench.KERNEL_SOURCES.items():
        assert all(os.path.exists(os.path.join(csrc, f)) for f in files), kernel
        assert len(bench.kernel_source_hash(kernel)) == 16


def test_a_kernels_hash_follows_only_its_own_sources(tmp_path, monkeypatch):
    import os
    import shutil
    src = os.path.join(bench.ROOT, "gemm_epilogue_gb300", "csrc")
    dst = tmp_path / "gemm_epilogue_gb300" / "csrc"
    shutil.copytree(src, dst)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    tc, sk = bench.kernel_source_hash("tc_gemm_kernel"), bench.kernel_source_hash("skinny_kernel")
    with open(dst / "skinny.cu", "a") as f:
        f.write("\nint an_added_line;\n")
    assert bench.kernel_source_hash("tc_gemm_kernel") == tc
    assert bench.kernel_source_hash("skinny_kernel") != sk
    with open(dst / "ptx.cuh", "a") as f:  # shared by both
        f.write("\nint another_line;\n")
    assert bench.kernel_source_hash("tc_gemm_kernel") != tc


def test_tensor_peak_per_operand_type():
    from gemm_epilogue_gb300 import inputs as gen
    pk = {"bf16_tflops": 1909.9}
    assert bench.tensor_peak(pk, gen.WORKLOADS["square_4096"]) == 1909.9
    assert bench.tensor_peak(pk, gen.WORKLOADS["square_fp8_4096"]) == 2 * 1909.9


def test_source_hash_ignores_comments_and_layout_only():
    src = 'int a; // note\n/* block\n comment */ const char* s = "// kept"; char c = \'/\';\nint  b;'
    assert bench.strip_comments(src).split() == ["int", "a;", "const", "char*", "s", "=",
                                                 '"//', 'kept";', "char", "c", "=", "'/';", "int",
                                                 "b;"]
    assert " ".join(bench.strip_comments(src).split()) != " ".join(
        bench.strip_comments(src.replace("int  b", "int b2")).split())
