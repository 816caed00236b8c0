"""The benchmark's JSON line (CPU): `bench.py --impl reference` runs the
oracle as the reference arm without a GPU and prints one line with the keys
the benchmark contract fixes, on the same config as the GPU arm."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] == 3
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    sys.path.insert(0, ROOT)
    import bench
    assert d["config"] == bench.hotpath_config()
    assert d["metric"] == bench.METRIC


def test_kernel_source_hash_ignores_comments_only():
    """The stored ncu traffic is tied to the kernels' code: comments and blank
    lines do not change the hash; code, including string literals, does."""
    sys.path.insert(0, ROOT)
    import bench
    src = ('int a = 1; // the count\n'
           '/* a block\n   comment */\n'
           'asm("mov.b32 %0, %1; // not a comment");\n'
           "char c = '/';\n")
    same = ('int a = 1;\n\n'
            'asm("mov.b32 %0, %1; // not a comment");   \n'
            "char c = '/'; /* trailing */\n")
    assert bench._code_only(src) == bench._code_only(same)
    assert "// not a comment" in bench._code_only(src)
    changed = src.replace("int a = 1", "int a = 2")
    assert bench._code_only(changed) != bench._code_only(src)
    changed_literal = src.replace("not a comment", "not a remark")
    assert bench._code_only(changed_literal) != bench._code_only(src)
    assert len(bench.kernel_source_hash()) == 16


def test_shapes_filter_rejects_unknown_names_before_any_gpu_work():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "shapes",
                        "--shape", "no_such_shape"], capture_output=True, text=True,
                       timeout=300, cwd=ROOT)
    assert r.returncode != 0
    assert "unknown --shape ['no_such_shape']" in r.stderr
    assert "tail_s4097_c3077_bf16" in r.stderr
