"""bench.py's reference arm (the oracle on the host cores) runs without a GPU
and prints one JSON line with the keys the measurement contract asks for."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                          "--warmup", "3", "--ref-seconds", "1", "--workload", "tiny"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 3 and d["warmup"] == 3 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]


def test_kernel_source_hash_ignores_comments_but_not_code():
    sys.path.insert(0, ROOT)
    import bench
    src = 'int a = 1; // one\n/* block\n comment */\nconst char* s = "x // y";\n\n  int b;  \n'
    assert bench._code_only(src) == 'int a = 1;\nconst char* s = "x // y";\n  int b;'
    rel = os.path.join("chunked_prefill_mixed_gb300", "csrc")
    real = {f: open(os.path.join(ROOT, rel, f)).read() for f in ("mixed_attn.cu", "sarathi_internal.h", "plan.cpp")}
    base = bench.kernel_source_sha()
    commented = bench.kernel_source_sha(lambda p: real[os.path.basename(p)] + "\n// a note\n/* another */\n")
    assert commented == base
    changed = bench.kernel_source_sha(
        lambda p: real[os.path.basename(p)] + ("\nint extra_symbol;\n" if p.endswith("plan.cpp") else ""))
    assert changed != base
