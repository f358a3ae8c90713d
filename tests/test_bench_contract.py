"""The bench's JSON contract, checked on the CPU: the reference arm (the CPU
oracle) prints one line with every required key, and the step's algorithmic
bytes are the three calls' (layout + notify as one call)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_step_bytes_are_the_three_calls():
    import bench
    from combine_get_dispatch_notify_gb300.workloads import CONFIGS
    w = CONFIGS["low_latency"]
    P = 13456
    b = bench.algorithmic_bytes(w, P)
    tok = w.R * w.T
    assert b["layout_notify"] == tok * 8 * w.K + tok * w.R + tok * w.R * 4
    assert bench.step_bytes_of(b) == b["layout_notify"] + b["dispatch"] + b["combine"]
    # the one call moves exactly the separate calls' bytes minus the membership rows read back
    assert b["layout"] + b["notify"] - b["layout_notify"] == tok * w.R


def test_reference_arm_prints_the_contract_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "tiny", "--steps", "2",
                          "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["higher_is_better"] is True
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["config"]["R"] == 2
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == d["value"]
    assert set(cb["per_op_ms"]) == {"layout", "notify", "dispatch", "combine"}
    assert cb["host"]["nproc"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_kernel_digest_ignores_comments_only():
    """The digest tying committed ncu traffic to a kernel source changes with the
    code, not with its comments or blank lines."""
    import bench
    a = "int f(int x) {\n    return x + 1;  // one more\n}\n"
    b = "// f: one more than x\nint f(int x) {\n\n    return x + 1;\n}\n/* end */\n"
    c = "int f(int x) {\n    return x + 2;\n}\n"
    assert bench.code_text(a) == bench.code_text(b)
    assert bench.code_text(a) != bench.code_text(c)
