"""bench.py's own command lines run end to end and print one well-formed JSON
line (the default forward line, and the backward, FP8 and decode modes)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
        "vs_baseline", "dtype", "data", "config", "roofline", "gpu_launches", "clocks", "e2e"}


def _run(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "3", "--warmup", "3", *args],
                         cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    assert KEYS <= set(d), sorted(KEYS - set(d))
    assert d["value"] > 0 and d["roofline"]["frac"] > 0 and d["e2e"]["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["d2h_bytes_per_step"] > 0
    return d


def test_default_forward_line():
    d = _run("--no-cpu-baseline")
    assert d["config"]["workload"] == "causal_fp16_b1h32n8192d128" and d["e2e"]["value"] > 0


@pytest.mark.parametrize("extra", [["--pass", "bwd", "--no-cpu-baseline"], ["--fp8", "--no-cpu-baseline"],
                                   ["--decode", "decode_bf16_b8h32kv8_nk32768d128", "--num-splits", "2"],
                                   ["--decode", "decode_bf16_b1h32kv8_nk131072d128", "--num-splits", "auto"]])
def test_other_modes(extra):
    _run(*extra)
