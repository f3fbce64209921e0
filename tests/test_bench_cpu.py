"""bench.py's reference arms of the two extra operations run on the host
alone and print one contract line each (the default operation's arm is
covered by the two-rank test in test_dist_cpu.py)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("op,tokens", [("kv_insert", 2048), ("query_absorb", 4)])
def test_reference_arm_of_extra_ops(op, tokens):
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--op", op,
           "--tokens", str(tokens), "--steps", "1", "--warmup", "3"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, OMP_NUM_THREADS="2"))
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["unit"] == "GB/s" and rec["value"] > 0
    assert rec["higher_is_better"] is True and rec["steps"] == 1 and rec["warmup"] == 3
    assert rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["e2e"]["d2h_bytes_per_step"] == 0
