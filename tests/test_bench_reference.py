"""bench.py's reference arm (the fp64 oracle on the host cores) on CPU: it prints
the GPU arm's config for the same workload, and it neither builds nor loads the
library."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROBE = r"""
import io, json, sys, contextlib
sys.path.insert(0, {root!r})
import bench
buf = io.StringIO()
with contextlib.redirect_stdout(buf):
    bench.main(["--impl", "reference", "--workload", {wl!r}, "--steps", "1", "--warmup", "3"])
line = json.loads(buf.getvalue().strip().splitlines()[-1])
w = bench.make_workload({wl!r})
if {wl!r}.startswith("single"):
    want = bench.serial_config(w, 1)
elif w.new_tokens is not None:
    want = bench.prefill_config(w, 1)
else:
    want = bench.decode_config(w, 1, int(w.shared_prefix))
print(json.dumps(dict(line=line, same=line["config"] == want,
                      product=[m for m in sys.modules if m.startswith("paged_kv_cache_decode")])))
"""


@pytest.mark.parametrize("workload", ["single_t128", "single_gqa_t2048", "prefix_bf16"])
def test_reference_arm_config_and_no_library(workload):
    r = subprocess.run([sys.executable, "-c", PROBE.format(root=ROOT, wl=workload)],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    out = json.loads(r.stdout.strip().splitlines()[-1])
    line = out["line"]
    assert out["same"], "reference config differs from the GPU arm's"
    assert out["product"] == [], "the reference arm imported the library package"
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["cpu_baseline"]["cores"] >= 1
