"""The configuration sweep runs end to end on its smallest configuration (C1):
graph capture of the library calls, both L2 flushes, the same-size contiguous
copy and the torch / cudaMemcpy2DAsync baselines, one JSON line per point and a
summary line."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_sweep_c1_runs_and_reports():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = subprocess.run([sys.executable, "-m", "ulysses_sequence_attention_tf_gb300.sweep", "--only", "C1"], cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.strip()]
    points = [x for x in lines if "sweep" in x]
    summary = [x["summary"] for x in lines if "summary" in x]
    assert len(points) == 2 and len(summary) == 1
    for p in points:
        assert p["sweep"] == "C1" and p["timing"] == "graph"
        for key in ("gbs_median", "gbs_median_flushed", "gbs_median_read_flushed", "eager_gbs_median_flushed",
                    "contiguous_copy_gbs_median_read_flushed"):
            assert p[key] > 0, key
        assert p["pass"] is None  # below the gated size
        base = p["baselines_gbs_median"]
        assert set(base) == {"torch_copy", "torch_permute", "memcpy2d"}
        for name in ("torch_copy", "torch_permute"):
            assert base[name]["read_flushed"] > 0 and base[name]["write_flushed"] > 0
    assert summary[0]["points"] == 2 and summary[0]["gated_points"] == 0
