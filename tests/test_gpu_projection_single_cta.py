"""The single-CTA form of the projection kernel against the oracle.

The library runs the projection on CTA pairs (the 2-SM MMA); the single-CTA
kernel is its fallback (taken when no pair cluster fits, and the form of the
build option TFU_GEMM_PAIR=0).  This test builds the library with that option
and runs the projection parity tests again, in a child process that loads that
build (TF_ULYSSES_LIBRARY), so both forms stay checked against the oracle.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_single_cta_projection_parity(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from ulysses_sequence_attention_tf_gb300 import build
    lib = build.build(defines=["TFU_GEMM_PAIR=0"], out=str(tmp_path / "libtf_ulysses.so"))
    env = dict(os.environ, TF_ULYSSES_LIBRARY=lib)
    cmd = [sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_gpu_projection.py"), "-x", "-q",
           "-m", "gpu", "-p", "no:cacheprovider"]
    r = subprocess.run(cmd, env=env, cwd=ROOT, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and "skipped" not in r.stdout.splitlines()[-1], r.stdout[-2000:]
