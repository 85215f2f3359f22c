"""The one-unit-at-a-time form of the block kernel against the oracle.

The block kernel streams its units (each lane group's last pass over a unit
already loads its rows of the next) except for V+Q+K launches of many rounds of
units and Q/K-only half-split launches, which walk one unit at a time.  The
small shapes of the parity, fuzz, layout and chunk tests all stream, so this
test builds the library with streaming off (TFU_BLOCK_STREAM=0) and runs those
tests again in a child process that loads that build (TF_ULYSSES_LIBRARY): both
loops stay checked against the oracle on ragged shapes, partial chunks and
B > 1.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_unstreamed_block_kernel_parity(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from ulysses_sequence_attention_tf_gb300 import build
    lib = build.build(defines=["TFU_BLOCK_STREAM=0"], out=str(tmp_path / "libtf_ulysses.so"))
    env = dict(os.environ, TF_ULYSSES_LIBRARY=lib)
    files = [os.path.join(ROOT, "tests", f)
             for f in ("test_gpu_fuzz.py", "test_gpu_layouts_neox.py", "test_gpu_parity.py", "test_gpu_chunks.py",
                       "test_gpu_edge_values.py")]
    cmd = [sys.executable, "-m", "pytest", *files, "-x", "-q", "-m", "gpu", "-p", "no:cacheprovider",
           "-k", "not video_dit and not full_size and not large"]
    r = subprocess.run(cmd, env=env, cwd=ROOT, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and "skipped" not in r.stdout.splitlines()[-1], r.stdout[-2000:]
