"""The block kernel's accesses checked against the planned buffers on the GPU.

compute-sanitizer is not available where these tests run, so the library has a
checked build (TFU_CHECKED=1): the host records, for every slot and shard or
head group, one past the last byte the plan allows a kernel to touch (from the
same shapes and strides the plan uses), and the block kernel tests each row
load and store, each (cos, sin) load and each copy into the table ring against
those ranges.  An access outside them is skipped and sets bit 2 of
tf_ulysses_device_status; nothing faults.

This test builds that library, once streamed (the default) and once with every
launch walking one unit at a time (TFU_BLOCK_STREAM=0), and runs the block
kernel's parity files on each in a child process (TF_ULYSSES_LIBRARY): every
result must still equal the oracle (a skipped access would change it), and the
parity file's last test -- run after the others -- requires the device status to
be 0.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FILES = ("test_gpu_fuzz.py", "test_gpu_layouts_neox.py", "test_gpu_chunks.py", "test_gpu_edge_values.py",
         "test_gpu_full_size.py", "test_gpu_parity.py", "test_zz_no_alloc.py")


@pytest.mark.parametrize("defines", [["TFU_CHECKED=1"], ["TFU_CHECKED=1", "TFU_BLOCK_STREAM=0"]],
                         ids=["streamed", "one_unit_at_a_time"])
def test_checked_build_parity(tmp_path, defines):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from ulysses_sequence_attention_tf_gb300 import build
    lib = build.build(defines=defines, out=str(tmp_path / "libtf_ulysses.so"))
    env = dict(os.environ, TF_ULYSSES_LIBRARY=lib)
    files = [os.path.join(ROOT, "tests", f) for f in FILES]
    cmd = [sys.executable, "-m", "pytest", *files, "-x", "-q", "-m", "gpu", "-p", "no:cacheprovider",
           "-k", "not projection and not large"]
    r = subprocess.run(cmd, env=env, cwd=ROOT, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and "skipped" not in r.stdout.splitlines()[-1], r.stdout[-2000:]
