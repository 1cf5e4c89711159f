"""The small GPU parity sweeps, run once more on the debug variant of the library
(libringattn_dbg.so, compiled with RA_DEBUG_BOUNDS: every tiled copy,
statistics copy and global row store is checked against the tensors' extents
before it is made, and a violation is reported as RA_ERR_DEVICE instead of
touching memory).  The sweeps run in a child process with RA_LIB_VARIANT set,
so the debug library is the one loaded there; each of its tests reads the
device error word, so a single failed check fails the run."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_parity_sweeps_pass_under_the_bounds_checks():
    from ring_attn_gb300.build import build

    build(debug_bounds=True)
    env = dict(os.environ, RA_LIB_VARIANT="debug_bounds")
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
           "tests/test_gpu_attention.py", "tests/test_gpu_permute_merge.py", "tests/test_gpu_dkdv_pair.py",
           "tests/test_gpu_gqa.py", "-k", "not full_size"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True,
                       timeout=1800)
    tail = "\n".join(r.stdout.splitlines()[-30:])
    assert r.returncode == 0, f"sweeps under the bounds checks failed:\n{tail}"
    assert " passed" in tail and "failed" not in tail


def test_the_debug_library_is_the_one_loaded_in_the_child():
    from ring_attn_gb300.build import build

    build(debug_bounds=True)
    env = dict(os.environ, RA_LIB_VARIANT="debug_bounds")
    code = "import ring_attn_gb300 as ra; print(ra.lib_path()); print(ra.load().ring_attn_debug_bounds())"
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, stdout=subprocess.PIPE, text=True, timeout=300)
    lines = r.stdout.split()
    assert r.returncode == 0 and lines[-2].endswith("libringattn_dbg.so") and lines[-1] == "1"
