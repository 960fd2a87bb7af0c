"""The checked build: libsgemm_gb300_checked.so, the same sources compiled
with -DSGEMM_CHECKED.  Its kernels test every hand-computed shared-memory
and workspace index before the access; a failure sets a bit of the status
word (reported as SGEMM_ERR_BOUNDS) and skips the access, where the normal
build would read or write out of range.  The GPU parity tests run against
it in a child process (SGEMM_GB300_LIBRARY=checked): every run there checks
device_status() == SGEMM_OK and oracle parity, so an index that leaves its
buffer on any of those shapes fails the test instead of corrupting memory.
This stands in for compute-sanitizer, which is closed on this machine."""
import os
import subprocess
import sys

import pytest

from conftest import ROOT


def test_checked_build_compiles():
    """The checked build links and exports the same entry points (no GPU)."""
    from dense_fp32_matrix_sm_gb300 import build as b

    path = b.build(checked=True)
    assert path.endswith("libsgemm_gb300_checked.so") and os.path.exists(path)
    out = subprocess.run([sys.executable, "-c", "import dense_fp32_matrix_sm_gb300 as s; l = s.lib(); "
                          "print(s._lib.LIB_PATH); print(all(hasattr(l, n) for n in s._lib.SIGNATURES))"],
                         cwd=ROOT, env=dict(os.environ, SGEMM_GB300_LIBRARY="checked"), capture_output=True,
                         text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = out.stdout.split()
    assert lines[0].endswith("libsgemm_gb300_checked.so") and lines[1] == "True", out.stdout


@pytest.mark.gpu
def test_parity_suite_on_the_checked_build():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_matrix_sm_gb300 import build as b

    b.build(checked=True)
    # everything but the largest problems (full-size 8192 x 14336 x 4096 and
    # the C of more than 2^31 elements) and the timing-driven autotuner
    sel = "not workload_full_size and not beyond_2_31 and not autotune and not full_size_sample"
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_gpu_parity.py"), "-m", "gpu",
                        "-q", "-x", "-k", sel, "-p", "no:cacheprovider"],
                       cwd=ROOT, env=dict(os.environ, SGEMM_GB300_LIBRARY="checked"), capture_output=True, text=True,
                       timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout, r.stdout[-2000:]
