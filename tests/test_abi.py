"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/*.h declares, and rejects bad arguments before it
touches CUDA."""
import ctypes
import glob
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def lib():
    from dense_fp32_matrix_sm_gb300 import build as b

    b.build()
    import dense_fp32_matrix_sm_gb300 as s

    return s.lib()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"\b(sgemm_\w+)\s*\(", text):
            names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_functions()
    assert "sgemm_plan" in declared and "sgemm_run" in declared
    missing = [n for n in sorted(declared) if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_header():
    from dense_fp32_matrix_sm_gb300._lib import SIGNATURES

    assert set(SIGNATURES) == _declared_functions()


def test_invalid_arguments_rejected_without_gpu(lib):
    h = ctypes.c_void_p()
    bad = [
        (-1, 4, 4, 4, 4, 4),    # negative M
        (4, -1, 4, 4, 4, 4),    # negative N
        (4, 4, -2, 4, 4, 4),    # negative K
        (4, 4, 8, 7, 4, 4),     # lda < K
        (4, 8, 4, 4, 7, 8),     # ldb < N
        (4, 8, 4, 4, 8, 7),     # ldc < N
        (4, 4, 0, 0, 4, 4),     # lda < 1
    ]
    for args in bad:
        assert lib.sgemm_plan(*args, ctypes.byref(h)) == -1, args
        assert not h.value
    assert lib.sgemm_plan(2 ** 31, 4, 4, 4, 4, 4, ctypes.byref(h)) == -2
    assert lib.sgemm_plan(4, 4, 4, 4, 4, 4, None) == -1
    assert lib.sgemm_plan_with_config(4, 4, 4, 4, 4, 4, -1, ctypes.byref(h)) == -1
    assert lib.sgemm_plan_with_config(4, 4, 4, 4, 4, 4, 10 ** 6, ctypes.byref(h)) == -1
    # run / describe / destroy on a NULL plan
    assert lib.sgemm_run(None, 1.0, None, None, 0.0, None, None) == -1
    assert lib.sgemm_run_host(None, 1.0, None, None, 0.0, None, None, None, None, None) == -1
    assert lib.sgemm_plan_describe(None, ctypes.create_string_buffer(8), 8) == -1
    assert lib.sgemm_plan_destroy(None) == 0


def test_plan_ex_batched_rejects_before_cuda(lib):
    """sgemm_plan_ex_batched checks the batch, strides and order before any CUDA call."""
    h = ctypes.c_void_p()
    f = lib.sgemm_plan_ex_batched
    ok = (0, 0, 0, 64, 32, 16, 16, 32, 32)
    assert f(*ok, -1, 0, 0, 0, -1, ctypes.byref(h)) == -1                 # negative batch
    assert f(*ok, 4, -4, 0, 2048, -1, ctypes.byref(h)) == -1              # negative stride
    assert f(*ok, 4, 0, 0, 2047, -1, ctypes.byref(h)) == -1               # row-major C overlap: needs 63*32+32
    assert f(1, 0, 0, 64, 32, 16, 64, 16, 64, 4, 0, 0, 2047, -1, ctypes.byref(h)) == -1  # column-major: 31*64+64
    assert f(*ok, 65536, 0, 0, 2048, -1, ctypes.byref(h)) == -2           # more products than a grid dimension
    assert f(*ok, 4, 0, 0, 2048, -2, ctypes.byref(h)) == -1               # bad config id
    assert f(2, 0, 0, 64, 32, 16, 16, 32, 32, 4, 0, 0, 2048, -1, ctypes.byref(h)) == -1  # bad order
    assert f(*ok, 4, 0, 0, 2048, -1, None) == -1                          # no output
    assert not h.value


def test_plan_ex_rejects_before_cuda(lib):
    """sgemm_plan_ex checks order, flags and stored leading dimensions before any CUDA call."""
    h = ctypes.c_void_p()
    f = lib.sgemm_plan_ex
    assert f(2, 0, 0, 8, 8, 8, 8, 8, 8, -1, ctypes.byref(h)) == -1        # bad order
    assert f(0, 3, 0, 8, 8, 8, 8, 8, 8, -1, ctypes.byref(h)) == -1        # bad transa
    assert f(0, 1, 0, 64, 32, 16, 63, 32, 32, -1, ctypes.byref(h)) == -1  # row-major A^T (K x M) needs lda >= M
    assert f(0, 0, 1, 64, 32, 16, 16, 15, 32, -1, ctypes.byref(h)) == -1  # row-major B^T (N x K) needs ldb >= K
    assert f(1, 0, 0, 64, 32, 16, 63, 16, 64, -1, ctypes.byref(h)) == -1  # column-major A (M x K) needs lda >= M
    assert f(1, 0, 0, 64, 32, 16, 64, 16, 63, -1, ctypes.byref(h)) == -1  # column-major C needs ldc >= M
    assert f(0, 0, 0, -1, 32, 16, 16, 32, 32, -1, ctypes.byref(h)) == -1  # negative M
    assert f(0, 0, 0, 8, 8, 8, 8, 8, 8, -1, None) == -1                   # no output
    assert not h.value


def test_spans_beyond_any_memory_are_refused_before_cuda(lib):
    """A stored matrix, or a strided batch of them, spanning more than 2^40
    elements (4 TiB of floats) cannot describe a real buffer: every plan
    entry refuses it with SGEMM_ERR_UNSUPPORTED before any CUDA call."""
    h = ctypes.c_void_p()
    big = 2 ** 20
    # row-major A, B, C in turn spanning (rows - 1) * ld + cols = 2^40 + 2^20
    assert lib.sgemm_plan(big + 1, 4, big, big, 4, 4, ctypes.byref(h)) == -2
    assert lib.sgemm_plan(4, big, big + 1, big + 1, big, big, ctypes.byref(h)) == -2
    assert lib.sgemm_plan(big + 1, big, 4, 4, big, big, ctypes.byref(h)) == -2
    # a strided batch: A 2^41 floats apart
    assert lib.sgemm_plan_batched(64, 64, 64, 64, 64, 64, 2, 2 ** 41, 4096, 4096, -1, ctypes.byref(h)) == -2
    # column-major A given transposed: M columns of K, lda apart
    assert lib.sgemm_plan_ex(1, 1, 0, big + 1, 4, big, big, big, big + 1, -1, ctypes.byref(h)) == -2
    # a strided batch of row-major C matrices 2^41 floats apart
    assert lib.sgemm_plan_ex_batched(0, 0, 0, 64, 32, 16, 16, 32, 32, 2, 0, 0, 2 ** 41, -1, ctypes.byref(h)) == -2
    assert not h.value
    dummy = 4096  # never dereferenced
    assert lib.sgemm_run_static_scratch(big + 1, 8, big, big, 8, 8, 1.0, dummy, dummy, 0.0, dummy, None) == -2


def test_autotune_rejects_bad_arguments_before_cuda(lib):
    h = ctypes.c_void_p()
    f = lib.sgemm_plan_autotune
    assert f(64, 64, 64, 63, 64, 64, 16, 16, 16, 0, None, None, ctypes.byref(h)) == -1   # lda < K
    assert f(64, 64, 64, 64, 64, 64, 16, 16, 16, 4, None, None, ctypes.byref(h)) == -1   # unknown flag
    assert f(64, 64, 64, 64, 64, 64, None, 16, 16, 0, None, None, ctypes.byref(h)) == -1  # no scratch A
    assert f(64, 64, 64, 64, 64, 64, 16, 16, 16, 0, None, None, None) == -1              # no output


def test_probe_rejects_bad_arguments_before_cuda(lib):
    t = ctypes.c_double()
    assert lib.sgemm_probe_ffma(1, None, ctypes.byref(t)) == -1
    assert lib.sgemm_probe_ffma(2, ctypes.byref(t), ctypes.byref(t)) == -1


def test_static_scratch_rejects_before_cuda(lib):
    """sgemm_run_static_scratch checks its arguments before any CUDA call."""
    f = lib.sgemm_run_static_scratch
    dummy = 4096  # never dereferenced: every case returns before a launch
    assert f(-1, 4, 4, 4, 4, 4, 1.0, dummy, dummy, 0.0, dummy, None) == -1   # negative M
    assert f(4, 8, 8, 7, 8, 8, 1.0, dummy, dummy, 0.0, dummy, None) == -1    # lda < K
    assert f(4, 8, 8, 8, 8, 8, 1.0, dummy, dummy, 0.0, None, None) == -1     # C missing
    assert f(4, 8, 8, 8, 8, 8, 1.0, None, dummy, 0.0, dummy, None) == -1     # A missing with a product
    assert f(0, 8, 8, 8, 8, 8, 1.0, None, None, 0.0, None, None) == 0        # M == 0: nothing to do
    assert f(4, 8, 8, 10, 8, 8, 1.0, dummy, dummy, 0.0, dummy, None) == -2   # lda % 4 != 0
    assert f(4, 8, 8, 8, 10, 8, 1.0, dummy, dummy, 0.0, dummy, None) == -2   # ldb % 4 != 0
    assert f(4, 8, 8, 8, 8, 8, 1.0, dummy + 4, dummy, 0.0, dummy, None) == -2  # A not 16-byte aligned
    assert f(2 ** 31, 8, 8, 8, 8, 8, 1.0, dummy, dummy, 0.0, dummy, None) == -2  # M beyond int32


def test_status_strings_and_configs(lib):
    import dense_fp32_matrix_sm_gb300 as s

    for code in (0, -1, -2, -3, -4, -5):
        assert s.status_string(code).startswith("SGEMM_")
    assert "unknown" in s.status_string(7)
    names = s.config_names()
    assert len(names) == s.num_configs() >= 2
    assert len(set(names)) == len(names)
    assert names[0].startswith("generic")
    assert any(n.startswith("tma_") for n in names)
    assert s.config_name(-1) is None
    assert lib.sgemm_set_wait_timeout_ns(0) == 0


def test_product_path_has_no_oracle_or_fallback():
    """The library package never imports the oracle and has no CPU path."""
    pkg = os.path.join(ROOT, "dense_fp32_matrix_sm_gb300")
    for path in glob.glob(os.path.join(pkg, "**", "*.py"), recursive=True):
        text = open(path).read()
        assert "import oracle" not in text and "from oracle" not in text, path
        assert "torch.matmul" not in text and "np.matmul" not in text, path


def test_wait_limit_follows_the_work():
    """The in-kernel wait limit of a launch is the larger of the process-wide
    setting (default 4 s) and the time the product would take at 1e10 FLOP/s
    per SM.  Values worked by hand: 2 * 4096^3 / (152 * 1e10) s = 0.0904 s,
    under the 4 s default; 2 * 65536^3 / (152 * 1e10) s = 370.3 s."""
    import dense_fp32_matrix_sm_gb300 as sg

    assert sg.wait_limit_ns(4096, 4096, 4096, 1, 152) == 4_000_000_000
    big = sg.wait_limit_ns(65536, 65536, 65536, 1, 152)
    assert abs(big - 2 * 65536 ** 3 / (152 * 1e10) * 1e9) < 1e3 and 370e9 < big < 371e9
    # the batch multiplies the work; fewer SMs raise the floor in proportion
    assert sg.wait_limit_ns(16384, 16384, 16384, 8, 152) == sg.wait_limit_ns(32768, 32768, 16384, 2, 152)
    assert abs(sg.wait_limit_ns(65536, 65536, 65536, 1, 76) - 2 * big) < 1e3
    # empty products take the setting
    assert sg.wait_limit_ns(0, 4096, 4096, 1, 152) == 4_000_000_000
    try:
        sg.set_wait_timeout_ns(10 ** 12)  # a longer setting wins over a smaller floor
        assert sg.wait_limit_ns(4096, 4096, 4096, 1, 152) == 10 ** 12
        assert sg.wait_limit_ns(65536, 65536, 65536, 1, 152) == 10 ** 12
    finally:
        sg.set_wait_timeout_ns(0)
    assert sg.wait_limit_ns(4096, 4096, 4096, 1, 152) == 4_000_000_000
    for bad in ((-1, 4, 4, 1, 152), (4, 4, 4, -1, 152), (4, 4, 4, 1, 0)):
        with pytest.raises(sg.SgemmError):
            sg.wait_limit_ns(*bad)
