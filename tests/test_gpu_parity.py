"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Bar (elementwise): |C_gpu - C_ref| <= 4*K*2^-24*(|A||B|)_ij + 1e-6.
Full comparison up to 1024^3-sized work; above that, a 65,536-entry
cross-product sample (rows x columns that always include both ends and one
index inside every edge tile).  Kernels that keep ascending-k order are also
compared bit for bit against the float32 fused-multiply-add chain when
alpha = 1 and beta = 0.
"""
import ctypes

import numpy as np
import pytest

import oracle
from dense_fp32_matrix_sm_gb300.inputs import (WORKLOADS, make_inputs, sample_rows_cols,
                                               workload_inputs)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

# The bar has one definition, oracle.acceptance_bound, pinned by a
# hand-computed value in test_oracle_pins.py.
_bound = oracle.acceptance_bound


@pytest.fixture(scope="module")
def sg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import os

    from dense_fp32_matrix_sm_gb300 import build as b

    # SGEMM_GB300_LIBRARY=checked: these tests run against the checked build
    # (tests/test_zy_checked_build.py), whose bounds failures show in device_status()
    b.build(checked=os.environ.get("SGEMM_GB300_LIBRARY") == "checked")
    import dense_fp32_matrix_sm_gb300 as s

    s.lib()
    return s


def _to_dev(x, ld=None, offset=0, fill=0.0):
    """Copy a 2-D float32 array to a device buffer with row stride ld
    (>= cols), starting `offset` floats into the allocation.  Returns
    (buffer, view-pointer, ld)."""
    rows, cols = x.shape
    ld = ld or max(1, cols)
    n = offset + (rows - 1) * ld + cols if rows > 0 else offset + 1
    buf = torch.full((max(n, 1),), fill, dtype=torch.float32, device="cuda")
    if rows > 0 and cols > 0:
        host = torch.full((max(n, 1),), fill, dtype=torch.float32)
        view = host[offset:offset + rows * ld].view(rows, ld) if rows * ld + offset <= host.numel() else None
        if view is None:
            for r in range(rows):
                host[offset + r * ld: offset + r * ld + cols] = torch.from_numpy(x[r])
        else:
            view[:, :cols] = torch.from_numpy(x)
        buf.copy_(host)
    return buf, buf.data_ptr() + 4 * offset, ld


def _from_dev(buf, rows, cols, ld, offset=0):
    host = buf.cpu().numpy()
    out = np.empty((rows, cols), np.float32)
    for r in range(rows):
        out[r] = host[offset + r * ld: offset + r * ld + cols]
    return out


def run_gpu(sg, A, B, C0, alpha, beta, config=None, lda=None, ldb=None, ldc=None, off_a=0, off_b=0,
            off_c=0, c_fill=None):
    M, K = A.shape
    N = B.shape[1]
    dA, pA, lda = _to_dev(A, lda, off_a)
    dB, pB, ldb = _to_dev(B, ldb, off_b)
    c_src = C0 if c_fill is None else np.full((M, N), c_fill, np.float32)
    dC, pC, ldc = _to_dev(c_src, ldc, off_c)
    plan = sg.Plan(M, N, K, lda, ldb, ldc, config=config)
    plan.run(alpha, pA, pB, beta, pC)
    torch.cuda.synchronize()
    assert sg.device_status() == sg.SGEMM_OK
    out = _from_dev(dC, M, N, ldc, off_c)
    name = plan.config_name
    run_gpu.last_info = plan.info()
    plan.close()
    return out, name


def assert_parity(C, Cref, S, K, what=""):
    C = C.astype(np.float64)
    assert C.shape == Cref.shape
    finite = np.isfinite(Cref)
    assert np.array_equal(np.isfinite(C), finite), f"{what}: non-finite mismatch"
    err = np.abs(C - Cref)[finite]
    bnd = _bound(K, S)[finite]
    bad = err > bnd
    if bad.any():
        idx = np.argmax(err / bnd)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} entries outside the bound; worst "
                             f"err {err[idx]:.3e} vs bound {bnd[idx]:.3e}")


def _variants(sg, M=None):
    """Variant names, without the few-row kernels when M is above their limits."""
    names = sg.config_names()
    if M is not None and M > 16:
        names = [n for n in names if not n.startswith("skinny")]
    if M is not None and M > 4:
        names = [n for n in names if not n.startswith("gemv")]
    return names


# ---- small and ragged shapes, every variant, full comparison ------------------

SWEEP = [1, 2, 3, 4, 5, 7, 8, 15, 16, 17, 31, 33, 63, 65, 127, 129, 255, 257]


def _shape_cases(n=40, seed=0):
    rng = np.random.default_rng(seed)
    cases = {(1, 1, 1), (257, 257, 257), (1, 257, 257), (257, 1, 257), (257, 257, 1), (128, 128, 128),
             (129, 127, 33), (16, 300, 129)}
    while len(cases) < n:
        cases.add(tuple(int(x) for x in rng.choice(SWEEP, 3)))
    return sorted(cases)


@pytest.mark.parametrize("variant_idx", range(48))
def test_shape_sweep_every_variant(sg, oracle_mod, variant_idx):
    names = _variants(sg)
    if variant_idx >= len(names):
        pytest.skip("fewer variants in this build")
    name = names[variant_idx]
    ran = 0
    for (M, N, K) in _shape_cases(36, seed=variant_idx):
        for alpha, beta in ((1.0, 0.0), (0.5, 3.0)):
            A, B, C0 = make_inputs(M, N, K, seed=M * 7 + N * 3 + K, dist_a=("normal", 1.0),
                                   dist_b=("uniform", 1.0))
            try:
                # row strides padded to multiples of 4 so the TMA variants accept every shape
                C, used = run_gpu(sg, A, B, C0, alpha, beta, config=name, lda=(K + 3) // 4 * 4 or 4,
                                  ldb=(N + 3) // 4 * 4)
            except sg.SgemmError as e:
                if e.status == sg.SGEMM_ERR_UNSUPPORTED:
                    break
                raise
            ran += 1
            Cref, S = oracle_mod.sgemm_ref(A, B, C0, alpha, beta)
            assert_parity(C, Cref, S, K, f"{name} {M}x{N}x{K} a={alpha} b={beta}")
            if alpha == 1.0 and beta == 0.0 and run_gpu.last_info.get("k_order") == "sequential":
                ii, jj = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
                chain = oracle_mod.fp32_chain_entries(A, B, ii.ravel(), jj.ravel()).reshape(M, N)
                assert np.array_equal(C, chain), f"{name} {M}x{N}x{K}: not the ascending-k fp32 chain"
    # every variant takes some of the shapes: none passes by refusing them all
    assert ran >= 4, f"{name} ran on {ran} of the sweep's shapes"


@pytest.mark.parametrize("shape", [(1024, 1024, 1024), (1000, 1100, 999), (300, 2000, 517)])
def test_medium_full_compare(sg, oracle_mod, shape):
    M, N, K = shape
    A, B, C0 = make_inputs(M, N, K, seed=sum(shape), dist_a=("normal", 1.0), dist_b=("normal", 1.0))
    Cref, S = oracle_mod.sgemm_ref(A, B, C0, 0.5, 3.0)
    C, _ = run_gpu(sg, A, B, C0, 0.5, 3.0)
    assert_parity(C, Cref, S, K, f"table {shape}")


# ---- few rows: the cluster split-K kernel ---------------------------------------

SKINNY_CASES = [(16, 16384 // 8, 8192 // 4), (1, 300, 1000), (7, 129, 33), (16, 128, 32), (13, 1000, 4097),
                (16, 2048, 96), (3, 5000, 8), (16, 77, 1), (9, 4096, 2000),
                # stream-K few-row kernel: ranges covering whole slabs (600 slabs x 2 k-slices),
                # one unit per CTA with 128 contributors per slab, and ragged N and K
                (16, 76800, 64), (16, 384, 4096), (5, 1000, 3000)]


@pytest.mark.parametrize("shape", SKINNY_CASES)
def test_skinny_variants(sg, oracle_mod, shape):
    M, N, K = shape
    A, B, C0 = make_inputs(M, N, K, seed=M + N + K, dist_a=("normal", 1.0), dist_b=("normal", 0.02))
    lda, ldb = (K + 3) // 4 * 4, (N + 3) // 4 * 4
    for name in [n for n in sg.config_names() if n.startswith("skinny")] + ["gemv_16x1024", None]:
        for alpha, beta in ((1.0, 0.0), (1.0, 1.0), (-0.75, 2.0)):
            try:
                C, used = run_gpu(sg, A, B, C0, alpha, beta, config=name, lda=lda, ldb=ldb)
            except sg.SgemmError as e:
                if e.status == sg.SGEMM_ERR_UNSUPPORTED and name is not None:
                    break  # this few-row variant does not take this shape
                raise
            info = run_gpu.last_info
            if name is None:
                # the table: one to four rows and (B of 16 MB or more) up to sixteen rows stream B
                # through the matrix-vector kernels, the rest take the few-row kernels
                expect = "gemv_4x512" if M <= 4 else "gemv_16x1024" if N * K >= 1 << 22 else "skinny"
                assert used.startswith(expect), (used, expect)
            Cref, S = oracle_mod.sgemm_ref(A, B, C0, alpha, beta)
            assert_parity(C, Cref, S, K, f"{used} {shape} split={info['split']} a={alpha} b={beta}")
            # a fixed reduction order: the same inputs give the same bits again
            C2, _ = run_gpu(sg, A, B, C0, alpha, beta, config=name, lda=lda, ldb=ldb)
            assert np.array_equal(C, C2)


def test_skinny_rejects_tall_m(sg):
    name = next(n for n in sg.config_names() if n.startswith("skinny"))
    with pytest.raises(sg.SgemmError) as e:
        sg.Plan(17, 256, 256, config=name)
    assert e.value.status == sg.SGEMM_ERR_UNSUPPORTED


# ---- layouts: leading dimensions, misaligned pointers, guard bands ------------

@pytest.mark.parametrize("lds", [(0, 0, 0), (4, 8, 12), (1, 0, 0), (0, 3, 0), (0, 0, 5), (7, 9, 11)])
@pytest.mark.parametrize("shape", [(200, 188, 148), (100, 96, 1000)])
def test_leading_dimensions(sg, oracle_mod, lds, shape):
    M, N, K = shape
    A, B, C0 = make_inputs(M, N, K, seed=3)
    Cref, S = oracle_mod.sgemm_ref(A, B, C0, 1.5, -0.5)
    C, used = run_gpu(sg, A, B, C0, 1.5, -0.5, lda=K + lds[0], ldb=N + lds[1], ldc=N + lds[2])
    assert_parity(C, Cref, S, K, f"ld pads {lds} ({used})")
    if K <= 512:
        assert used == "tiny_32x32", used      # tiny products: whole K-panels, any leading dimension
    elif lds[1] % 4:
        assert used.startswith("generic")      # B's rows are not 16-byte multiples: scalar loads
    elif lds[0] % 4:
        assert used.startswith("cpa")          # A copied 4 bytes at a time: any lda


@pytest.mark.parametrize("config", ["tiny_32x32", "small_64x64"])
@pytest.mark.parametrize("shape", [(32, 32, 256), (31, 33, 257), (100, 70, 511), (64, 96, 512), (512, 512, 512),
                                   (45, 200, 300), (130, 65, 1000)])
def test_tiny_k_chunks(sg, oracle_mod, config, shape):
    # K streamed in 64-deep chunks through the ring (one chunk, several, a
    # ragged last one); 16-byte copies, then 4-byte copies (odd lda), and a
    # strided batch of the same shape
    M, N, K = shape
    A, B, C0 = make_inputs(M, N, K, seed=M * 7 + K, dist_a=("normal", 1.0), dist_b=("normal", 1.0))
    for lda, alpha, beta in ((K + (-K) % 4, 1.0, 0.0), (K + 1, -0.5, 2.0)):
        C, used = run_gpu(sg, A, B, C0, alpha, beta, config=config, lda=lda)
        Cref, S = oracle_mod.sgemm_ref(A, B, C0, alpha, beta)
        assert_parity(C, Cref, S, K, f"{config} {shape} lda={lda}")
        C2, _ = run_gpu(sg, A, B, C0, alpha, beta, config=config, lda=lda)
        assert np.array_equal(C, C2)
    if M * N <= 64 * 96:
        batch = 3
        As = np.stack([A * (z + 1) for z in range(batch)])
        Bs = np.stack([B - z for z in range(batch)])
        Cs0 = np.stack([C0 + z for z in range(batch)])
        dA, dB, dC = (torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (As, Bs, Cs0))
        plan = sg.Plan(M, N, K, config=config, batch=batch, stride_a=M * K, stride_b=K * N, stride_c=M * N)
        try:
            plan.run(1.0, dA, dB, 1.0, dC)
            torch.cuda.synchronize()
            assert sg.device_status() == 0
        finally:
            plan.close()
        out = dC.cpu().numpy()
        for z in range(batch):
            Cref, S = oracle_mod.sgemm_ref(As[z], Bs[z], Cs0[z], 1.0, 1.0)
            assert_parity(out[z], Cref, S, K, f"{config} batch {z} {shape}")


@pytest.mark.parametrize("case", [
    # (M, N, K, the table's variant): 17 to 64 rows past the tiny kernel's K <= 512 range
    (32, 4096, 4096, "tiny_32x32"),        # 128 tiles of 32 x 32: K streamed, no split
    (30, 4000, 700, "tiny_32x32"),
    (20, 3000, 2000, "tmat_64x256x32_s3_b1"),  # 94 tiles: too few for the tiny kernel, which does not split K
    (48, 4096, 4096, "tmat_64x256x32_s3_b1"),
    (64, 1000, 1500, "tmat_64x256x32_s3_b1"),  # ragged N and K
    (40, 700, 3001, "tmat_64x256x32_s3_b1"),
    (65, 4096, 4096, None),                # more than 64 rows: the 128-row tiles
    (768, 768, 512, "small_64x64"),        # a short k loop, at most two 64 x 64 tiles per SM
    (1000, 1100, 333, "small_64x64"),
])
def test_seventeen_to_sixtyfour_rows(sg, oracle_mod, case):
    M, N, K, expect = case
    plan = sg.Plan(M, N, K)
    used = plan.info()["variant"]
    plan.close()
    if expect is None:
        assert used.startswith("tmat_128"), used
    else:
        assert used == expect, (used, expect)
    A, B, C0 = make_inputs(M, N, K, seed=M + N + K, dist_a=("normal", 1.0), dist_b=("normal", 1.0))
    for alpha, beta in ((1.0, 0.0), (0.5, -2.0)):
        C, used2 = run_gpu(sg, A, B, C0, alpha, beta)
        assert used2 == used
        Cref, S = oracle_mod.sgemm_ref(A, B, C0, alpha, beta)
        assert_parity(C, Cref, S, K, f"{used} {case} a={alpha} b={beta}")
    C2, _ = run_gpu(sg, A, B, C0, 0.5, -2.0)
    assert np.array_equal(C, C2)


@pytest.mark.parametrize("offs", [(1, 0, 0), (0, 1, 0), (0, 0, 1), (2, 3, 1)])
def test_misaligned_pointers(sg, oracle_mod, offs):
    M, N, K = 140, 260, 96
    A, B, C0 = make_inputs(M, N, K, seed=5)
    Cref, S = oracle_mod.sgemm_ref(A, B, C0, 1.0, 1.0)
    for name in _variants(sg, M):
        try:
            C, _ = run_gpu(sg, A, B, C0, 1.0, 1.0, config=name, off_a=offs[0], off_b=offs[1], off_c=offs[2])
        except sg.SgemmError as e:
            # the fused split-TF32 form reads A and B by TMA as stored and
            # refuses unaligned bases; every other variant must fall back
            assert name.startswith("tf32x3f") and e.status == sg.SGEMM_ERR_UNSUPPORTED, name
            assert offs[0] or offs[1]
            continue
        assert_parity(C, Cref, S, K, f"{name} offsets {offs}")


@pytest.mark.parametrize("pads", [(1, 0), (0, 1), (1, 3)])
def test_unaligned_leading_dimensions_are_repacked(sg, oracle_mod, pads):
    """From 256^3 of work on, an operand whose rows are not 16-byte multiples
    is copied into padded rows each run, so the TMA kernels still serve it."""
    M, N, K = 700, 600, 520
    lda, ldb = K + pads[0], N + pads[1]
    A, B, C0 = make_inputs(M, N, K, seed=91 + pads[1], dist_a=("normal", 1.0), dist_b=("normal", 1.0))
    Cref, S = oracle_mod.sgemm_ref(A, B, C0, 0.75, -0.5)
    C, used = run_gpu(sg, A, B, C0, 0.75, -0.5, lda=lda, ldb=ldb)
    info = run_gpu.last_info
    assert info["repack"] == (1 if lda % 4 else 0) | (2 if ldb % 4 else 0), info
    assert used.startswith("tmat"), used
    assert_parity(C, Cref, S, K, f"repacked lda={lda} ldb={ldb} {used}")
    # the same storage read as column-major: C^T = B^T A^T, operands swapped
    memA, memB = _stored(A, "col", False, 0), _stored(B, "col", False, 0)
    dA, pA, _ = _to_dev(memA[0], M + pads[0])
    dB, pB, _ = _to_dev(memB[0], K + pads[1])
    memC, ldc = _stored(C0, "col", False, 0)
    dC, pC, _ = _to_dev(memC, ldc)
    plan = sg.Plan(M, N, K, M + pads[0], K + pads[1], ldc, order="col")
    assert plan.info()["repack"] == (1 if (M + pads[0]) % 4 else 0) | (2 if (K + pads[1]) % 4 else 0), plan.info()
    plan.run(0.75, pA, pB, -0.5, pC)
    torch.cuda.synchronize()
    assert sg.device_status() == sg.SGEMM_OK
    Cc = _from_dev(dC, memC.shape[0], memC.shape[1], ldc).T
    plan.close()
    assert_parity(Cc, Cref, S, K, f"column-major repacked {pads}")


@pytest.mark.parametrize("ldc_pad", [7, 4])
def test_guard_bands_untouched(sg, ldc_pad):
    M, N, K = 131, 132, 76
    A, B, C0 = make_inputs(M, N, K, seed=9)
    sentinel = 12345.0
    ldc = N + ldc_pad
    off = 3 * ldc + 4
    total = off + (M - 1) * ldc + N + 64
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    mask = np.ones(total, bool)
    for r in range(M):
        mask[off + r * ldc: off + r * ldc + N] = False
    for name in _variants(sg, M):
        for beta in (0.0, 1.0):
            dC = torch.full((total,), sentinel, dtype=torch.float32, device="cuda")
            plan = sg.Plan(M, N, K, K, N, ldc, config=name)
            plan.run(1.0, dA, dB, beta, dC.data_ptr() + 4 * off)
            torch.cuda.synchronize()
            out = dC.cpu().numpy()
            assert np.all(out[mask] == sentinel), f"{name} wrote outside C (ldc={ldc}, beta={beta})"
            plan.close()


# ---- degenerate cases ---------------------------------------------------------

def test_beta_zero_ignores_nan_c(sg, oracle_mod):
    M, N, K = 150, 172, 64
    A, B, C0 = make_inputs(M, N, K, seed=1)
    Cref, S = oracle_mod.sgemm_ref(A, B, None, 1.0, 0.0)
    for name in _variants(sg, M):
        C, _ = run_gpu(sg, A, B, C0, 1.0, 0.0, config=name, c_fill=np.nan)
        assert_parity(C, Cref, S, K, f"{name} beta=0 over NaN")


def test_alpha_zero_and_k_zero(sg, oracle_mod):
    M, N = 70, 90
    A, B, C0 = make_inputs(M, N, 33, seed=2)
    Cref, S = oracle_mod.sgemm_ref(A, B, C0, 0.0, -2.0)
    C, _ = run_gpu(sg, A, B, C0, 0.0, -2.0)
    assert_parity(C, Cref, S, 33, "alpha=0")
    A0 = np.zeros((M, 0), np.float32)
    B0 = np.zeros((0, N), np.float32)
    Cref, S = oracle_mod.sgemm_ref(A0, B0, C0, 1.0, 3.0)
    C, _ = run_gpu(sg, A0, B0, C0, 1.0, 3.0)
    assert_parity(C, Cref, S, 0, "K=0")
    C, _ = run_gpu(sg, A0, B0, C0, 1.0, 0.0)
    assert np.all(C == 0.0)


def test_empty_m_or_n(sg):
    for (M, N, K) in ((0, 5, 5), (5, 0, 5), (0, 0, 0)):
        plan = sg.Plan(M, N, K)
        plan.run(1.0, None, None, 0.0, None)
        assert plan.launches == 0
        plan.close()
    torch.cuda.synchronize()


def test_argument_errors_on_gpu(sg):
    plan = sg.Plan(8, 8, 8)
    with pytest.raises(sg.SgemmError) as e:
        plan.run(1.0, None, None, 0.0, None)
    assert e.value.status == sg.SGEMM_ERR_INVALID_ARG
    # the binding refuses host and non-float32 tensors before the library sees them
    dev = torch.zeros(8, 8, device="cuda")
    with pytest.raises(TypeError):
        plan.run(1.0, torch.zeros(8, 8), dev, 0.0, dev)
    with pytest.raises(TypeError):
        plan.run(1.0, dev, dev.half(), 0.0, dev)
    plan.close()
    with pytest.raises(sg.SgemmError) as e:
        sg.Plan(64, 64, 64, lda=65, config=next(n for n in sg.config_names() if n.startswith("tma_")))
    assert e.value.status == sg.SGEMM_ERR_UNSUPPORTED


# ---- the wait limit -------------------------------------------------------------

def test_wait_timeout_selftest(sg):
    assert sg.device_status() == sg.SGEMM_OK
    rc = sg.selftest_wait_timeout(2_000_000)          # 2 ms on a phase nobody completes
    assert rc == sg.SGEMM_ERR_TIMEOUT
    assert sg.device_status() == sg.SGEMM_OK           # the self-test cleared its bit
    # the context is still usable
    x = torch.ones(4, device="cuda")
    assert float(x.sum()) == 4.0


# ---- host-buffer entry point ------------------------------------------------------

def test_run_host_matches_device_path(sg, oracle_mod):
    M, N, K = 257, 300, 128
    A, B, C0 = make_inputs(M, N, K, seed=21)
    hA = torch.from_numpy(A).pin_memory()
    hB = torch.from_numpy(B).pin_memory()
    hC = torch.from_numpy(C0.copy()).pin_memory()
    dA = torch.empty_like(hA, device="cuda")
    dB = torch.empty_like(hB, device="cuda")
    dC = torch.empty_like(hC, device="cuda")
    plan = sg.Plan(M, N, K)
    plan.run_host(0.5, hA, hB, 3.0, hC, dA, dB, dC)
    torch.cuda.synchronize()
    Cdev, _ = run_gpu(sg, A, B, C0, 0.5, 3.0)
    assert np.array_equal(hC.numpy(), Cdev)
    Cref, S = oracle_mod.sgemm_ref(A, B, C0, 0.5, 3.0)
    assert_parity(hC.numpy(), Cref, S, K, "run_host")
    plan.close()


# ---- the five workloads at full size, in the launch configuration the bench times --

@pytest.mark.parametrize("wname", list(WORKLOADS))
def test_workload_full_size(sg, oracle_mod, wname):
    w = WORKLOADS[wname]
    A, B, C0 = workload_inputs(w)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dC = torch.from_numpy(C0).cuda()
    plan = sg.Plan(w.M, w.N, w.K)
    plan.run(w.alpha, dA, dB, w.beta, dC)
    torch.cuda.synchronize()
    assert sg.device_status() == sg.SGEMM_OK
    info = plan.info()
    plan.close()
    if w.M * w.N * w.K <= 1024 ** 3:
        C = dC.cpu().numpy()
        Cref, S = oracle_mod.sgemm_ref(A, B, C0, w.alpha, w.beta)
        assert_parity(C, Cref, S, w.K, wname)
        return
    rows, cols = sample_rows_cols(w.M, w.N, seed=w.seed)
    r_t = torch.from_numpy(rows).cuda()
    c_t = torch.from_numpy(cols).cuda()
    C = dC.index_select(0, r_t).index_select(1, c_t).cpu().numpy()
    As = np.ascontiguousarray(A[rows])
    Bs = np.ascontiguousarray(B[:, cols])
    Cs = np.ascontiguousarray(C0[np.ix_(rows, cols)])
    Cref, S = oracle_mod.sgemm_ref(As, Bs, Cs, w.alpha, w.beta)
    assert C.size >= 65536
    assert_parity(C, Cref, S, w.K, f"{wname} ({info['variant']})")
    if w.alpha == 1.0 and w.beta == 0.0 and info.get("k_order") == "sequential":
        sub_r = np.arange(0, len(rows), 4)
        ii, jj = np.meshgrid(sub_r, np.arange(len(cols)), indexing="ij")
        chain = oracle_mod.fp32_chain_entries(As, Bs, ii.ravel(), jj.ravel())
        assert np.array_equal(C[ii.ravel(), jj.ravel()], chain), f"{wname}: not the ascending-k chain"


def test_misaligned_and_guarded_few_rows(sg, oracle_mod):
    """The few-row kernels under a misaligned A (scalar-load fallback), a
    padded ldc and NaN in C with beta = 0."""
    M, N, K = 11, 700, 300
    A, B, C0 = make_inputs(M, N, K, seed=77)
    Cref, S = oracle_mod.sgemm_ref(A, B, None, 1.0, 0.0)
    for name in [n for n in sg.config_names() if n.startswith("skinny")] + ["gemv_16x1024"]:
        C, _ = run_gpu(sg, A, B, C0, 1.0, 0.0, config=name, ldc=N + 5, c_fill=np.nan)
        assert_parity(C, Cref, S, K, f"{name} nan C")
        C, used = run_gpu(sg, A, B, C0, 1.0, 0.0, config=name, off_a=1)
        assert_parity(C, Cref, S, K, f"{name} misaligned A -> {used}")


def test_transposed_a_variants_take_any_lda(sg, oracle_mod):
    """The kernels that copy A themselves accept any lda and any A alignment
    and stay on their own path (no scalar-load fallback)."""
    M, N, K = 190, 260, 133
    A, B, C0 = make_inputs(M, N, K, seed=31, dist_a=("normal", 1.0), dist_b=("normal", 1.0))
    Cref, S = oracle_mod.sgemm_ref(A, B, C0, 0.5, 3.0)
    for name in [n for n in sg.config_names() if n.startswith("cpa")]:
        for lda, off_a in ((K, 0), (K + 1, 0), (K + 3, 1)):
            C, used = run_gpu(sg, A, B, C0, 0.5, 3.0, config=name, lda=lda, off_a=off_a)
            assert used == name
            assert_parity(C, Cref, S, K, f"{name} lda={lda} off_a={off_a}")


TAIL_SHORTER_THAN_GRID = [(1152, 1152, 256), (1152, 2176, 256), (1152, 4352, 256)]


@pytest.mark.parametrize("shape", [(2048, 2048, 1024), (1500, 3000, 780), (2560, 1408, 256),
                                   # fewer tiles than CTA slots: every tile split along K
                                   (1024, 1024, 1024), (512, 520, 8200), (1000, 300, 3000),
                                   # a tail with fewer k-slices than CTAs (64 x 128 tiles: 10 x 8; 128 x 128
                                   # and 128 x 256 tiles: 1 x 8) runs as a plain partial wave
                                   (1152, 1152, 256), (1152, 2176, 256), (1152, 4352, 256)])
def test_stream_k_tail(sg, oracle_mod, shape):
    """Tile counts that overshoot the resident grid: full waves run
    data-parallel and the leftover tiles are split along K across all CTAs
    (partials through a workspace, added in CTA order).  With fewer tiles
    than CTA slots there is no data-parallel wave: every tile is split.
    Waits are limited to 0.5 s here, so a schedule that leaves a finisher
    waiting fails fast with SGEMM_ERR_TIMEOUT."""
    sg.set_wait_timeout_ns(500_000_000)
    try:
        _stream_k_tail(sg, oracle_mod, shape)
    finally:
        sg.set_wait_timeout_ns(0)  # back to the default


def _stream_k_tail(sg, oracle_mod, shape):
    M, N, K = shape
    A, B, C0 = make_inputs(M, N, K, seed=M + 3 * N + K, dist_a=("normal", 1.0), dist_b=("normal", 1.0))
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    names = [n for n in sg.config_names() if n.startswith("tmat")]
    saw_streamk = False
    for name in names:
        plan = sg.Plan(M, N, K, config=name)
        info = plan.info()
        outs = []
        for _ in range(3):  # three runs: three epochs on the same flags
            dC = torch.from_numpy(C0).cuda()
            plan.run(0.5, dA, dB, 3.0, dC)
            torch.cuda.synchronize()
            assert sg.device_status() == sg.SGEMM_OK
            outs.append(dC.cpu().numpy())
        plan.close()
        assert all(np.array_equal(outs[0], o) for o in outs[1:]), f"{name}: runs differ"
        if info["streamk"]:
            saw_streamk = True
            assert info["k_order"] == "split"
            if info["tiles"] < info["grid"]:
                assert info["dp_waves"] == 0, info
        rows, cols = sample_rows_cols(M, N, n_rows=192, n_cols=192, seed=7)
        Cs = outs[0][np.ix_(rows, cols)]
        Cref, S = oracle_mod.sgemm_ref(np.ascontiguousarray(A[rows]), np.ascontiguousarray(B[:, cols]),
                                       np.ascontiguousarray(C0[np.ix_(rows, cols)]), 0.5, 3.0)
        assert_parity(Cs, Cref, S, K, f"{name} {shape} streamk={info['streamk']} dp_waves={info['dp_waves']}")
    if shape not in TAIL_SHORTER_THAN_GRID:
        assert saw_streamk, "no variant split its tail for these shapes"


# ---- split-TF32 tensor-core variant (reported apart from the FFMA path) -------

TC = "tf32x3_128x256x32_s2"
TC_VARIANTS = ["tf32x3_128x256x32_s2", "tf32x3_128x128x32_s3", "tf32x3f_128x128x32_s3", "tf32x3p_128x128x32_s3",
               "tf32x3p_128x256x32_s2"]


@pytest.mark.parametrize("tc", TC_VARIANTS)
@pytest.mark.parametrize("case", [
    # (M, N, K, lda pad, ldb pad, ldc pad, A offset, B offset, alpha, beta, distribution)
    (1024, 1024, 1024, 0, 0, 0, 0, 0, 1.0, 0.0, "normal"),
    (1000, 1100, 999, 1, 3, 5, 1, 2, 0.5, 3.0, "normal"),
    (300, 2000, 517, 0, 0, 0, 0, 0, -1.25, 1.0, "normal"),
    (129, 257, 16, 0, 0, 0, 0, 0, 1.0, 0.0, "normal"),
    # all-positive inputs: partial sums grow to |A||B|, the worst case for accumulator rounding
    (512, 768, 4096, 0, 0, 0, 0, 0, 1.0, 0.0, "positive"),
])
def test_split_tf32_variant(sg, oracle_mod, case, tc):
    M, N, K, pa, pb, pc, oa, ob, alpha, beta, dist = case
    if tc.startswith("tf32x3f") and (pa % 4 or pb % 4 or oa % 4 or ob % 4 or K % 4 or N % 4):
        pytest.skip("the fused form reads A and B by TMA: 16-byte rows and bases")
    d = ("uniform", 1.0) if dist == "normal" else ("uniform", 1.0)
    A, B, C0 = make_inputs(M, N, K, seed=M + N + K, dist_a=("normal", 1.0) if dist == "normal" else d, dist_b=d)
    if dist == "positive":
        A, B = np.abs(A), np.abs(B)
    Cref, S = oracle_mod.sgemm_ref(A, B, C0, alpha, beta)
    C, used = run_gpu(sg, A, B, C0, alpha, beta, config=tc, lda=K + pa, ldb=N + pb, ldc=N + pc, off_a=oa,
                      off_b=ob)
    assert used == tc and run_gpu.last_info["k_order"] == "tf32x3"
    assert_parity(C, Cref, S, K, f"{tc} {M}x{N}x{K} {dist}")
    C2, _ = run_gpu(sg, A, B, C0, alpha, beta, config=tc, lda=K + pa, ldb=N + pb, ldc=N + pc, off_a=oa, off_b=ob)
    assert np.array_equal(C, C2)


def test_split_tf32_rejects_short_k(sg):
    with pytest.raises(sg.SgemmError) as e:
        sg.Plan(256, 256, 15, config=TC)
    assert e.value.status == sg.SGEMM_ERR_UNSUPPORTED
    plan = sg.Plan(256, 256, 16, config=TC)
    assert plan.launches == 3
    plan.close()


def test_split_tf32_full_size_sample(sg, oracle_mod):
    w = WORKLOADS["square4096"]
    A, B, C0 = workload_inputs(w)
    C, used = run_gpu(sg, A, B, C0, w.alpha, w.beta, config=TC)
    rows, cols = sample_rows_cols(w.M, w.N, tile_n=256, seed=5)
    Cref, S = oracle_mod.sgemm_ref(np.ascontiguousarray(A[rows]), np.ascontiguousarray(B[:, cols]),
                                   np.ascontiguousarray(C0[np.ix_(rows, cols)]), w.alpha, w.beta)
    assert_parity(C[np.ix_(rows, cols)], Cref, S, w.K, f"{TC} square4096 sample")


# ---- storage order and transposition (sgemm_plan_ex) --------------------------

def _stored(X, order, trans, pad):
    """Memory (row-major view) and leading dimension of logical operand X stored
    as X or X^T (trans) in `order`, each row/column padded by `pad` floats."""
    S = X.T if trans else X
    mem = S if order == "row" else S.T  # a column-major matrix is its transpose in row-major memory
    mem = np.ascontiguousarray(mem, dtype=np.float32)
    return mem, mem.shape[1] + pad


@pytest.mark.parametrize("order", ["row", "col"])
@pytest.mark.parametrize("ta,tb", [(False, False), (False, True), (True, False), (True, True)])
@pytest.mark.parametrize("shape,config,pad", [((257, 131, 77), None, 0), ((200, 300, 100), None, 3),
                                              ((12, 1000, 515), None, 0), ((300, 520, 96), "tf32x3_128x256x32_s2", 1),
                                              ((300, 520, 96), "tf32x3f_128x128x32_s3", 0),
                                              ((16, 8192, 4096), None, 0),
                                              ((7, 1000, 520), "skinny_sk_16x128x32_w4_s3_b3_ef", 0),
                                              # transposed-A kernels: 128x64, 128x128, 128x256 stream-K;
                                              # A given transposed is read natively (no transpose launch)
                                              ((1000, 1100, 520), None, 0), ((2048, 2048, 1024), None, 0),
                                              ((2560, 2560, 512), None, 0), ((1000, 1100, 520), None, 1)])
def test_order_and_transpose(sg, oracle_mod, order, ta, tb, shape, config, pad):
    M, N, K = shape
    if config and config.startswith("skinny") and order == "col":
        pytest.skip("column-major swaps M and N: not a few-row product")
    opA, opB, C0 = make_inputs(M, N, K, seed=M + 2 * N + 3 * K + ta + 2 * tb, dist_a=("normal", 1.0),
                               dist_b=("normal", 1.0))
    alpha, beta = 0.75, -1.5
    Cref, S = oracle_mod.sgemm_ref(opA, opB, C0, alpha, beta)
    memA, lda = _stored(opA, order, ta, pad)
    memB, ldb = _stored(opB, order, tb, pad)
    memC, ldc = _stored(C0, order, False, pad)
    dA, pA, _ = _to_dev(memA, lda)
    dB, pB, _ = _to_dev(memB, ldb)
    dC, pC, _ = _to_dev(memC, ldc)
    plan = sg.Plan(M, N, K, lda, ldb, ldc, config=config, order=order, transa=ta, transb=tb)
    info = plan.info()
    assert info["order"] == order and info["op"] == ("T" if ta else "N") + ("T" if tb else "N")
    assert info["M"] == M and info["N"] == N
    if info["variant"].startswith("tmat"):
        # column-major runs the row-major product of the swapped operands, so the
        # product's A is given transposed when (row) transa or (column) transb;
        # it is read natively when its stored row length is a multiple of 4
        a_side_transposed = ta if order == "row" else tb
        b_side_transposed = tb if order == "row" else ta
        native_a = a_side_transposed and (lda if order == "row" else ldb) % 4 == 0
        # plus one padding copy per untransposed operand with unaligned rows (repack bits)
        expected = 1 + (a_side_transposed and not native_a) + b_side_transposed + bin(info["repack"]).count("1")
        assert plan.launches == expected, (plan.launches, expected, info)
    plan.run(alpha, pA, pB, beta, pC)
    torch.cuda.synchronize()
    assert sg.device_status() == sg.SGEMM_OK
    out = _from_dev(dC, memC.shape[0], memC.shape[1], ldc)
    C = out if order == "row" else out.T
    plan.close()
    assert_parity(C, Cref, S, K, f"{order} op={info['op']} {shape} {info['variant']}")


@pytest.mark.parametrize("config", [None, "tf32x3_128x128x32_s3"])
def test_transposed_operand_with_more_than_65535_row_tiles(sg, oracle_mod, config):
    """A stored K x M with K = 4.2 M, more than 65535 tiles of 32 rows: the
    transposing kernels walk row tiles past the grid's y limit."""
    M, N, K = 8, 8, 4_200_000
    opA, opB, C0 = make_inputs(M, N, K, seed=77, dist_a=("normal", 1.0), dist_b=("normal", 1.0))
    Cref, S = oracle_mod.sgemm_ref(opA, opB, C0, 1.0, 0.5)
    memA, lda = _stored(opA, "row", True, 0)
    memB, ldb = _stored(opB, "row", False, 0)
    dA, pA, _ = _to_dev(memA, lda)
    dB, pB, _ = _to_dev(memB, ldb)
    dC, pC, _ = _to_dev(C0, N)
    plan = sg.Plan(M, N, K, lda, ldb, N, config=config, transa=True)
    plan.run(1.0, pA, pB, 0.5, pC)
    torch.cuda.synchronize()
    assert sg.device_status() == sg.SGEMM_OK
    C = _from_dev(dC, M, N, N)
    variant = plan.info()["variant"]
    plan.close()
    assert_parity(C, Cref, S, K, f"TN K={K} {variant}")


def test_order_and_transpose_host_buffers(sg, oracle_mod):
    """sgemm_run_host copies each operand with its stored shape."""
    M, N, K = 150, 90, 70
    opA, opB, C0 = make_inputs(M, N, K, seed=31, dist_a=("normal", 1.0), dist_b=("normal", 1.0))
    Cref, S = oracle_mod.sgemm_ref(opA, opB, C0, 1.0, 2.0)
    memA, lda = _stored(opA, "col", True, 0)
    memB, ldb = _stored(opB, "col", False, 0)
    memC, ldc = _stored(C0, "col", False, 0)
    plan = sg.Plan(M, N, K, lda, ldb, ldc, order="col", transa=True, transb=False)
    hA = torch.from_numpy(memA).pin_memory()
    hB = torch.from_numpy(memB).pin_memory()
    hC = torch.from_numpy(memC.copy()).pin_memory()
    dA = torch.empty_like(hA, device="cuda")
    dB = torch.empty_like(hB, device="cuda")
    dC = torch.empty_like(hC, device="cuda")
    plan.run_host(1.0, hA, hB, 2.0, hC, dA, dB, dC)
    torch.cuda.synchronize()
    plan.close()
    assert_parity(hC.numpy().T, Cref, S, K, "col-major TN via host buffers")


def test_plan_ex_argument_errors(sg):
    l = sg.lib()
    h = ctypes.c_void_p()
    # row-major A stored K x M needs lda >= M; column-major C needs ldc >= M
    assert l.sgemm_plan_ex(0, 1, 0, 64, 32, 16, 63, 32, 32, -1, ctypes.byref(h)) == sg.SGEMM_ERR_INVALID_ARG
    assert l.sgemm_plan_ex(1, 0, 0, 64, 32, 16, 64, 16, 63, -1, ctypes.byref(h)) == sg.SGEMM_ERR_INVALID_ARG
    assert l.sgemm_plan_ex(2, 0, 0, 64, 32, 16, 64, 16, 64, -1, ctypes.byref(h)) == sg.SGEMM_ERR_INVALID_ARG
    assert l.sgemm_plan_ex(0, 2, 0, 64, 32, 16, 64, 32, 32, -1, ctypes.byref(h)) == sg.SGEMM_ERR_INVALID_ARG


# ---- strided batches (sgemm_plan_batched) -------------------------------------

@pytest.mark.parametrize("case", [
    # (M, N, K, batch, config, shared A?)  None = the table's choice
    (96, 80, 72, 7, None, False),                       # small products: 128 x 64 tiles over the batch
    (300, 520, 260, 3, None, False),                    # ragged tiles in every product
    (640, 1024, 256, 9, "tmat_128x256x32_s3_b1", False),  # 180 tiles: a stream-K tail over batches 7 and 8
    (640, 768, 256, 4, "tmat_128x128x32_s4_b1", True),  # A shared by every product (stride 0)
    (65, 33, 17, 9, "generic_64x64x16", False),
    # up to 64 rows with a long k loop: 64-row tiles over the batch; 17 to 32 rows: 32 x 32 tiles
    (48, 2048, 1024, 3, None, False),
    (24, 1024, 2048, 5, None, True),
    # few rows with 2^22 or more elements of B over the batch: the sixteen-row matrix-vector kernel
    (16, 1024, 512, 8, None, False),
    (12, 2048, 700, 6, None, True),                     # ragged K, A shared
    # fewer: the stream-K few-row kernel over (product, slab, k-slice) units
    (16, 512, 256, 4, None, False),
    (7, 300, 520, 5, None, True),                       # ragged N and K, A shared
    (1, 4096, 256, 3, None, False),
])
def test_strided_batch(sg, oracle_mod, case):
    M, N, K, batch, config, shared_a = case
    rng = np.random.default_rng(M * N + K + batch)
    A = rng.standard_normal((1 if shared_a else batch, M, K), dtype=np.float32)
    B = rng.standard_normal((batch, K, N), dtype=np.float32)
    C0 = rng.uniform(-1, 1, (batch, M, N)).astype(np.float32)
    alpha, beta = 1.25, 0.5
    # strides padded past the matrices (16-byte multiples), A shared when stride_a = 0
    sa = 0 if shared_a else M * K + 8
    sb, sc = K * N + 4, M * N + 12
    dA = torch.zeros(max(1, (0 if shared_a else batch - 1) * sa + M * K), device="cuda")
    dB = torch.zeros((batch - 1) * sb + K * N, device="cuda")
    dC = torch.zeros((batch - 1) * sc + M * N, device="cuda")
    for z in range(batch):
        if not shared_a or z == 0:
            dA[z * sa: z * sa + M * K] = torch.from_numpy(A[z].ravel())
        dB[z * sb: z * sb + K * N] = torch.from_numpy(B[z].ravel())
        dC[z * sc: z * sc + M * N] = torch.from_numpy(C0[z].ravel())
    plan = sg.Plan(M, N, K, config=config, batch=batch, stride_a=sa, stride_b=sb, stride_c=sc)
    info = plan.info()
    assert info["batch"] == batch
    if config is None and M <= 16:
        expect = "gemv_4x512" if M <= 4 else "gemv_16x1024" if batch * N * K >= 1 << 22 else "skinny_sk"
        assert info["variant"].startswith(expect), info
    plan.run(alpha, dA, dB, beta, dC)
    torch.cuda.synchronize()
    assert sg.device_status() == sg.SGEMM_OK
    out = dC.cpu().numpy()
    for z in range(batch):
        Cref, S = oracle_mod.sgemm_ref(A[0 if shared_a else z], B[z], C0[z], alpha, beta)
        Cz = out[z * sc: z * sc + M * N].reshape(M, N)
        assert_parity(Cz, Cref, S, K, f"batch {z}/{batch} {info['variant']} {M}x{N}x{K}")
        # the padding between products is untouched
        if z + 1 < batch:
            assert np.all(out[z * sc + M * N: (z + 1) * sc] == 0.0)
    plan.close()


@pytest.mark.parametrize("order", ["row", "col"])
@pytest.mark.parametrize("ta,tb", [(False, False), (False, True), (True, False), (True, True)])
@pytest.mark.parametrize("case", [
    # (M, N, K, batch, shared A?): more than 16 rows (the transposed-A kernels read
    # A given transposed), few rows (the few-row kernel reads B given transposed)
    (300, 260, 96, 3, False), (16, 520, 264, 4, False), (7, 300, 100, 3, True), (200, 136, 64, 2, True),
    # one to four rows (K in two chunks, partial sums added by a second kernel)
    (2, 300, 1100, 3, False)])
def test_batched_order_and_transpose(sg, oracle_mod, order, ta, tb, case):
    """sgemm_plan_ex_batched: every order x transpose combination of a strided
    batch, against the oracle product by product."""
    M, N, K, batch, shared_a = case
    rng = np.random.default_rng(M + N + K + batch + 2 * ta + tb)
    opA = rng.standard_normal((batch, M, K), dtype=np.float32)
    if shared_a:
        opA[1:] = opA[0]
    opB = rng.standard_normal((batch, K, N), dtype=np.float32)
    C0 = rng.uniform(-1, 1, (batch, M, N)).astype(np.float32)
    alpha, beta = 0.5, -1.25
    mems_a = [_stored(opA[z], order, ta, 0) for z in range(batch)]
    mems_b = [_stored(opB[z], order, tb, 0) for z in range(batch)]
    mems_c = [_stored(C0[z], order, False, 0) for z in range(batch)]
    lda, ldb, ldc = mems_a[0][1], mems_b[0][1], mems_c[0][1]

    def pack(mems, shared=False):
        size = mems[0][0].size
        stride = 0 if shared else (size + 3) // 4 * 4 + 4  # 16-byte multiples, padding between products
        buf = torch.zeros(max(1, (0 if shared else len(mems) - 1) * stride + size), device="cuda")
        for z, (m, _) in enumerate(mems[:1] if shared else mems):
            buf[z * stride: z * stride + size] = torch.from_numpy(m.ravel())
        return buf, stride

    dA, sa = pack(mems_a, shared_a)
    dB, sb = pack(mems_b)
    dC, sc = pack(mems_c)
    plan = sg.Plan(M, N, K, lda, ldb, ldc, order=order, transa=ta, transb=tb, batch=batch, stride_a=sa,
                   stride_b=sb, stride_c=sc)
    info = plan.info()
    assert info["batch"] == batch and info["order"] == order
    plan.run(alpha, dA, dB, beta, dC)
    torch.cuda.synchronize()
    assert sg.device_status() == sg.SGEMM_OK
    out = dC.cpu().numpy()
    size_c = mems_c[0][0].size
    for z in range(batch):
        Cref, S = oracle_mod.sgemm_ref(opA[z], opB[z], C0[z], alpha, beta)
        mem = out[z * sc: z * sc + size_c].reshape(mems_c[0][0].shape)
        Cz = mem if order == "row" else mem.T
        assert_parity(Cz, Cref, S, K, f"batch {z}/{batch} {order} op={info['op']} {info['variant']} {case}")
        if z + 1 < batch:
            assert np.all(out[z * sc + size_c: (z + 1) * sc] == 0.0)
    plan.close()


def test_strided_batch_argument_errors(sg):
    l = sg.lib()
    h = ctypes.c_void_p()
    f = l.sgemm_plan_batched
    assert f(64, 64, 64, 64, 64, 64, 2, 4096, 4096, 4095, -1, ctypes.byref(h)) == sg.SGEMM_ERR_INVALID_ARG  # C overlap
    assert f(64, 64, 64, 64, 64, 64, -1, 4096, 4096, 4096, -1, ctypes.byref(h)) == sg.SGEMM_ERR_INVALID_ARG
    assert f(64, 64, 64, 64, 64, 64, 70000, 4096, 4096, 4096, -1, ctypes.byref(h)) == sg.SGEMM_ERR_UNSUPPORTED
    skinny = sg.config_id("skinny_16x128x32_w4_s3_b3_ef_pa")
    assert f(16, 256, 64, 64, 256, 256, 2, 1024, 16384, 4096, skinny, ctypes.byref(h)) == sg.SGEMM_ERR_UNSUPPORTED
    empty = sg.Plan(64, 64, 64, batch=0)
    assert empty.launches == 0
    empty.run(1.0, 0, 0, 0.0, 0)  # nothing to do
    empty.close()


# ---- a C of more than 2^31 elements: 64-bit offsets in every epilogue ---------

@pytest.mark.parametrize("config,off_a", [(None, 0), ("generic_64x64x16", 1), ("tf32x3_128x128x32_s3", 0),
                                          ("tf32x3f_128x128x32_s3", 0)])
def test_c_beyond_2_31_elements(sg, oracle_mod, config, off_a):
    M, N, K = 65536 + 17, 32768 + 9, 40
    assert M * N > 2 ** 31
    rng = np.random.default_rng(17)  # A and B only: a host C0 of this size is not needed (beta = 0)
    A = rng.standard_normal((M, K), dtype=np.float32)
    B = rng.standard_normal((K, N), dtype=np.float32)
    ldb = N + 3  # 16-byte rows for the TMA-fed kernels
    dA, pA, lda = _to_dev(A, None, off_a)
    dB, pB, _ = _to_dev(B, ldb)
    dC = torch.full((M, N), float("nan"), device="cuda")  # beta = 0: every entry must be written
    plan = sg.Plan(M, N, K, lda, ldb, N, config=config)
    plan.run(1.0, pA, pB, 0.0, dC)
    torch.cuda.synchronize()
    assert sg.device_status() == sg.SGEMM_OK
    used = plan.config_name
    plan.close()
    rows = np.array([0, 1, 2 ** 31 // N - 1, 2 ** 31 // N, 2 ** 31 // N + 1, M - 2, M - 1])
    assert (rows * N).max() > 2 ** 31
    Cs = dC[torch.from_numpy(rows).cuda()].cpu().numpy()
    del dC
    Cref, S = oracle_mod.sgemm_ref(np.ascontiguousarray(A[rows]), B, None, 1.0, 0.0)
    assert_parity(Cs, Cref, S, K, f"{used} rows {rows.tolist()} of {M}x{N}")


def test_run_host_pipelined(sg, oracle_mod):
    """Six different products streamed from pinned host memory through two buffer sets."""
    M, N, K = 300, 260, 196
    plan = sg.Plan(M, N, K)
    ins = [make_inputs(M, N, K, seed=100 + i, dist_a=("normal", 1.0), dist_b=("normal", 1.0)) for i in range(6)]
    hA = [torch.from_numpy(a).pin_memory() for a, _, _ in ins]
    hB = [torch.from_numpy(b).pin_memory() for _, b, _ in ins]
    hC = [torch.from_numpy(c.copy()).pin_memory() for _, _, c in ins]
    dA = [torch.empty(M, K, device="cuda") for _ in range(2)]
    dB = [torch.empty(K, N, device="cuda") for _ in range(2)]
    dC = [torch.empty(M, N, device="cuda") for _ in range(2)]
    stream = torch.cuda.Stream()
    plan.run_host_pipelined(0.5, hA, hB, 2.0, hC, dA, dB, dC, stream=stream)
    stream.synchronize()
    assert sg.device_status() == sg.SGEMM_OK
    for i, (a, b, c) in enumerate(ins):
        Cref, S = oracle_mod.sgemm_ref(a, b, c, 0.5, 2.0)
        assert_parity(hC[i].numpy(), Cref, S, K, f"pipelined product {i}")
    plan.close()


def test_few_row_transposed_b_is_read_natively(sg, oracle_mod):
    """y = x W^T with W stored N x K (the weight layout of decode): the
    stream-K few-row kernel reads W as stored, with no transpose kernel."""
    M, N, K = 16, 8192, 4096
    x, Wt, C0 = make_inputs(M, N, K, seed=77, dist_a=("normal", 1.0), dist_b=("normal", 0.02))
    W = np.ascontiguousarray(Wt.T)  # N x K
    plan = sg.Plan(M, N, K, transb=True)
    info = plan.info()
    assert info["variant"].startswith("skinny_sk") and info["op"] == "NT"
    assert plan.launches == 1
    dA = torch.from_numpy(x).cuda()
    dB = torch.from_numpy(W).cuda()
    dC = torch.from_numpy(C0).cuda()
    plan.run(1.0, dA, dB, 1.0, dC)
    torch.cuda.synchronize()
    assert sg.device_status() == sg.SGEMM_OK
    Cref, S = oracle_mod.sgemm_ref(x, Wt, C0, 1.0, 1.0)
    assert_parity(dC.cpu().numpy(), Cref, S, K, "few-row NT")
    plan.close()


# ---- one to four rows: the matrix-vector kernels -----------------------------

GEMV_CASES = [(1, 1, 1), (1, 511, 1000), (2, 513, 1023), (3, 4097, 1025), (4, 1000, 3000), (1, 77, 5000),
              (4, 8, 64), (1, 3, 70000), (2, 16384, 8192)]


@pytest.mark.parametrize("shape", GEMV_CASES)
@pytest.mark.parametrize("layout", ["nn", "nn_odd", "nt", "nt_odd"])
def test_gemv_rows(sg, oracle_mod, shape, layout):
    """M <= 4 through the table: B as stored (K x N) or given transposed
    (N x K), 16-byte and 4-byte loads (odd row strides, B one float off a
    16-byte boundary), one or several K chunks; bit-identical on a rerun; C
    with NaN ignored at beta = 0; the padding of C untouched."""
    M, N, K = shape
    tb = layout.startswith("nt")
    odd = layout.endswith("odd")
    A, B, C0 = make_inputs(M, N, K, seed=M * 5 + N + K + len(layout), dist_a=("normal", 1.0),
                           dist_b=("normal", 0.05))
    stored_b = np.ascontiguousarray(B.T) if tb else B
    lda = K + (3 if odd else 0)
    ldb = stored_b.shape[1] + (1 if odd else 0)
    ldc = N + 5
    dA, pA, _ = _to_dev(A, lda, 1 if odd else 0)
    dB, pB, _ = _to_dev(stored_b, ldb, 1 if odd else 0)
    for alpha, beta in ((1.0, 0.0), (-0.5, 2.0)):
        dC, pC, _ = _to_dev(np.full((M, N), np.nan, np.float32) if beta == 0.0 else C0, ldc, 0, fill=7.0)
        plan = sg.Plan(M, N, K, lda, ldb, ldc, transb=tb)
        info = plan.info()
        assert info["variant"] == "gemv_4x512" and info["op"] == ("NT" if tb else "NN"), info
        assert plan.launches in (1, 2) and (info["split"] > 1 or plan.launches == 1), (plan.launches, info)
        outs = []
        for _ in range(2):
            if beta != 0.0:
                dC.copy_(_to_dev(C0, ldc, 0, fill=7.0)[0])
            plan.run(alpha, pA, pB, beta, pC)
            torch.cuda.synchronize()
            assert sg.device_status() == sg.SGEMM_OK
            outs.append(dC.cpu().numpy().copy())
        plan.close()
        assert np.array_equal(outs[0], outs[1], equal_nan=True), "not reproducible"
        host = outs[0]
        C = np.stack([host[m * ldc: m * ldc + N] for m in range(M)])
        for m in range(M):
            assert np.all(host[m * ldc + N: (m + 1) * ldc if m + 1 < M else host.size] == 7.0), "padding written"
        Cref, S = oracle_mod.sgemm_ref(A, B, C0 if beta != 0.0 else None, alpha, beta)
        assert_parity(C, Cref, S, K, f"gemv {layout} {shape} split={info['split']} a={alpha} b={beta}")
        if not tb and alpha == 1.0 and beta == 0.0 and info["k_order"] == "sequential":
            ii, jj = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
            chain = oracle_mod.fp32_chain_entries(A, B, ii.ravel(), jj.ravel()).reshape(M, N)
            assert np.array_equal(C, chain), f"{shape}: not the ascending-k fp32 chain"


def test_gemv_refuses_more_than_four_rows(sg):
    with pytest.raises(sg.SgemmError) as e:
        sg.Plan(5, 256, 256, config="gemv_4x512")
    assert e.value.status == sg.SGEMM_ERR_UNSUPPORTED


# ---- five to sixteen rows: the cp.async-ring matrix-vector kernel ------------

ROWS_CASES = [(5, 1, 1), (16, 1024, 640), (9, 1025, 641), (16, 4100, 2000), (8, 300, 7), (12, 16384, 1024),
              (16, 3, 9000), (13, 2048, 4096)]


@pytest.mark.parametrize("shape", ROWS_CASES)
@pytest.mark.parametrize("layout", ["nn", "nn_odd"])
def test_sixteen_rows(sg, oracle_mod, shape, layout):
    """gemv_16x1024 (5 to 16 rows, B as stored): 16-byte and 4-byte copies
    (odd row strides, A and B one float off a 16-byte boundary), one K chunk
    and several (partial sums added by the reduce kernel), N and K ragged
    against the 1024-column CTA and the 4-row copy groups; bit-identical on a
    rerun; NaN in C ignored at beta = 0; the padding of C untouched."""
    M, N, K = shape
    odd = layout == "nn_odd"
    A, B, C0 = make_inputs(M, N, K, seed=M * 3 + N + 7 * K + len(layout), dist_a=("normal", 1.0),
                           dist_b=("normal", 0.05))
    lda = K + (3 if odd else 0)
    ldb = N + (1 if odd else 0)
    ldc = N + 5
    dA, pA, _ = _to_dev(A, lda, 1 if odd else 0)
    dB, pB, _ = _to_dev(B, ldb, 1 if odd else 0)
    for alpha, beta in ((1.0, 0.0), (-0.5, 2.0)):
        dC, pC, _ = _to_dev(np.full((M, N), np.nan, np.float32) if beta == 0.0 else C0, ldc, 0, fill=7.0)
        plan = sg.Plan(M, N, K, lda, ldb, ldc, config="gemv_16x1024")
        info = plan.info()
        assert info["variant"] == "gemv_16x1024", info
        assert plan.launches in (1, 2) and (info["split"] > 1 or plan.launches == 1), (plan.launches, info)
        outs = []
        for _ in range(2):
            if beta != 0.0:
                dC.copy_(_to_dev(C0, ldc, 0, fill=7.0)[0])
            plan.run(alpha, pA, pB, beta, pC)
            torch.cuda.synchronize()
            assert sg.device_status() == sg.SGEMM_OK
            outs.append(dC.cpu().numpy().copy())
        plan.close()
        assert np.array_equal(outs[0], outs[1], equal_nan=True), "not reproducible"
        host = outs[0]
        C = np.stack([host[m * ldc: m * ldc + N] for m in range(M)])
        for m in range(M):
            assert np.all(host[m * ldc + N: (m + 1) * ldc if m + 1 < M else host.size] == 7.0), "padding written"
        Cref, S = oracle_mod.sgemm_ref(A, B, C0 if beta != 0.0 else None, alpha, beta)
        assert_parity(C, Cref, S, K, f"rows16 {layout} {shape} split={info['split']} a={alpha} b={beta}")


@pytest.mark.parametrize("shared_a", [False, True])
def test_sixteen_rows_batched_any_stride(sg, oracle_mod, shared_a):
    """gemv_16x1024 over a strided batch whose strides are not multiples of 4
    (B's rows are then copied 4 bytes at a time) and whose A may be shared
    (stride 0), product by product against the oracle; the padding between
    the products' C untouched; bit-identical on a rerun."""
    M, N, K, batch = 11, 1500, 700, 3
    rng = np.random.default_rng(1611)
    A = rng.standard_normal((batch, M, K), dtype=np.float32)
    B = (rng.standard_normal((batch, K, N), dtype=np.float32) * np.float32(0.05)).astype(np.float32)
    C0 = rng.uniform(-1, 1, (batch, M, N)).astype(np.float32)
    sa = 0 if shared_a else M * K + 5
    sb, sc = K * N + 3, M * N + 7
    dA = torch.zeros(max(1, (0 if shared_a else batch - 1) * sa + M * K), device="cuda")
    dB = torch.zeros((batch - 1) * sb + K * N, device="cuda")
    dC = torch.zeros((batch - 1) * sc + M * N, device="cuda")
    for z in range(batch):
        if not shared_a or z == 0:
            dA[z * sa: z * sa + M * K] = torch.from_numpy(A[z].ravel())
        dB[z * sb: z * sb + K * N] = torch.from_numpy(B[z].ravel())
        dC[z * sc: z * sc + M * N] = torch.from_numpy(C0[z].ravel())
    c_init = dC.clone()
    plan = sg.Plan(M, N, K, config="gemv_16x1024", batch=batch, stride_a=sa, stride_b=sb, stride_c=sc)
    outs = []
    for _ in range(2):
        dC.copy_(c_init)
        plan.run(-0.5, dA, dB, 2.0, dC)
        torch.cuda.synchronize()
        assert sg.device_status() == sg.SGEMM_OK
        outs.append(dC.cpu().numpy().copy())
    plan.close()
    assert np.array_equal(outs[0], outs[1]), "not reproducible"
    out = outs[0]
    for z in range(batch):
        Cref, S = oracle_mod.sgemm_ref(A[0 if shared_a else z], B[z], C0[z], -0.5, 2.0)
        assert_parity(out[z * sc: z * sc + M * N].reshape(M, N), Cref, S, K, f"rows16 batch {z} shared_a={shared_a}")
        if z + 1 < batch:
            assert np.all(out[z * sc + M * N: (z + 1) * sc] == 0.0)


def test_sixteen_rows_table_and_limits(sg):
    """The table sends one product of 5 to 16 rows with B as stored and 16 MB
    or more of B to gemv_16x1024 (no padding copy, even for odd ldb), B given
    transposed to the few-row kernel that reads it as stored; the variant
    refuses 17 rows."""
    for (M, N, K, ldb) in ((16, 16384, 8192, 16384), (5, 4096, 1024, 4096), (16, 16384, 8192, 16385)):
        plan = sg.Plan(M, N, K, ldb=ldb)
        info = plan.info()
        assert info["variant"] == "gemv_16x1024" and info["repack"] == 0, info
        plan.close()
    plan = sg.Plan(16, 16384, 8192, transb=True)
    assert plan.info()["variant"].startswith("skinny_sk"), plan.info()
    plan.close()
    with pytest.raises(sg.SgemmError) as e:
        sg.Plan(17, 256, 256, config="gemv_16x1024")
    assert e.value.status == sg.SGEMM_ERR_UNSUPPORTED


def test_ffma_probe(sg):
    """The FMA-only probe: its rate is near the nominal SMs x 128 x 2 x clock, and the clock read inside the
    kernel is a plausible SM clock."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for paired in (True, False):
        tflops, mhz = sg.probe_ffma(paired)
        assert 300.0 < mhz < 3500.0, mhz
        nominal = sms * 128 * 2 * mhz * 1e6 / 1e12
        assert 0.5 * nominal < tflops < 1.05 * nominal, (paired, tflops, nominal)


def test_c_overlapping_a_or_b_is_refused(sg):
    M, N, K = 64, 64, 64
    buf = torch.zeros(3 * 64 * 64, device="cuda")
    plan = sg.Plan(M, N, K)
    a, b, c = buf.data_ptr(), buf.data_ptr() + 4 * 64 * 64, buf.data_ptr() + 8 * 64 * 64
    plan.run(1.0, a, b, 0.0, c)  # disjoint spans: fine
    for cc in (a, b, b + 4 * 100):
        with pytest.raises(sg.SgemmError) as e:
            plan.run(1.0, a, b, 0.0, cc)
        assert e.value.status == sg.SGEMM_ERR_UNSUPPORTED
    plan.run(1.0, a, a, 0.0, c)  # A and B may alias each other
    torch.cuda.synchronize()
    plan.close()


@pytest.mark.parametrize("shape,config", [((2048, 2048, 1024), None), ((4096, 4096, 1024), None),
                                          ((16, 16384, 4096), "skinny_sk_16x128x32_w4_s3_b3_ef")])
def test_stream_k_plan_replays_in_a_cuda_graph(sg, oracle_mod, shape, config):
    """A stream-K plan captured in a CUDA graph and replayed on new inputs: the
    finishers clear the flags they consumed, so the fixed epoch of the
    captured launch stays valid replay after replay."""
    M, N, K = shape
    plan = sg.Plan(M, N, K, config=config)
    info = plan.info()
    assert info["streamk"] == 1, info
    dA = torch.zeros(M, K, device="cuda")
    dB = torch.zeros(K, N, device="cuda")
    dC = torch.zeros(M, N, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        plan.run(1.0, dA, dB, 0.0, dC, stream=s)  # warm: kernel attributes and modules before capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        plan.run(1.0, dA, dB, 0.0, dC, stream=s)
    rows, cols = sample_rows_cols(M, N, n_rows=min(M, 128), n_cols=128, seed=1)
    for rep in range(3):
        A, B, _ = make_inputs(M, N, K, seed=400 + rep, dist_a=("normal", 1.0), dist_b=("normal", 1.0), dist_c=None)
        dA.copy_(torch.from_numpy(A))
        dB.copy_(torch.from_numpy(B))
        g.replay()
        torch.cuda.synchronize()
        assert sg.device_status() == sg.SGEMM_OK
        Cs = dC.cpu().numpy()[np.ix_(rows, cols)]
        Cref, S = oracle_mod.sgemm_ref(np.ascontiguousarray(A[rows]), np.ascontiguousarray(B[:, cols]), None, 1.0, 0.0)
        assert_parity(Cs, Cref, S, K, f"graph replay {rep} of {info['variant']}")
    plan.close()


@pytest.mark.parametrize("shape", [(1, 16384, 8192), (16, 16384, 4096), (7, 3000, 5000)])
def test_matrix_vector_plan_replays_in_a_cuda_graph(sg, oracle_mod, shape):
    """A matrix-vector plan whose K is cut into chunks (the chunk kernel, then
    its reduce kernel as a programmatic dependent launch) captured in a CUDA
    graph and replayed on new inputs with beta != 0."""
    M, N, K = shape
    plan = sg.Plan(M, N, K)
    info = plan.info()
    assert info["kind"] == "gemv" and info["split"] > 1 and plan.launches == 2, info
    dA = torch.zeros(M, K, device="cuda")
    dB = torch.zeros(K, N, device="cuda")
    dC = torch.zeros(M, N, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        plan.run(1.0, dA, dB, 0.5, dC, stream=s)  # warm: kernel attributes and modules before capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        plan.run(-0.75, dA, dB, 0.5, dC, stream=s)
    for rep in range(3):
        A, B, C0 = make_inputs(M, N, K, seed=500 + rep, dist_a=("normal", 1.0), dist_b=("normal", 0.05))
        dA.copy_(torch.from_numpy(A))
        dB.copy_(torch.from_numpy(B))
        dC.copy_(torch.from_numpy(C0))
        g.replay()
        torch.cuda.synchronize()
        assert sg.device_status() == sg.SGEMM_OK
        Cref, S = oracle_mod.sgemm_ref(A, B, C0, -0.75, 0.5)
        assert_parity(dC.cpu().numpy(), Cref, S, K, f"graph replay {rep} of {info['variant']}")
    plan.close()


def test_autotune_picks_the_fastest_and_caches_it(sg, oracle_mod):
    M, N, K = 1000, 1100, 512
    dA = torch.randn(M, K, device="cuda")
    dB = torch.randn(K, N, device="cuda")
    dC = torch.empty(M, N, device="cuda")
    plan, times = sg.autotune(M, N, K, dA, dB, dC, with_times=True)
    assert times and plan.config_name == min(times, key=times.get)
    assert not any(n.startswith("tf32x3") for n in times)  # FFMA variants only by default
    again = sg.autotune(M, N, K, dA, dB, dC)  # cached: same choice, no timing
    assert again.config_name == plan.config_name
    A, B, C0 = make_inputs(M, N, K, seed=9, dist_a=("normal", 1.0), dist_b=("normal", 1.0))
    C, used = run_gpu(sg, A, B, C0, 0.5, 2.0, config=plan.config_name)
    Cref, S = oracle_mod.sgemm_ref(A, B, C0, 0.5, 2.0)
    assert_parity(C, Cref, S, K, f"autotuned {used}")
    _, with_tc = sg.autotune(M, N, K, dA, dB, dC, tensor_cores=True, with_times=True)
    assert any(n.startswith("tf32x3") for n in with_tc)
    plan.close()
    again.close()


def test_sgemm_helper_reuses_its_plan(sg, oracle_mod):
    """sgemm() keeps its plan per (device, shape, layout, config, stream): at a
    stream-K shape the first call allocates the plan's workspace, later calls
    allocate no device memory, and every result is within the bound."""
    M, N, K = 2048, 4096, 1024
    sg.clear_plan_cache()
    A, B, C0 = make_inputs(M, N, K, seed=77, dist_a=("normal", 1.0), dist_b=("normal", 1.0))
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dC = torch.from_numpy(C0).cuda()
    assert sg.Plan(M, N, K).info()["streamk"] == 1  # the table's plan has a workspace at this shape
    sg.sgemm(dA, dB, dC, alpha=1.0, beta=0.0)
    torch.cuda.synchronize()
    assert sg.plan_cache_size() == 1
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        sg.sgemm(dA, dB, dC, alpha=0.5, beta=0.0)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"device memory changed across calls: {free0} -> {free1}"
    assert sg.plan_cache_size() == 1
    assert sg.device_status() == sg.SGEMM_OK
    rows, cols = sample_rows_cols(M, N, n_rows=128, n_cols=128, seed=3)
    Cref, S = oracle_mod.sgemm_ref(np.ascontiguousarray(A[rows]), np.ascontiguousarray(B[:, cols]), None, 0.5, 0.0)
    got = dC.cpu().numpy()[np.ix_(rows, cols)].astype(np.float64)
    assert np.all(np.abs(got - Cref) <= _bound(K, S))
    # another stream gets its own plan (runs on two streams may overlap)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        sg.sgemm(dA, dB, dC, alpha=1.0, beta=0.0, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert sg.plan_cache_size() == 2
    sg.clear_plan_cache()
    assert sg.plan_cache_size() == 0


@pytest.mark.parametrize("shape", [(4096, 4096, 4096, None, None), (4096, 4096, 4096, 4097, None),
                                   (16, 16384, 8192, None, None), (1, 4096, 4096, None, None),
                                   (128, 128, 128, None, None), (32, 4096, 4096, None, None),
                                   (64, 4096, 4096, None, None), (768, 768, 512, None, None),
                                   (1408, 1408, 1408, None, None), (200, 130, 100, 101, 131),
                                   (100, 96, 1000, None, 97), (8, 300, 520, None, None)])
def test_plan_follows_the_host_table(sg, shape):
    # a plan's variant is the one sgemm_table_choice computes on the host for this device's SM count
    M, N, K, lda, ldb = shape
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    expect, rp_a, rp_b = sg.table_choice(M, N, K, lda=lda, ldb=ldb, num_sms=sms)
    plan = sg.Plan(M, N, K, lda or K, ldb or N, N)
    try:
        info = plan.info()
        assert info["variant"] == expect, (shape, info["variant"], expect)
        assert info["repack"] == (1 if rp_a else 0) | (2 if rp_b else 0), (shape, info["repack"], rp_a, rp_b)
    finally:
        plan.close()
