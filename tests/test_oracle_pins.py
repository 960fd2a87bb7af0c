"""Pins for the CPU oracle itself: values fixed by hand, by the mathematics
and by independent routines, so the oracle is not trusted on its own word.

Each pin is chosen so that a plausible mistake in the oracle (dropped beta
term, wrong sign, transposed operand, off-by-one in the sum, double
rounding) fails at least one of them; the last group of tests plants those
mistakes and checks that the pins catch them.
"""
import numpy as np
import pytest

from conftest import load_golden
from dense_fp32_matrix_sm_gb300.inputs import WORKLOADS, make_inputs, workload_inputs

GOLDEN_CASES = ["hand_2x2.txt", "hand_3x3.txt", "hand_2x3x4.txt"]


def _golden_inputs(g):
    A = g["A"].astype(np.float32)
    B = g["B"].astype(np.float32)
    C0 = g["C0"].astype(np.float32)
    return A, B, C0, g["alpha"], g["beta"]


def _golden_matches(g, C, S=None):
    ok = C.shape == g["C"].shape and np.array_equal(C, g["C"])
    if S is not None:
        ok = ok and np.array_equal(S, g["S"])
    return ok


# ---- 1. hand-worked products -------------------------------------------------

@pytest.mark.parametrize("name", GOLDEN_CASES)
def test_hand_worked_full(oracle_mod, name):
    g = load_golden(name)
    A, B, C0, alpha, beta = _golden_inputs(g)
    C, S = oracle_mod.sgemm_ref(A, B, C0, alpha, beta, threads=1)
    assert A.shape == (g["M"], g["K"]) and B.shape == (g["K"], g["N"])
    assert np.array_equal(C, g["C"]), (C, g["C"])
    assert np.array_equal(S, g["S"]), (S, g["S"])


@pytest.mark.parametrize("name", GOLDEN_CASES)
def test_hand_worked_entries(oracle_mod, name):
    g = load_golden(name)
    A, B, C0, alpha, beta = _golden_inputs(g)
    ii, jj = np.meshgrid(np.arange(g["M"]), np.arange(g["N"]), indexing="ij")
    c, s = oracle_mod.sgemm_ref_entries(A, B, C0, alpha, beta, ii.ravel(), jj.ravel())
    assert np.array_equal(c.reshape(g["M"], g["N"]), g["C"])
    assert np.array_equal(s.reshape(g["M"], g["N"]), g["S"])


@pytest.mark.parametrize("name", GOLDEN_CASES)
def test_hand_worked_bruteforce(oracle_mod, name):
    g = load_golden(name)
    A, B, C0, alpha, beta = _golden_inputs(g)
    C, S = oracle_mod.bruteforce_py(A.tolist(), B.tolist(), C0.tolist(), alpha, beta)
    assert np.array_equal(np.array(C), g["C"])
    assert np.array_equal(np.array(S), g["S"])


# ---- 2. identity and permutation matrices ------------------------------------

def test_identity_and_permutation(oracle_mod):
    rng = np.random.default_rng(11)
    A = rng.standard_normal((13, 9), dtype=np.float32)
    B = rng.standard_normal((9, 17), dtype=np.float32)
    I9 = np.eye(9, dtype=np.float32)
    I13 = np.eye(13, dtype=np.float32)
    C, _ = oracle_mod.sgemm_ref(A, I9, alpha=1.0, beta=0.0)
    assert np.array_equal(C, A.astype(np.float64))
    C, _ = oracle_mod.sgemm_ref(I9, B, alpha=1.0, beta=0.0)
    assert np.array_equal(C, B.astype(np.float64))
    perm = rng.permutation(13)
    P = I13[perm]                      # (P A)[i] = A[perm[i]]
    C, _ = oracle_mod.sgemm_ref(P, A, alpha=1.0, beta=0.0)
    assert np.array_equal(C, A[perm].astype(np.float64))
    perm9 = rng.permutation(9)
    Q = I9[:, perm9]                   # (A Q)[:, j] = A[:, perm9[j]]
    C, _ = oracle_mod.sgemm_ref(A, Q, alpha=1.0, beta=0.0)
    assert np.array_equal(C, A[:, perm9].astype(np.float64))


# ---- 3. integer-valued inputs: every result exact -----------------------------

@pytest.mark.parametrize("shape", [(7, 5, 3), (16, 33, 64), (31, 1, 17), (1, 40, 64)])
def test_integer_exact(oracle_mod, shape):
    M, N, K = shape
    A, B, C0 = make_inputs(M, N, K, seed=M * 1000 + N, dist_a=("int", 8), dist_b=("int", 8),
                           dist_c=("int", 8))
    exact = A.astype(np.int64) @ B.astype(np.int64)
    C, S = oracle_mod.sgemm_ref(A, B, C0, alpha=1.0, beta=0.0)
    assert np.array_equal(C, exact.astype(np.float64))
    assert np.array_equal(S, (np.abs(A).astype(np.int64) @ np.abs(B).astype(np.int64)).astype(np.float64))
    C, _ = oracle_mod.sgemm_ref(A, B, C0, alpha=2.0, beta=-1.0)
    assert np.array_equal(C, (2 * exact - C0.astype(np.int64)).astype(np.float64))


# ---- 4. the FLOP count ------------------------------------------------------------

def test_flop_count():
    # "Writing a Fast Matmul in CUDA, Step by Step", Step 1: 2 * 4096^3 = 137.4 billion.
    assert WORKLOADS["square4096"].flops == 137_438_953_472
    assert 2 * 4096 ** 3 == 137_438_953_472
    # "How a Matmul Kernel Gets Fast", section 1: 2 * 4092^3 ~ 137 billion.
    assert abs(WORKLOADS["square4092"].flops - 137e9) < 0.5e9


def test_acceptance_bound_hand_values(oracle_mod):
    # The bar is |C - C_ref| <= 4*K*2^-24*S + 1e-6, elementwise.  Worked by
    # hand: K = 4096, S = 100 gives 4 * 4096 * 100 / 16777216 = 1638400 /
    # 16777216 = 0.09765625, plus 1e-6.  K = 1, S = 0 leaves the absolute
    # term alone; K = 2^22, S = 1 gives 4 * 2^22 / 2^24 = 1, plus 1e-6.
    assert oracle_mod.acceptance_bound(4096, 100.0) == 0.09765625 + 1e-6
    assert oracle_mod.acceptance_bound(1, 0.0) == 1e-6
    assert oracle_mod.acceptance_bound(2 ** 22, 1.0) == 1.0 + 1e-6
    # elementwise over an array of S, and linear in S and in K
    got = oracle_mod.acceptance_bound(4096, np.array([[0.0, 100.0], [200.0, 50.0]]))
    want = np.array([[1e-6, 0.09765625 + 1e-6], [0.1953125 + 1e-6, 0.048828125 + 1e-6]])
    assert got.shape == (2, 2) and np.array_equal(got, want)


@pytest.mark.parametrize("shape", [(3, 4, 5), (17, 1, 9), (1, 1, 1), (8, 8, 0)])
def test_instrumented_fma_count(oracle_mod, shape):
    M, N, K = shape
    A, B, C0 = make_inputs(M, N, K, seed=5)
    _, _, n = oracle_mod.sgemm_ref(A, B, C0, 1.0, 0.0, count_fmas=True, threads=2)
    assert n == M * N * K          # one multiply and one add each: 2*M*N*K flops


# ---- 5. brute force and an independent library routine -------------------------

@pytest.mark.parametrize("seed", range(6))
def test_bruteforce_tiny_random(oracle_mod, seed):
    rng = np.random.default_rng(seed)
    M, N, K = (int(x) for x in rng.integers(1, 8, size=3))
    A, B, C0 = make_inputs(M, N, K, seed=100 + seed, dist_a=("normal", 1.0), dist_b=("normal", 1.0))
    alpha, beta = 0.7, -1.3
    C, S = oracle_mod.sgemm_ref(A, B, C0, alpha, beta)
    Cb, Sb = oracle_mod.bruteforce_py(A.tolist(), B.tolist(), C0.tolist(), alpha, beta)
    # same per-element order of additions (ascending p) in IEEE double: identical bits
    assert np.array_equal(C, np.array(Cb))
    assert np.array_equal(S, np.array(Sb))


def test_numpy_float64_matmul(oracle_mod):
    A, B, C0 = make_inputs(61, 47, 300, seed=7, dist_a=("normal", 1.0), dist_b=("uniform", 1.0))
    C, S = oracle_mod.sgemm_ref(A, B, C0, 0.5, 3.0)
    ref = 0.5 * (A.astype(np.float64) @ B.astype(np.float64)) + 3.0 * C0.astype(np.float64)
    assert np.max(np.abs(C - ref)) <= 1e-12 * np.max(S)


# ---- 6. rank-1 closed form --------------------------------------------------------

def test_rank_one_closed_form(oracle_mod):
    rng = np.random.default_rng(3)
    M, N, K = 9, 11, 24
    u = rng.standard_normal(M, dtype=np.float32)
    v = rng.standard_normal(N, dtype=np.float32)
    A = np.repeat(u[:, None], K, axis=1)       # A = u 1^T
    B = np.repeat(v[None, :], K, axis=0)       # B = 1 v^T
    C, S = oracle_mod.sgemm_ref(A, B, alpha=1.0, beta=0.0)
    expect = K * np.outer(u.astype(np.float64), v.astype(np.float64))
    assert np.array_equal(C, expect)           # K copies of one exact product: exact for K <= 32
    assert np.array_equal(S, np.abs(expect))


# ---- 7. statistics of the headline workload -------------------------------------

def test_square4096_entry_statistics(oracle_mod):
    # Uniform[-1,1] inputs at n = 4096: each entry is a sum of 4096 products of
    # variance 1/9, so its standard deviation is sqrt(4096/9) ~ 21.3 -- the
    # "entries of typical size 21" in "Writing a Fast Matmul in CUDA", Step 1.
    w = WORKLOADS["square4096"]
    A, B, C0 = workload_inputs(w)
    rng = np.random.default_rng(0)
    rows = rng.integers(0, w.M, 3000)
    cols = rng.integers(0, w.N, 3000)
    c, s = oracle_mod.sgemm_ref_entries(A, B, C0, w.alpha, w.beta, rows, cols)
    sd = float(np.std(c))
    assert abs(sd - np.sqrt(w.K / 9.0)) < 0.06 * np.sqrt(w.K / 9.0), sd
    # the float32 chain lands within the page's reported 1e-4 of float64 on such entries
    chain = oracle_mod.fp32_chain_entries(A, B, rows[:200], cols[:200])
    err = np.max(np.abs(chain.astype(np.float64) - c[:200]))
    assert 1e-7 < err < 3e-4, err
    assert np.all(np.abs(chain - c[:200]) <= oracle_mod.acceptance_bound(w.K, s[:200]))


# ---- 8. two loop orders, same bits; threads do not change results -------------

def test_full_equals_entries_bitwise(oracle_mod):
    A, B, C0 = make_inputs(37, 29, 53, seed=9, dist_a=("normal", 1.0), dist_b=("normal", 1.0))
    C, S = oracle_mod.sgemm_ref(A, B, C0, 0.5, 3.0, threads=1)
    ii, jj = np.meshgrid(np.arange(37), np.arange(29), indexing="ij")
    c, s = oracle_mod.sgemm_ref_entries(A, B, C0, 0.5, 3.0, ii.ravel(), jj.ravel())
    assert np.array_equal(C.ravel(), c)
    assert np.array_equal(S.ravel(), s)
    C8, S8 = oracle_mod.sgemm_ref(A, B, C0, 0.5, 3.0, threads=8)
    assert np.array_equal(C, C8) and np.array_equal(S, S8)


def test_strided_views(oracle_mod):
    A, B, C0 = make_inputs(20, 24, 30, seed=4)
    big_a = np.zeros((20, 37), np.float32)
    big_a[:, :30] = A
    C1, _ = oracle_mod.sgemm_ref(A, B, C0, 1.0, 1.0)
    C2, _ = oracle_mod.sgemm_ref(big_a[:, :30], B, C0, 1.0, 1.0)
    assert np.array_equal(C1, C2)


# ---- 9. degenerate cases (BLAS conventions) --------------------------------------

def test_degenerate_cases(oracle_mod):
    A, B, C0 = make_inputs(5, 6, 4, seed=1)
    # K == 0: C = beta*C0
    C, S = oracle_mod.sgemm_ref(np.zeros((5, 0), np.float32), np.zeros((0, 6), np.float32), C0, 2.0, 3.0)
    assert np.array_equal(C, 3.0 * C0.astype(np.float64)) and np.all(S == 0)
    # alpha == 0: the product term is dropped even if A holds NaN
    An = A.copy()
    An[0, 0] = np.nan
    C, _ = oracle_mod.sgemm_ref(An, B, C0, 0.0, -2.0)
    assert np.array_equal(C, -2.0 * C0.astype(np.float64))
    # beta == 0: C0 is not read, NaN there does not propagate
    Cn = np.full_like(C0, np.nan)
    C, _ = oracle_mod.sgemm_ref(A, B, Cn, 1.0, 0.0)
    assert np.all(np.isfinite(C))
    # M == 0 / N == 0: empty
    C, _ = oracle_mod.sgemm_ref(np.zeros((0, 4), np.float32), B, None, 1.0, 0.0)
    assert C.shape == (0, 6)
    C, _ = oracle_mod.sgemm_ref(A, np.zeros((4, 0), np.float32), None, 1.0, 0.0)
    assert C.shape == (5, 0)


def test_bad_arguments_rejected(oracle_mod):
    A, B, C0 = make_inputs(4, 4, 4, seed=2)
    with pytest.raises(ValueError):
        oracle_mod.sgemm_ref(A, B[:3], C0, 1.0, 0.0)
    with pytest.raises(ValueError):
        oracle_mod.sgemm_ref_entries(A, B, C0, 1.0, 0.0, [4], [0])


# ---- 10. the float32 chain diagnostic uses one rounding per step ----------------

def test_fp32_chain_single_rounding(oracle_mod):
    e = np.float32(1.0 + 2.0 ** -12)
    A = np.array([[e, e]], dtype=np.float32)
    B = np.array([[e], [-e]], dtype=np.float32)
    chain = oracle_mod.fp32_chain_entries(A, B, [0], [0])
    # acc1 = fl(e*e) = 1 + 2^-11 (tie to even); acc2 = fl(e*(-e) + acc1) = -2^-24 exactly.
    # A multiply rounded before the add would give 0.
    assert chain[0] == np.float32(-(2.0 ** -24))
    C, _ = oracle_mod.sgemm_ref(A, B, alpha=1.0, beta=0.0)
    assert C[0, 0] == 0.0           # the exact sum


def test_fp32_chain_integer_exact(oracle_mod):
    A, B, _ = make_inputs(9, 10, 64, seed=8, dist_a=("int", 8), dist_b=("int", 8))
    ii, jj = np.meshgrid(np.arange(9), np.arange(10), indexing="ij")
    chain = oracle_mod.fp32_chain_entries(A, B, ii.ravel(), jj.ravel())
    assert np.array_equal(chain.reshape(9, 10), (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float32))


# ---- 11. planted mistakes fail the pins --------------------------------------------

def _golden_check(name, compute):
    g = load_golden(name)
    A, B, C0, alpha, beta = _golden_inputs(g)
    try:
        C = compute(A, B, C0, alpha, beta)
    except ValueError:
        return False
    return _golden_matches(g, np.asarray(C))


def test_planted_mistakes_are_caught(oracle_mod):
    def ref(A, B, C0, al, be):
        return oracle_mod.sgemm_ref(A, B, C0, al, be)[0]

    for name in GOLDEN_CASES:
        assert _golden_check(name, ref)
        # dropped beta term
        assert not _golden_check(name, lambda A, B, C0, al, be: ref(A, B, C0, al, 0.0))
        # wrong sign on alpha
        assert not _golden_check(name, lambda A, B, C0, al, be: ref(A, B, C0, -al, be))
        # alpha applied to beta*C0 as well
        assert not _golden_check(name, lambda A, B, C0, al, be: al * ref(A, B, C0, 1.0, be))
        # sum stops one step early
        assert not _golden_check(name, lambda A, B, C0, al, be: ref(A[:, :-1], B[:-1], C0, al, be))
        # transposed operand
        assert not _golden_check(name, lambda A, B, C0, al, be: ref(A, B.T.copy(), C0, al, be)
                                 if B.shape[0] == B.shape[1] else ref(A, B[::-1].copy(), C0, al, be))
        assert not _golden_check(name, lambda A, B, C0, al, be: ref(A.T.copy(), B, C0, al, be)
                                 if A.shape[0] == A.shape[1] else ref(A[:, ::-1].copy(), B, C0, al, be))
