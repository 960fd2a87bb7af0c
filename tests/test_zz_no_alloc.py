"""sgemm_run_static_scratch: the stream-K kernel with its scratch in a
static device array, called through the C ABI.

Named to be collected last; it also passes when run alone (the first call
in the process does the per-device set-up).  Each case runs two calls in a
row on different inputs and compares each, bit for bit, with sgemm_run of
a plan made with the same kernel variant (same schedule, same sum order),
and with the fp64 oracle within the acceptance bound."""

import numpy as np
import pytest

from dense_fp32_matrix_sm_gb300.inputs import make_inputs, sample_rows_cols

torch = pytest.importorskip("torch")

VARIANT = "tmat_128x256x32_s3_b1"


@pytest.fixture(scope="module")
def sg():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import dense_fp32_matrix_sm_gb300 as sg

    return sg


def _static(sg, M, N, K, alpha, dA, dB, beta, dC, lda=None, ldb=None, ldc=None):
    return sg.run_static_scratch(M, N, K, alpha, dA, dB, beta, dC, lda=lda, ldb=ldb, ldc=ldc)


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(2048, 4096, 1024), (2100, 2900, 700), (640, 1024, 512)])
def test_static_scratch_matches_plan_two_calls(sg, oracle_mod, shape):
    M, N, K = shape
    plan = sg.Plan(M, N, K, config=VARIANT)
    info = plan.info()
    for call, (seed, alpha, beta) in enumerate(((11, 1.0, 0.0), (12, 0.5, 3.0))):
        A, B, C0 = make_inputs(M, N, K, seed=seed + M, dist_a=("normal", 1.0), dist_b=("normal", 1.0))
        dA = torch.from_numpy(A).cuda()
        dB = torch.from_numpy(B).cuda()
        want = torch.from_numpy(C0).cuda()
        plan.run(alpha, dA, dB, beta, want)
        got = torch.from_numpy(C0).cuda()
        _static(sg, M, N, K, alpha, dA, dB, beta, got)
        torch.cuda.synchronize()
        assert sg.device_status() == sg.SGEMM_OK
        got_h = got.cpu().numpy()
        assert np.array_equal(got_h, want.cpu().numpy()), \
            f"call {call}: static-scratch result differs from the plan's ({info['variant']} streamk={info['streamk']})"
        rows, cols = sample_rows_cols(M, N, n_rows=128, n_cols=128, seed=call)
        Cref, S = oracle_mod.sgemm_ref(np.ascontiguousarray(A[rows]), np.ascontiguousarray(B[:, cols]),
                                       np.ascontiguousarray(C0[np.ix_(rows, cols)]), alpha, beta)
        err = np.abs(got_h[np.ix_(rows, cols)].astype(np.float64) - Cref)
        assert np.all(err <= oracle_mod.acceptance_bound(K, S)), f"call {call}: outside the acceptance bound"
    plan.close()
    if shape == (2048, 4096, 1024):
        assert info["streamk"] == 1  # 256 tiles on 152 CTAs: the scratch is used


@pytest.mark.gpu
def test_static_scratch_makes_no_allocation(sg):
    M, N, K = 2048, 4096, 1024
    A, B, C0 = make_inputs(M, N, K, seed=5)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dC = torch.from_numpy(C0).cuda()
    _static(sg, M, N, K, 1.0, dA, dB, 0.0, dC)  # set-up happens here if no earlier call did it
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for i in range(5):
        _static(sg, M, N, K, 1.0, dA, dB, 0.5, dC)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"device memory changed across calls: {free0} -> {free1}"
    assert sg.device_status() == sg.SGEMM_OK


@pytest.mark.gpu
def test_static_scratch_rejections(sg):
    M, N, K = 256, 512, 256
    A, B, C0 = make_inputs(M, N, K, seed=6)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dC = torch.from_numpy(C0).cuda()
    with pytest.raises(sg.SgemmError) as e:  # lda not a multiple of 4
        _static(sg, M, N, K - 2, 1.0, dA, dB, 0.0, dC, lda=K - 2)
    assert e.value.status == sg.SGEMM_ERR_UNSUPPORTED
    with pytest.raises(sg.SgemmError) as e:  # A not 16-byte aligned
        _static(sg, M, N, K - 4, 1.0, dA.data_ptr() + 4, dB, 0.0, dC, lda=K)
    assert e.value.status == sg.SGEMM_ERR_UNSUPPORTED
    with pytest.raises(sg.SgemmError) as e:  # lda < K
        _static(sg, M, N, K, 1.0, dA, dB, 0.0, dC, lda=K - 4)
    assert e.value.status == sg.SGEMM_ERR_INVALID_ARG
    with pytest.raises(sg.SgemmError) as e:  # C missing
        _static(sg, M, N, K, 1.0, dA, dB, 0.0, 0)
    assert e.value.status == sg.SGEMM_ERR_INVALID_ARG
    # C sharing its span with A or B is refused, as sgemm_run refuses it;
    # A and B may alias each other
    buf = torch.zeros(3 * 64 * 64, device="cuda")
    a, b, c = buf.data_ptr(), buf.data_ptr() + 4 * 64 * 64, buf.data_ptr() + 8 * 64 * 64
    _static(sg, 64, 64, 64, 1.0, a, b, 0.0, c)  # disjoint spans: fine
    for cc in (a, b, b + 4 * 100):
        with pytest.raises(sg.SgemmError) as e:
            _static(sg, 64, 64, 64, 1.0, a, b, 0.0, cc)
        assert e.value.status == sg.SGEMM_ERR_UNSUPPORTED
    _static(sg, 64, 64, 64, 1.0, a, a, 0.0, c)
    _static(sg, 0, N, K, 1.0, dA, dB, 0.0, 0)  # empty: nothing to do
    # K == 0: C = beta * C, A and B not read
    _static(sg, M, N, 0, 1.0, 0, 0, 2.0, dC, lda=1)
    torch.cuda.synchronize()
    assert np.array_equal(dC.cpu().numpy(), (np.float32(2.0) * C0).astype(np.float32))
    assert sg.device_status() == sg.SGEMM_OK
