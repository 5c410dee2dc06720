"""The allocation-free tf32 entry point against the plan-based one (needs a GB300).

b2b_run_tf32_noalloc serves callers that cannot allocate device memory (for
example code running inside a framework that owns all of the GPU's memory, or
callers that must not create plans, which own device memory): it uses a fixed
scratch array owned by the library instead of a plan's workspace.  It runs
the same kernels as b2b_run on a B2B_TF32 plan, so its results must be
identical to that path's, bit for bit, on two calls in a row with different
inputs (the shared scratch keeps the previous call's contents, which must not
leak into the next result); a call that fills the scratch array exactly is
also checked against the CPU oracle.  This file is collected last on purpose,
so that a run stopping at the first failure has run every other test already.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

b2b = pytest.importorskip("fusion_b2b_gemm_gb300")

TOL = 5e-3          # the tf32 tolerance of the parity tests
SCRATCH_WORDS = 1 << 20


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    torch.cuda.set_device(0)


def _noalloc(w, dev, out):
    A, B, C = dev
    code = b2b.b2b_run_tf32_noalloc(w.batch, w.M, w.K, w.N[0], w.N[1], A.data_ptr(), B.data_ptr(),
                                    C.data_ptr(), out.data_ptr(),
                                    torch.cuda.current_stream().cuda_stream or None)
    assert code == 0, b2b.b2b_status_string(code).decode()


def _oracle(host):
    A = oracle.widen(host[0])
    return oracle.chain(A, [oracle.widen(t) for t in host[1:]], oracle.F32, oracle.TF32, oracle.F32)


def _rel(got, want):
    got = got.double().cpu().numpy()
    return float(np.max(np.abs(got - want)) / max(np.max(np.abs(want)), 1e-300))


def test_two_calls_in_a_row_match_the_plan_path():
    shapes = [wl.Workload("na1", "tf32", 1, 640, 256, (256, 256), "normal", 1.0 / 16, 41),
              wl.Workload("na2", "tf32", 2, 300, 128, (192, 136), "normal", 1.0 / 16, 42),
              # more 128-row tiles than SMs: the CTA-pair kernel
              wl.Workload("na_pairs", "tf32", 2, 10000, 64, (96, 128), "normal", 1.0 / 16, 44)]
    for w in shapes:
        host = wl.make_inputs(w)
        dev = [t.cuda() for t in host]
        plan = b2b.Plan("tf32", w.batch, w.M, w.K, *w.N)
        want = plan.run(*dev).clone()
        for _ in range(2):
            got = torch.full_like(want, float("nan"))
            _noalloc(w, dev, got)
            torch.cuda.synchronize()
            assert torch.equal(got, want), w.name
        assert plan.status() == 0


def test_back_to_back_calls_with_different_inputs():
    w = wl.Workload("na3", "tf32", 1, 512, 256, (256, 128), "normal", 1.0 / 16, 43)
    first = [t.cuda() for t in wl.make_inputs(w, seed=101)]
    second = [t.cuda() for t in wl.make_inputs(w, seed=102)]
    plan = b2b.Plan("tf32", w.batch, w.M, w.K, *w.N)
    want1 = plan.run(*first).clone()
    want2 = plan.run(*second).clone()
    out1 = torch.empty_like(want1)
    out2 = torch.empty_like(want2)
    _noalloc(w, first, out1)
    _noalloc(w, second, out2)
    torch.cuda.synchronize()
    assert torch.equal(out1, want1)
    assert torch.equal(out2, want2)
    assert not torch.equal(out1, out2)


def test_a_call_that_fills_the_scratch_array_exactly():
    # batch * (K*N1 + N1*N2) = 8 * (256*256 + 256*256) = 2^20 words: the
    # transposed weights of the last batch end at the array's last word
    w = wl.Workload("na_full", "tf32", 8, 200, 256, (256, 256), "normal", 1.0 / 16, 45)
    assert w.batch * (w.K * w.N[0] + w.N[0] * w.N[1]) == SCRATCH_WORDS
    host = wl.make_inputs(w)
    dev = [t.cuda() for t in host]
    want = _oracle(host)
    plan = b2b.Plan("tf32", w.batch, w.M, w.K, *w.N)
    via_plan = plan.run(*dev).clone()
    for _ in range(2):
        got = torch.full_like(via_plan, float("nan"))
        _noalloc(w, dev, got)
        torch.cuda.synchronize()
        assert torch.equal(got, via_plan)
        assert _rel(got, want) <= TOL


def test_rejects_sizes_beyond_the_scratch_array():
    A = torch.zeros(16, dtype=torch.float32, device="cuda")
    # 16 * (256*256 + 256*256) words, and the smallest step past the limit:
    # 8 * (260*256 + 256*256)
    for batch, K in ((16, 256), (8, 260)):
        assert batch * (K * 256 + 256 * 256) > SCRATCH_WORDS
        code = b2b.b2b_run_tf32_noalloc(batch, 128, K, 256, 256, A.data_ptr(), A.data_ptr(), A.data_ptr(),
                                        A.data_ptr(), None)
        assert code == 2
