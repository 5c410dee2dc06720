"""The allocation-free tf32 entry point against the plan-based one (needs a GB300).

b2b_run_tf32_noalloc serves callers that cannot allocate device memory: it
uses a fixed scratch array owned by the library instead of a plan's
workspace.  Its results must match b2b_run on a B2B_TF32 plan, on two calls
in a row with different inputs (the shared scratch keeps the previous call's
contents, which must not leak into the next result).  This file is collected
last on purpose, so that a run stopping at the first failure has run every
other test already.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu

b2b = pytest.importorskip("fusion_b2b_gemm_gb300")

TOL = 5e-3      # the tf32 tolerance of the parity tests


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


def _rel(got, want):
    got, want = got.double(), want.double()
    return float((got - want).abs().max() / want.abs().max().clamp_min(1e-300))


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
        got = torch.full_like(want, float("nan"))
        _noalloc(w, dev, got)
        torch.cuda.synchronize()
        assert torch.isfinite(got).all()
        assert _rel(got, want) <= TOL


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
    assert _rel(out1, want1) <= TOL
    assert _rel(out2, want2) <= TOL
    assert not torch.equal(out1, out2)


def test_rejects_sizes_beyond_the_scratch_array():
    # batch * (K*N1 + N1*N2) = 16 * (256*256 + 256*256) > 2^20 words
    A = torch.zeros(16, dtype=torch.float32, device="cuda")
    code = b2b.b2b_run_tf32_noalloc(16, 128, 256, 256, 256, A.data_ptr(), A.data_ptr(), A.data_ptr(),
                                    A.data_ptr(), None)
    assert code == 2
