"""Failure detection without a GPU fault (needs a GB300).

Every wait inside the tensor-core kernels has a time budget.  The test knob
B2B_DEBUG_DROP_FIRST_LOAD arms the first shared-memory stage of every CTA
but never fills it, so the MMA thread's wait on it runs out.  The kernel must
then unwind by itself (no trap, no hang), the plan's status word must report
B2B_ERR_TIMEOUT, and the same plan must compute correct results on the next
normal run.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

b2b = pytest.importorskip("fusion_b2b_gemm_gb300")

TIMEOUT = 7
KINDS = {"f16": (oracle.F32, oracle.F16, oracle.F16), "bf16": (oracle.F32, oracle.BF16, oracle.BF16),
         "tf32": (oracle.F32, oracle.TF32, oracle.F32), "tf32_bf16": (oracle.F32, oracle.BF16, oracle.F32)}
TOL = {"f16": 1e-2, "bf16": 1e-2, "tf32": 5e-3, "tf32_bf16": 1e-2}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    torch.cuda.set_device(0)


CASES = [
    wl.Workload("fail_res_f16", "f16", 2, 512, 128, (128, 128), "normal_fanin", 1.0, 51),
    wl.Workload("fail_stream_bf16_3", "bf16", 1, 384, 512, (256, 256, 512), "normal_fanin", 1.0, 52),
    wl.Workload("fail_tf32", "tf32", 1, 384, 256, (256, 256), "normal", 1.0 / 16, 53),
    wl.Workload("fail_deep5_f16", "f16", 1, 600, 128, (256, 512, 128, 256, 384), "normal_fanin", 1.0, 54),
    wl.Workload("fail_mixed_bf16", "tf32_bf16", 1, 400, 64, (256, 128, 256), "normal_fanin", 1.0, 55),
    # resident weights over many batches: CTAs walk the batch-aware schedule
    wl.Workload("fail_sched_f16", "f16", 40, 2000, 128, (128, 128), "normal_fanin", 1.0, 56),
    # a tf32 chain on CTA pairs with one unit per cluster (the set-up barrier
    # passed before the L2 prefetches are issued)
    wl.Workload("fail_one_tile_tf32", "tf32", 1, 4096, 128, (128, 256), "normal", 1.0 / 16, 57),
    # a tf32 chain on CTA pairs, several units per cluster
    wl.Workload("fail_tf32_pairs", "tf32", 2, 10000, 64, (128, 128), "normal", 1.0 / 16, 58),
    # the one-CTA tf32 kernel (a last GEMM wider than 256 columns), one tile
    # per CTA, output staged in the ring
    wl.Workload("fail_tf32_one_cta", "tf32", 1, 4096, 128, (128, 384), "normal", 1.0 / 16, 59),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_timeout_is_reported_and_the_plan_recovers(w):
    host = wl.make_inputs(w)
    dev = [t.cuda() for t in host]
    plan = b2b.ChainPlan(w.dtype, w.batch, w.M, w.K, w.N)
    out = plan.empty_out()
    out.fill_(0)
    plan.set_wait_budget(20_000_000)          # 20 ms
    plan.set_debug(1)
    t0 = time.perf_counter()
    plan.run(dev[0], dev[1:], D=out)
    status = plan.status()                    # synchronises
    elapsed = time.perf_counter() - t0
    assert status == TIMEOUT
    assert elapsed < 5.0
    assert torch.all(out == 0)                # nothing was stored
    assert plan.status() == 0                 # the status word was cleared
    # the context and the plan are healthy: a normal run is correct
    plan.set_debug(0)
    plan.set_wait_budget(0)
    plan.run(dev[0], dev[1:], D=out)
    assert plan.status() == 0
    acc, mid, fin = KINDS[w.dtype]
    want = oracle.chain(oracle.widen(host[0]), [oracle.widen(t) for t in host[1:]], acc, mid, fin)
    got = out.double().cpu().numpy()
    assert np.max(np.abs(got - want)) / np.max(np.abs(want)) <= TOL[w.dtype]


def test_debug_flags_are_validated():
    plan = b2b.Plan("f16", 1, 128, 64, 64, 64)
    with pytest.raises(b2b.B2BError) as e:
        plan.set_debug(2)
    assert e.value.code == 1
