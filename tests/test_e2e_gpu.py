"""End-to-end calls from pinned host buffers (needs a GB300): the pipelined
form (chunks over the batch or the rows, copies on side streams) gives the
same result as one device call."""
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu

b2b = pytest.importorskip("fusion_b2b_gemm_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    torch.cuda.set_device(0)


CASES = [
    wl.Workload("e2e_batched_f16", "f16", 12, 700, 128, (128, 128), "normal_fanin", 1.0, 81),
    wl.Workload("e2e_rows_bf16_3", "bf16", 1, 3000, 256, (256, 128, 320), "normal_fanin", 1.0, 82),
    wl.Workload("e2e_tf32", "tf32", 3, 1000, 128, (128, 64), "normal", 1.0 / 16, 83),
    wl.Workload("e2e_mixed", "tf32_f16", 1, 1500, 64, (256, 128), "normal_fanin", 1.0, 84),
    wl.Workload("e2e_f64", "f64", 5, 300, 64, (64, 32), "uniform", 1.0, 85),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("chunks", [1, 3])
def test_pipelined_call_matches_device_call(w, chunks):
    host = [t.pin_memory() for t in wl.make_inputs(w)]
    dev = [t.cuda() for t in host]
    plan = b2b.ChainPlan(w.dtype, w.batch, w.M, w.K, w.N)
    want = plan.run(dev[0], dev[1:]).cpu()
    dev_in = [torch.empty_like(t) for t in dev]
    dev_out = plan.empty_out()
    host_out = torch.empty(plan.out_shape(), dtype=plan.io_dtypes()[1]).pin_memory()
    s = torch.cuda.Stream()
    h2d, d2h = plan.run_from_host(host, host_out, dev_in, dev_out, stream=s, chunks=chunks)
    s.synchronize()
    assert plan.status() == 0
    assert h2d == sum(t.numel() * t.element_size() for t in host)
    assert d2h == host_out.numel() * host_out.element_size()
    assert torch.equal(host_out.view(torch.uint8), want.view(torch.uint8))
