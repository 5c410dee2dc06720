"""Host-side logic that needs no GPU: workload shapes and storage types, the
bench's roofline arithmetic, and how an end-to-end call is cut into chunks."""
import numpy as np
import pytest
import torch

import bench
import workloads as wl


def test_input_types_of_mixed_workloads():
    w = wl.ALL_WORKLOADS["mixed_tf32_bf16"]
    assert wl.input_dtypes(w.dtype, w.stages) == [torch.float32, torch.float32, torch.bfloat16, torch.bfloat16]
    host = wl.make_inputs(w.with_(M=8))
    assert [t.dtype for t in host] == [torch.float32, torch.float32, torch.bfloat16, torch.bfloat16]
    assert [tuple(t.shape) for t in host] == [s for s in w.with_(M=8).shapes()]
    # one type throughout for the others; draws unchanged by the mixed types
    for name in wl.WORKLOADS:
        v = wl.WORKLOADS[name]
        assert len(set(wl.input_dtypes(v.dtype, v.stages))) == 1


def test_unique_bytes_count_each_input_in_its_own_type():
    w = wl.ALL_WORKLOADS["mixed_tf32_bf16"]
    a, w0, w1, w2 = (int(np.prod(s)) for s in w.shapes())
    assert w.unique_bytes() == 4 * (a + w0) + 2 * (w1 + w2) + 4 * w.batch * w.M * w.N[-1]
    c2 = wl.WORKLOADS["batched_f16"]
    assert c2.unique_bytes() == 138_412_032


def test_roofline_picks_the_binding_side():
    peaks = {"hbm_gbs": 6683.5, "tensor": {"f16": 1920.8, "bf16": 1920.8, "tf32": 960.0}}
    c2 = wl.WORKLOADS["batched_f16"]
    r = bench.roofline_for(c2, 0.026, peaks)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(c2.unique_bytes() / 26e-6 / 1e9)
    c5 = wl.WORKLOADS["three_stage_bf16"]
    r = bench.roofline_for(c5, 0.0424, peaks)
    assert r["bound"] == "tensor" and r["frac"] == pytest.approx(c5.flops() / 42.4e-6 / 1e12 / 1920.8)


def test_roofline_of_a_mixed_cascade_blends_the_two_rates():
    peaks = {"hbm_gbs": 1e9, "tensor": {"bf16": 2000.0, "tf32": 1000.0}}  # compute-bound
    w = wl.ALL_WORKLOADS["mixed_tf32_bf16"]
    r = bench.roofline_for(w, 1.0, peaks)
    f0 = 2 * w.batch * w.M * w.K * w.N[0]
    t = f0 / 1000e12 + (w.flops() - f0) / 2000e12
    assert r["bound"] == "tensor"
    assert r["peak"] == pytest.approx(w.flops() / t / 1e12)
    assert 1000.0 < r["peak"] < 2000.0


def test_compute_types_reported_by_the_bench():
    for name, w in wl.ALL_WORKLOADS.items():
        assert w.dtype in bench.COMPUTE_DTYPE
    assert bench.COMPUTE_DTYPE["tf32_bf16"] == "tf32+bf16"


class _Shape:
    """Stand-in with the attributes Plan._host_chunks reads."""

    def __init__(self, batch, M):
        self.batch, self.M = batch, M


def _chunks(batch, M, chunks, nbytes=1 << 30):
    import fusion_b2b_gemm_gb300 as b2b
    return b2b.Plan._host_chunks(_Shape(batch, M), chunks, nbytes)


@pytest.mark.parametrize("batch,M,chunks", [(64, 4096, 4), (3, 100, 4), (1, 65536, 4), (1, 1000, 3),
                                            (1, 200, 4), (7, 1, 2), (1, 70000, 16)])
def test_end_to_end_chunks_cover_the_work_once(batch, M, chunks):
    pieces = _chunks(batch, M, chunks)
    assert pieces[0][0] == 0
    assert all(a[1] == b[0] for a, b in zip(pieces, pieces[1:]))
    assert all(hi > lo for lo, hi in pieces)
    if batch > 1:
        assert pieces[-1][1] == batch and len(pieces) == min(chunks, batch)
    else:
        assert pieces[-1][1] == M
        # row chunks start on 256-row boundaries (whole tiles of either kernel)
        assert all(lo % 256 == 0 for lo, _ in pieces)


def test_end_to_end_chunk_count_follows_the_size():
    assert len(_chunks(64, 4096, None, nbytes=138 << 20)) == 4
    assert len(_chunks(64, 4096, None, nbytes=34 << 20)) == 2
    assert len(_chunks(64, 4096, None, nbytes=1 << 20)) == 1


def test_compact_per_config_records_stay_short():
    """The headline line ends with one short record per workload, so that the
    last 1.5 KB of the output hold all nine."""
    import json
    w = wl.ALL_WORKLOADS["three_stage_bf16"]
    peaks = {"hbm_gbs": 6683.5, "tensor": {"bf16": 1920.8}}
    entry = {"workload": "three_stage_bf16", "fused_ms": 0.041312345, "unfused_torch_ms": 0.0449876,
             "unfused_own_ms": None, "speedup_vs_best_unfused": 1.08912345, "fused_tflops": 1039.9876,
             "roofline": bench.roofline_for(w, 0.041312345, peaks), "cpu_oracle": {"value": 0.0241234567}}
    c = bench.compact_config(entry)
    assert c["fused_us"] == 41.3 and c["own_us"] is None and c["speedup"] == 1.09
    assert c["bound"] == "tensor" and c["frac"] == round(c["frac"], 3)
    assert len(json.dumps(c)) * len(wl.ALL_WORKLOADS) < 1500
