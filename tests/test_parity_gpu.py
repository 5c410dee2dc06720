"""Parity of the CUDA path with the CPU oracle (needs a GB300).

Every call goes through the C ABI (via the thin binding).  Bars:
  - integer-valued inputs: bit-exact (every product and partial sum is an
    integer below 2^24, so fp32 accumulation is exact and both sides round
    the same exact values);
  - random inputs: max|gpu - oracle| / max|oracle| <= 1e-2 (fp16, bf16),
    5e-3 (tf32), 1e-12 (fp64);
  - full-size workloads: the same bound on sampled rows, which the oracle
    computes one by one.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

b2b = pytest.importorskip("fusion_b2b_gemm_gb300")

KINDS = {
    "f16_f32out": (oracle.F32, oracle.F16, oracle.F32),
    "f16": (oracle.F32, oracle.F16, oracle.F16),
    "bf16": (oracle.F32, oracle.BF16, oracle.BF16),
    "bf16_f32out": (oracle.F32, oracle.BF16, oracle.F32),
    "tf32": (oracle.F32, oracle.TF32, oracle.F32),
    "f64": (oracle.NONE, oracle.NONE, oracle.NONE),
    # mixed: tf32 first GEMM, 16-bit intermediates and later GEMMs, fp32 out
    "tf32_f16": (oracle.F32, oracle.F16, oracle.F32),
    "tf32_bf16": (oracle.F32, oracle.BF16, oracle.F32),
}
TOL = {"f16_f32out": 1e-2, "f16": 1e-2, "bf16": 1e-2, "bf16_f32out": 1e-2, "tf32": 5e-3, "f64": 1e-12,
       "tf32_f16": 1e-2, "tf32_bf16": 1e-2}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    torch.cuda.set_device(0)


def run_gpu(w, host):
    dev = [t.cuda() for t in host]
    if w.stages <= 3:
        plan = b2b.Plan(w.dtype, w.batch, w.M, w.K, *w.N)
        out = plan.run(*dev)
    else:
        plan = b2b.ChainPlan(w.dtype, w.batch, w.M, w.K, w.N)
        out = plan.run(dev[0], dev[1:])
    torch.cuda.synchronize()
    assert plan.status() == 0
    return out.cpu()


def run_oracle(w, host, rows=None, batches=None):
    A = oracle.widen(host[0])
    Ws = [oracle.widen(t) for t in host[1:]]
    if batches is not None:
        A = A[batches]
        Ws = [x[batches] for x in Ws]
    if rows is not None:
        A = A[:, rows]
    acc, mid, fin = KINDS[w.dtype]
    return oracle.chain(A, Ws, acc, mid, fin)


def rel_err(got, want):
    got = got.double().numpy() if isinstance(got, torch.Tensor) else got
    return float(np.max(np.abs(got - want)) / max(np.max(np.abs(want)), 1e-300))


def bits_equal(got: torch.Tensor, want: np.ndarray, dtype: str) -> bool:
    """Exact equality of every output value (the oracle's values are already
    rounded to the output type; +0 and -0 compare equal)."""
    _, out_dt = wl.io_dtypes(dtype)
    want_t = torch.from_numpy(want).to(out_dt)
    return bool(torch.equal(got.double(), want_t.double()))


# ------------------------------------------------------------ bit-exact --

EXACT = [
    wl.Workload("x_f16_f32out", "f16_f32out", 2, 300, 64, (64, 64), "int", 2, 11),
    wl.Workload("x_f16", "f16", 3, 257, 128, (128, 128), "int", 2, 12),
    wl.Workload("x_bf16_3", "bf16", 1, 300, 512, (256, 256, 512), "int", 1, 13),
    wl.Workload("x_tf32", "tf32", 1, 333, 256, (256, 256), "int", 2, 14),
    # a single 128-row tile: the one-CTA kernel (two or more go to CTA pairs)
    wl.Workload("x_tf32_one_tile", "tf32", 1, 128, 256, (256, 256), "int", 2, 95),
    wl.Workload("x_f64", "f64", 2, 77, 64, (64, 64), "int", 2, 15),
    # three-stage chains run as CTA pairs sharing each MMA (256-row tiles):
    # padded narrow widths, batches whose last pair tile is half past M, the
    # final GEMM in one, two (Z buffers) or three passes
    wl.Workload("x_f16_3_narrow", "f16", 3, 384, 64, (64, 64, 64), "int", 1, 16),
    wl.Workload("x_bf16_f32out_3", "bf16_f32out", 2, 200, 128, (128, 128, 256), "int", 1, 17),
    wl.Workload("x_f16_f32out_3", "f16_f32out", 1, 700, 192, (96, 160, 384), "int", 1, 18),
    # longer cascades and intermediates wider than 256 columns (every
    # partial sum stays below 2^24: |value| <= K * N1 * N2 ...)
    wl.Workload("x_f16_4", "f16", 2, 300, 32, (32, 32, 32, 64), "int", 1, 19),
    wl.Workload("x_f16_f32out_5", "f16_f32out", 1, 520, 16, (16, 16, 16, 16, 128), "int", 1, 20),
    wl.Workload("x_bf16_wide384", "bf16", 1, 300, 32, (384, 64), "int", 1, 41),
    wl.Workload("x_bf16_wide512_3", "bf16", 1, 260, 16, (512, 16, 256), "int", 1, 42),
    # intermediates partly in tensor memory, partly in the operand image:
    # the first (the next one fits a region) and the last (one final pass)
    # are packed in tensor memory, the 256- and 384-column ones between go
    # through shared memory
    wl.Workload("x_bf16_5_mixed_homes", "bf16", 1, 300, 16, (128, 256, 384, 128, 256), "int", 1, 97),
    # mixed types: tf32 first GEMM (integers below 2^10 are exact in tf32),
    # then fp16 / bf16
    wl.Workload("x_tf32_f16_2", "tf32_f16", 2, 300, 64, (128, 64), "int", 2, 71),
    wl.Workload("x_tf32_bf16_4", "tf32_bf16", 1, 520, 32, (256, 32, 32, 256), "int", 1, 72),
    # a tf32 chain with more 128-row tiles than SMs runs on CTA pairs, its
    # intermediate kept in tensor memory (ragged widths)
    wl.Workload("x_tf32_pairs", "tf32", 4, 5000, 96, (200, 136), "int", 2, 87),
    # tf32 weights read as stored with widths that are not a multiple of 32
    # columns (one 32-column box at a time, the last one partly past N): the
    # pair kernel, the one-CTA kernel (a single tile) and the first GEMM of a
    # mixed-type cascade
    wl.Workload("x_tf32_ragged", "tf32", 2, 300, 60, (200, 136), "int", 2, 93),
    wl.Workload("x_tf32_ragged_one_tile", "tf32", 1, 100, 60, (200, 136), "int", 2, 98),
    wl.Workload("x_tf32_bf16_ragged", "tf32_bf16", 1, 300, 36, (72, 40, 104), "int", 1, 94),
]


@pytest.mark.parametrize("w", EXACT, ids=lambda w: w.name)
def test_integer_inputs_bit_exact(w):
    host = wl.make_inputs(w)
    got = run_gpu(w, host)
    want = run_oracle(w, host)
    assert np.max(np.abs(want)) < 2 ** 24
    assert bits_equal(got, want, w.dtype), f"max abs diff {np.max(np.abs(got.double().numpy() - want))}"


# ------------------------------------------------------ random, reduced --

REDUCED = [
    wl.small(wl.WORKLOADS["tiny_f16"], M=256),
    wl.small(wl.WORKLOADS["batched_f16"], M=500, batch=3),
    wl.small(wl.WORKLOADS["tf32"], M=640),
    wl.small(wl.WORKLOADS["f64"], M=200, batch=3),
    wl.small(wl.WORKLOADS["three_stage_bf16"], M=520),
    wl.small(wl.EXTRA_WORKLOADS["four_stage_bf16"], M=777),
    wl.small(wl.EXTRA_WORKLOADS["wide_f16"], M=600, batch=2),
]


@pytest.mark.parametrize("w", REDUCED, ids=lambda w: w.name)
def test_random_inputs_within_tolerance(w):
    host = wl.make_inputs(w)
    got = run_gpu(w, host)
    want = run_oracle(w, host)
    err = rel_err(got, want)
    assert err <= TOL[w.dtype], err


# ---------------------------------------------------------- edge cases --

EDGES = [
    wl.Workload("m1_f16", "f16_f32out", 1, 1, 64, (64, 64), "uniform", 1.0, 21),
    wl.Workload("m5_batch3_f16", "f16", 3, 5, 128, (128, 128), "normal_fanin", 1.0, 22),
    wl.Workload("narrow_n_f16", "f16_f32out", 2, 130, 64, (40, 56), "uniform", 1.0, 23),
    wl.Workload("ragged_n_f16", "f16", 1, 129, 128, (96, 120), "normal_fanin", 1.0, 24),
    wl.Workload("k_tail_f16", "f16", 2, 140, 72, (128, 128), "normal_fanin", 1.0, 25),
    wl.Workload("n3_partial_bf16", "bf16", 1, 150, 512, (256, 256, 320), "normal_fanin", 1.0, 26),
    wl.Workload("ragged_tf32", "tf32", 1, 190, 256, (200, 136), "normal", 1.0 / 16, 27),
    wl.Workload("ragged_tf32_one_tile", "tf32", 1, 77, 60, (200, 136), "normal", 1.0 / 16, 96),
    wl.Workload("m13_f64", "f64", 3, 13, 64, (64, 64), "uniform", 1.0, 28),
    wl.Workload("small_f64", "f64", 2, 40, 32, (32, 16), "uniform", 1.0, 29),
    wl.Workload("n1_192_f16", "f16", 2, 200, 64, (192, 136), "normal_fanin", 1.0, 30),
    wl.Workload("n1_160_tf32", "tf32", 2, 150, 128, (160, 200), "normal", 1.0 / 16, 31),
    wl.Workload("n2_176_bf16_3", "bf16", 1, 140, 64, (176, 144, 200), "normal_fanin", 1.0, 32),
    wl.Workload("m100_bf16_3", "bf16", 1, 100, 64, (256, 128, 72), "normal_fanin", 1.0, 33),
    wl.Workload("batch3_m384_f16_3", "f16", 3, 384, 64, (128, 64, 128), "normal_fanin", 1.0, 34),
    wl.Workload("k_tail_bf16_3", "bf16", 2, 300, 200, (128, 128, 128), "normal_fanin", 1.0, 35),
    # streamed weights with more tiles than SMs: A panels through their own ring
    wl.Workload("streamed_many_f16", "f16", 1, 40000, 512, (128, 128), "normal_fanin", 1.0, 36),
    wl.Workload("streamed_many_tf32", "tf32", 2, 10000, 96, (64, 64), "normal", 1.0 / 16, 37),
    wl.Workload("streamed_many_bf16_npass", "bf16", 1, 20000, 64, (128, 384), "normal_fanin", 1.0, 38),
    # resident weights over many batches: the batch-aware tile schedule, with
    # CTAs that take the leftover tiles of two batches
    wl.Workload("sched_res_f16", "f16", 40, 2000, 128, (128, 128), "normal_fanin", 1.0, 39),
    wl.Workload("sched_res_bf16_f32out", "bf16_f32out", 33, 1100, 64, (64, 128), "normal_fanin", 1.0, 40),
    # longer cascades (one kernel for every stage) and wide intermediates
    wl.Workload("deep6_bf16", "bf16", 1, 520, 256, (256, 128, 256, 192, 256, 320), "normal_fanin", 1.0, 43),
    wl.Workload("eight_f16", "f16", 1, 260, 64, (128,) * 7 + (64,), "normal_fanin", 1.0, 44),
    wl.Workload("wide512_f16_3", "f16", 1, 700, 128, (512, 512, 256), "normal_fanin", 1.0, 45),
    wl.Workload("wide384_bf16_3", "bf16_f32out", 2, 300, 64, (384, 200, 136), "normal_fanin", 1.0, 46),
    wl.Workload("wide512_bf16_2", "bf16", 1, 300, 96, (512, 1000), "normal_fanin", 1.0, 47),
    wl.Workload("wide_tail_f16_4", "f16", 1, 129, 72, (264, 40, 392, 8), "normal_fanin", 1.0, 48),
    wl.Workload("streamed_many_bf16_4", "bf16", 1, 40000, 128, (128, 128, 128, 512), "normal_fanin", 1.0, 49),
    # mixed types: ragged K (a partial 32-element tf32 panel), wide first
    # intermediate, several stages, more tiles than clusters
    wl.Workload("mixed_f16_ktail", "tf32_f16", 2, 333, 200, (256, 136), "normal_fanin", 1.0, 73),
    # the largest sizes a plan takes: eight GEMMs, 512-wide intermediates and
    # a 4096-wide last GEMM; a long K; one row
    wl.Workload("max_widths_f16_8", "f16", 1, 300, 2048, (512,) * 7 + (4096,), "normal_fanin", 1.0, 79),
    wl.Workload("long_k_bf16", "bf16", 2, 257, 8192, (256, 256), "normal_fanin", 1.0, 80),
    wl.Workload("one_row_bf16_8", "bf16_f32out", 2, 1, 64, (128, 512, 64, 256, 384, 8, 512, 72), "normal_fanin", 1.0, 86),
    # K = 4 mod 8: fp32 rows of A are 16-byte aligned, 16-bit ones would not be
    wl.Workload("mixed_bf16_k4mod8", "tf32_bf16", 2, 260, 92, (328, 216), "normal_fanin", 1.0, 77),
    wl.Workload("tf32_k4mod8", "tf32", 2, 300, 68, (96, 200), "normal", 1.0 / 16, 78),
    wl.Workload("mixed_bf16_wide", "tf32_bf16", 1, 300, 128, (512, 128, 384), "normal_fanin", 1.0, 74),
    wl.Workload("mixed_f16_5", "tf32_f16", 1, 700, 96, (128, 256, 128, 256, 72), "normal_fanin", 1.0, 75),
    wl.Workload("mixed_bf16_many", "tf32_bf16", 1, 30000, 256, (256, 256), "normal_fanin", 1.0, 76),
    # tf32 chains on CTA pairs (more 128-row tiles than SMs): a partial K
    # panel, a 128-column last pass, a last pair tile whose odd half lies
    # wholly past M
    wl.Workload("tf32_pairs_ktail", "tf32", 2, 10000, 68, (256, 256), "normal", 1.0 / 16, 88),
    wl.Workload("tf32_pairs_n128", "tf32", 1, 20000, 256, (128, 96), "normal", 1.0 / 16, 89),
    wl.Workload("tf32_pairs_mtail", "tf32", 3, 7000, 32, (72, 256), "normal", 1.0 / 16, 90),
    # a tf32 chain with more tiles than SMs but a last GEMM wider than 256
    # columns stays on the one-CTA kernel, several tiles per CTA
    wl.Workload("tf32_wide_many_tiles", "tf32", 2, 10000, 64, (128, 384), "normal", 1.0 / 16, 92),
]


@pytest.mark.parametrize("w", EDGES, ids=lambda w: w.name)
def test_edge_shapes(w):
    host = wl.make_inputs(w)
    got = run_gpu(w, host)
    want = run_oracle(w, host)
    assert rel_err(got, want) <= TOL[w.dtype]


def test_tf32_chains_take_pairs_from_two_tiles():
    # a single 128-row tile, or a last GEMM wider than 256 columns: the
    # one-CTA kernel; two tiles or more: CTA pairs (384 threads, an even grid)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    one = b2b.Plan("tf32", 1, 128, 256, 256, 256).info()
    wide = b2b.Plan("tf32", 1, 128 * sms, 256, 256, 384).info()
    for m in (129, 128 * sms, 128 * sms + 1):
        many = b2b.Plan("tf32", 1, m, 256, 256, 256).info()
        assert many["threads"] == 384 and many["grid"] % 2 == 0
    assert one["threads"] != 384 and wide["threads"] != 384


def test_empty_chain_is_a_no_op():
    plan = b2b.Plan("f16", 1, 0, 64, 64, 64)
    assert plan.info()["launches_per_run"] == 0
    a = torch.zeros(16, dtype=torch.float16, device="cuda")
    d = torch.full((16,), 7.0, dtype=torch.float16, device="cuda")
    plan.run(a, a, a, None, d)
    torch.cuda.synchronize()
    assert torch.all(d == 7.0)


def test_chain_plan_matches_plan_bitwise():
    """The S-stage interface and the three-argument one run the same kernel."""
    w = wl.small(wl.WORKLOADS["three_stage_bf16"], M=300)
    host = wl.make_inputs(w)
    dev = [t.cuda() for t in host]
    a = b2b.Plan(w.dtype, w.batch, w.M, w.K, *w.N).run(*dev)
    b = b2b.ChainPlan(w.dtype, w.batch, w.M, w.K, w.N).run(dev[0], dev[1:])
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_chain_plan_of_one_and_two_stages():
    """ChainPlan with one or two widths runs the single-GEMM and two-stage plans."""
    for N in ((128,), (128, 64)):
        w = wl.Workload("short", "f16_f32out", 2, 200, 64, N, "normal_fanin", 1.0, 61)
        host = wl.make_inputs(w)
        plan = b2b.ChainPlan(w.dtype, w.batch, w.M, w.K, w.N)
        out = plan.run(host[0].cuda(), [t.cuda() for t in host[1:]])
        torch.cuda.synchronize()
        assert plan.status() == 0
        want = oracle.chain(oracle.widen(host[0]), [oracle.widen(t) for t in host[1:]],
                            oracle.F32, oracle.F16, oracle.F32)
        assert rel_err(out.cpu(), want) <= 1e-2


def test_more_than_three_stages_need_chain_run():
    plan = b2b.ChainPlan("f16", 1, 128, 64, (64, 64, 64, 64))
    A = torch.zeros((1, 128, 64), dtype=torch.float16, device="cuda")
    W = torch.zeros((1, 64, 64), dtype=torch.float16, device="cuda")
    D = torch.zeros((1, 128, 64), dtype=torch.float16, device="cuda")
    assert b2b.b2b_run(plan._h, A.data_ptr(), W.data_ptr(), W.data_ptr(), W.data_ptr(),
                       D.data_ptr(), None) == 1
    with pytest.raises(b2b.B2BError) as e:       # a weight missing
        plan.run(A, [W, W, W, None], D)
    assert e.value.code == 1
    plan.run(A, [W, W, W, W], D)
    torch.cuda.synchronize()
    assert plan.status() == 0 and torch.all(D == 0)


def test_runs_are_deterministic():
    w = wl.small(wl.WORKLOADS["batched_f16"], M=384, batch=2)
    host = wl.make_inputs(w)
    dev = [t.cuda() for t in host]
    plan = b2b.Plan(w.dtype, w.batch, w.M, w.K, *w.N)
    a = plan.run(*dev).clone()
    b = plan.run(*dev).clone()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_argument_errors_on_device():
    plan = b2b.Plan("f16", 1, 128, 64, 64, 64)
    A = torch.zeros((1, 128, 64), dtype=torch.float16, device="cuda")
    B = torch.zeros((1, 64, 64), dtype=torch.float16, device="cuda")
    D = torch.zeros((1, 128, 64), dtype=torch.float16, device="cuda")
    with pytest.raises(b2b.B2BError) as e:       # C missing
        plan.run(A, B, None, None, D)
    assert e.value.code == 1
    with pytest.raises(b2b.B2BError) as e:       # F given to a two-stage plan
        plan.run(A, B, B, B, D)
    assert e.value.code == 1
    with pytest.raises(b2b.B2BError) as e:       # output on top of an input
        plan.run(A, B, B, None, A)
    assert e.value.code == 4
    raw = torch.zeros(128 * 64 + 8, dtype=torch.float16, device="cuda")
    with pytest.raises(b2b.B2BError) as e:       # 2-byte offset: not 16-byte aligned
        plan.run(raw[1:1 + 128 * 64], B, B, None, D)
    assert e.value.code == 3
    with pytest.raises(ValueError):              # A shorter than the plan's rows
        plan.run(A[:, :64].contiguous(), B, B, None, D)
    with pytest.raises(TypeError):               # output of another type
        plan.run(A, B, B, None, D.float())
    torch.cuda.synchronize()
    assert plan.status() == 0                    # nothing was launched


# ------------------------------------------ unfused reference building block --

@pytest.mark.parametrize("dtype,K,N,M", [("f16", 128, 128, 300), ("f16_f32out", 64, 64, 300),
                                         ("bf16", 256, 512, 300), ("tf32", 256, 256, 300), ("f64", 64, 64, 300),
                                         # more tiles than SMs: A through its own ring, several
                                         # tiles per CTA
                                         ("tf32", 256, 256, 20000), ("tf32", 128, 512, 20000),
                                         ("bf16_f32out", 256, 256, 20000), ("f16", 64, 384, 20000)])
def test_single_gemm_plan(dtype, K, N, M):
    w = wl.Workload("gemm", dtype, 2, M, K, (N,), "normal", 0.2, 31)
    host = wl.make_inputs(w)
    plan = b2b.GemmPlan(dtype, w.batch, w.M, K, N)
    dev = [t.cuda() for t in host]
    out = plan.run(*dev)
    torch.cuda.synchronize()
    assert plan.status() == 0
    acc, _, fin = KINDS[dtype]
    if dtype == "tf32":
        fin = oracle.F32
    want = oracle.chain(oracle.widen(host[0]), [oracle.widen(host[1])], acc, oracle.NONE, fin)
    tol = 5e-3 if dtype == "tf32" else TOL[dtype]
    assert rel_err(out.cpu(), want) <= tol


# ------------------------------------------------ full-size, sampled rows --

@pytest.mark.parametrize("name", list(wl.ALL_WORKLOADS))
def test_full_size_sampled_rows(name):
    w = wl.ALL_WORKLOADS[name]
    host = wl.make_inputs(w)
    got = run_gpu(w, host)
    rng = np.random.default_rng(99)
    batches = sorted(set([0, w.batch - 1] + list(rng.integers(0, w.batch, size=min(4, w.batch)))))
    rows = sorted(set([0, 1, 127, 128, w.M - 1] + list(rng.integers(0, w.M, size=60))))
    want = run_oracle(w, host, rows=rows, batches=batches)
    sub = got[batches][:, rows]
    assert rel_err(sub, want) <= TOL[w.dtype]
    assert torch.isfinite(got.float()).all()


# ------------------------------------------------ seeded random shapes --

def _random_cases(n=16, seed=2026, narrow=False, first=100):
    """Cascades with random stage counts, widths, types and sizes (fixed seed);
    narrow: every width at most 256 columns (intermediates then mostly stay
    in tensor memory)."""
    import random
    rng = random.Random(seed)
    cases = []
    for i in range(n):
        dtype = rng.choice(["f16", "bf16", "f16_f32out", "bf16_f32out", "tf32_f16", "tf32_bf16"])
        S = rng.randint(2, 6)
        widths = []
        for s in range(S):
            hi = 256 if narrow else (512 if s < S - 1 else 640)
            widths.append(8 * rng.randint(1, hi // 8))
        K = (4 if dtype.startswith("tf32") else 8) * rng.randint(1, 48)
        if not dtype.startswith("tf32"):
            K = 8 * rng.randint(1, 40)
        batch = rng.randint(1, 3)
        M = rng.randint(1, 1200)
        cases.append(wl.Workload(f"rand{'n' if narrow else ''}{i}_{dtype}_s{S}", dtype, batch, M, K,
                                 tuple(widths), "normal_fanin", 1.0, first + i))
    return cases


@pytest.mark.parametrize("w", _random_cases() + _random_cases(8, 2027, narrow=True, first=120),
                         ids=lambda w: w.name)
def test_random_cascades(w):
    host = wl.make_inputs(w)
    dev = [t.cuda() for t in host]
    plan = b2b.ChainPlan(w.dtype, w.batch, w.M, w.K, w.N)
    out = plan.run(dev[0], dev[1:])
    torch.cuda.synchronize()
    assert plan.status() == 0
    want = run_oracle(w, host)
    assert rel_err(out.cpu(), want) <= TOL[w.dtype], (w.N, w.K, w.M)


def _random_two_stage(n=16, seed=7):
    """Two-stage chains of the one-CTA kernels (16-bit with N1 <= 256, tf32,
    fp64) and single GEMMs, random sizes (fixed seed)."""
    import random
    rng = random.Random(seed)
    cases = []
    for i in range(n):
        dtype = rng.choice(["f16", "bf16", "f16_f32out", "bf16_f32out", "tf32", "f64"])
        if dtype == "f64":
            N = (rng.choice([16, 32, 64]), rng.choice([16, 32, 64]))
            K = 4 * rng.randint(1, 32)
        elif dtype == "tf32":
            N = (4 * rng.randint(1, 64), 4 * rng.randint(1, 160))
            K = 4 * rng.randint(1, 96)
        else:
            N = (8 * rng.randint(1, 32), 8 * rng.randint(1, 80))
            K = 8 * rng.randint(1, 64)
        batch = rng.randint(1, 40)
        M = rng.randint(1, 3000 // batch + 1)
        dist = "uniform" if dtype == "f64" else ("normal" if dtype == "tf32" else "normal_fanin")
        scale = 1.0 / 16 if dtype == "tf32" else 1.0
        cases.append(wl.Workload(f"rand2s{i}_{dtype}", dtype, batch, M, K, N, dist, scale, 200 + i))
    return cases


@pytest.mark.parametrize("w", _random_two_stage(), ids=lambda w: w.name)
def test_random_two_stage(w):
    host = wl.make_inputs(w)
    got = run_gpu(w, host)
    want = run_oracle(w, host)
    assert rel_err(got, want) <= TOL[w.dtype], (w.N, w.K, w.M, w.batch)


def test_one_plan_on_two_streams_at_once():
    """Runs of one plan may overlap on different streams (the plan is not
    modified by a run): both results must be the single-stream ones."""
    cases = [wl.small(wl.WORKLOADS["batched_f16"], M=1000, batch=40),
             wl.small(wl.WORKLOADS["three_stage_bf16"], M=3000)]
    for w in cases:
        plan = b2b.ChainPlan(w.dtype, w.batch, w.M, w.K, w.N)
        ins = [[t.cuda() for t in wl.make_inputs(w, seed=s)] for s in (1, 2)]
        want = [plan.run(x[0], x[1:]).clone() for x in ins]
        torch.cuda.synchronize()
        streams = [torch.cuda.Stream(), torch.cuda.Stream()]
        outs = [plan.empty_out(), plan.empty_out()]
        for rep in range(5):
            for x, o, s in zip(ins, outs, streams):
                plan.run(x[0], x[1:], o, stream=s)
        torch.cuda.synchronize()
        assert plan.status() == 0
        for o, ref in zip(outs, want):
            assert torch.equal(o.view(torch.int16), ref.view(torch.int16))
