"""Pins of the CPU oracle against facts outside itself (no GPU needed).

Each test fixes the oracle to something it does not compute itself:
independent conversions (numpy float16, torch bfloat16, numpy float32, the
tf32 bit definition), closed forms (identity, permutation, diagonal), exact
integer arithmetic (associativity, brute force with Python integers) and
numpy's fp64 matmul.  A dropped term, a wrong index, a transposed operand or
a misplaced rounding makes at least one of them fail: the last test plants
each such mistake in a compiled copy of the oracle and checks that a pin
catches it.
"""
import itertools
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import BF16, F16, F32, NONE, TF32, TF32_RNE

RNG = np.random.default_rng(12345)


# --------------------------------------------------------------- rounding --

def test_f16_every_pattern_round_trips():
    bits = np.arange(1 << 16, dtype=np.uint16)
    vals = bits.view(np.float16).astype(np.float64)
    got = oracle.round_to(F16, vals)
    finite = np.isfinite(vals)
    assert np.array_equal(got[finite], vals[finite])
    assert np.all(np.isnan(got[np.isnan(vals)]))
    assert np.array_equal(got[np.isinf(vals)], vals[np.isinf(vals)])


def test_bf16_every_pattern_round_trips():
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    vals = bits.view(np.float32).astype(np.float64)
    got = oracle.round_to(BF16, vals)
    finite = np.isfinite(vals)
    assert np.array_equal(got[finite], vals[finite])
    assert np.all(np.isnan(got[np.isnan(vals)]))


def _fp32_samples(n):
    """Random fp32 values over the whole range, plus ties and edges."""
    bits = RNG.integers(0, 1 << 32, size=n, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    edges = np.array([0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 65536.0, 1e-8, 6e-8,
                      5.960464477539063e-08, 2.9802322387695312e-08, 6.103515625e-05,
                      3.4e38, -3.4e38, 1.17549435e-38, 1e-45, 2049.0, 2051.0, 4097.0],
                     dtype=np.float32)
    # exact midpoints between neighbouring fp16 values (ties)
    h = np.arange(0x0001, 0x7bff, 97, dtype=np.uint16).view(np.float16).astype(np.float64)
    h2 = (np.arange(0x0001, 0x7bff, 97, dtype=np.uint16) + 1).view(np.float16).astype(np.float64)
    ties = ((h + h2) / 2).astype(np.float32)
    return np.concatenate([x, edges, ties, -ties])


def test_f16_matches_numpy_cast():
    x = _fp32_samples(200_000)
    want = x.astype(np.float16).astype(np.float64)
    got = oracle.round_to(F16, x.astype(np.float64))
    assert np.array_equal(got, want)


def test_bf16_matches_torch_cast():
    x = _fp32_samples(200_000)
    # bf16 ties: the fp32 values exactly halfway between two bf16 values
    b = (RNG.integers(0, 0x7f7f, size=5000, dtype=np.uint32) << 16) | 0x8000
    x = np.concatenate([x, b.view(np.float32), -b.view(np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_to(BF16, x.astype(np.float64))
    assert np.array_equal(got, want)


def test_f32_matches_numpy_cast():
    x = np.concatenate([RNG.normal(size=100_000) * 10.0 ** RNG.integers(-40, 39, size=100_000),
                        np.array([1 + 2.0 ** -24, 1 + 3 * 2.0 ** -24, 3.4028235677973366e38,
                                  3.4028235e38 * 1.0000001, 1e-46, 7e-46])])
    with np.errstate(over="ignore"):
        want = x.astype(np.float32).astype(np.float64)
    got = oracle.round_to(F32, x)
    assert np.array_equal(got, want)


def _tf32_rna_bits(x32: np.ndarray) -> np.ndarray:
    """Round half away on the bit pattern: add half a tf32 ulp, clear 13 bits."""
    b = x32.view(np.uint32).astype(np.uint64)
    r = ((b + 0x1000) & 0xFFFFE000).astype(np.uint32)
    return r.view(np.float32).astype(np.float64)


def test_tf32_round_half_away_matches_bit_definition():
    x = RNG.normal(size=200_000).astype(np.float32) * np.float32(100.0)
    ties = (RNG.integers(0x00800000, 0x7f000000, size=20_000, dtype=np.uint32) & 0xFFFFE000) | 0x1000
    x = np.concatenate([x, ties.view(np.float32), -ties.view(np.float32)])
    got = oracle.round_to(TF32, x.astype(np.float64))
    assert np.array_equal(got, _tf32_rna_bits(x))


def test_tf32_ties_away_vs_even():
    one = 1.0
    tie = one + 2.0 ** -11                     # halfway between 1 and 1 + 2^-10
    assert oracle.round_to(TF32, [tie])[0] == one + 2.0 ** -10
    assert oracle.round_to(TF32, [-tie])[0] == -(one + 2.0 ** -10)
    assert oracle.round_to(TF32_RNE, [tie])[0] == one
    assert oracle.round_to(TF32, [tie - 2.0 ** -23])[0] == one


# -------------------------------------------------------------- the chain --

CHAIN_KINDS = {
    "f16_f32out": (F32, F16, F32),
    "f16": (F32, F16, F16),
    "bf16": (F32, BF16, BF16),
    "tf32": (F32, TF32, F32),
    "f64": (NONE, NONE, NONE),
}


@pytest.mark.parametrize("kind", list(CHAIN_KINDS))
def test_identity(kind):
    acc, mid, out = CHAIN_KINDS[kind]
    A = oracle.round_to(mid, RNG.uniform(-2, 2, size=(2, 5, 8)))
    A = oracle.round_to(out, A)
    eye = np.eye(8)
    got = oracle.chain(A, [eye, eye], acc, mid, out)
    assert np.array_equal(got, A)
    got3 = oracle.chain(A, [eye, eye, eye], acc, mid, out)
    assert np.array_equal(got3, A)


@pytest.mark.parametrize("kind", list(CHAIN_KINDS))
def test_permutation(kind):
    acc, mid, out = CHAIN_KINDS[kind]
    A = oracle.round_to(out, oracle.round_to(mid, RNG.uniform(-3, 3, size=(1, 7, 6))))
    p1 = RNG.permutation(6)
    p2 = RNG.permutation(6)
    P1 = np.eye(6)[p1]          # (A @ P1)[:, j] = A[:, argwhere p1 == j]
    P2 = np.eye(6)[p2]
    got = oracle.chain(A, [P1, P2], acc, mid, out)
    want = A[..., np.argsort(p1)][..., np.argsort(p2)]
    assert np.array_equal(got, want)


@pytest.mark.parametrize("kind", list(CHAIN_KINDS))
def test_diagonal_closed_form(kind):
    acc, mid, out = CHAIN_KINDS[kind]
    A = oracle.round_to(mid, RNG.uniform(-1, 1, size=(1, 9, 4)))
    b = oracle.round_to(mid, RNG.uniform(-1, 1, size=4))
    c = oracle.round_to(mid, RNG.uniform(-1, 1, size=4))
    got = oracle.chain(A, [np.diag(b), np.diag(c)], acc, mid, out)
    p = oracle.round_to(mid, oracle.round_to(acc, A * b))          # one product per entry
    want = oracle.round_to(out, oracle.round_to(acc, p * c))
    assert np.array_equal(got, want)


def test_intermediate_is_rounded_to_operand_type():
    # P = (1 + 2^-10)^2 = 1 + 2^-9 + 2^-20 is exact in fp32 but not in fp16
    a = np.array([[[1 + 2.0 ** -10]]])
    got = oracle.chain(a, [a[0], np.array([[1.0]])], F32, F16, F32)
    assert got[0, 0, 0] == 1 + 2.0 ** -9
    got_wide = oracle.chain(a, [a[0], np.array([[1.0]])], F32, NONE, F32)
    assert got_wide[0, 0, 0] == 1 + 2.0 ** -9 + 2.0 ** -20


@pytest.mark.parametrize("stages", [2, 3])
def test_associativity_exact_integers(stages):
    K, Ns = 24, [16, 8, 12][:stages]
    A = RNG.integers(-2, 3, size=(3, 11, K))
    Ws = []
    kin = K
    for n in Ns:
        Ws.append(RNG.integers(-2, 3, size=(3, kin, n)))
        kin = n
    # right-to-left product with exact int64 arithmetic: A.(W1.(W2...))
    R = Ws[-1]
    for W in reversed(Ws[:-1]):
        R = np.matmul(W, R)
    want = np.matmul(A, R).astype(np.float64)
    assert np.abs(want).max() < 2 ** 24
    for kind in ("f16_f32out", "tf32", "f64"):
        acc, mid, out = CHAIN_KINDS[kind]
        got = oracle.chain(A.astype(np.float64), [w.astype(np.float64) for w in Ws], acc, mid, out)
        assert np.array_equal(got, want), kind


def _brute(A, Ws):
    """Triple products with Python integers / Fractions, no numpy."""
    batch, M, K = len(A), len(A[0]), len(A[0][0])
    out = []
    for b in range(batch):
        rows = []
        for m in range(M):
            cur = [Fraction(v) for v in A[b][m]]
            for W in Ws:
                n_out = len(W[b][0])
                cur = [sum(cur[k] * Fraction(W[b][k][n]) for k in range(len(cur))) for n in range(n_out)]
            rows.append(cur)
        out.append(rows)
    return out


def test_brute_force_tiny_shapes():
    vals = (-1, 0, 1)
    count = 0
    for M, K, N1, N2 in itertools.product((1, 2, 3), (1, 2, 3), (1, 2, 3), (1, 2)):
        for trial in range(3):
            A = RNG.choice(vals, size=(1, M, K))
            B = RNG.choice(vals, size=(1, K, N1))
            C = RNG.choice(vals, size=(1, N1, N2))
            want = np.array(_brute(A.tolist(), [B.tolist(), C.tolist()]), dtype=np.float64)
            got = oracle.chain(A.astype(float), [B.astype(float), C.astype(float)], NONE, NONE, NONE)
            assert np.array_equal(got, want)
            got16 = oracle.chain(A.astype(float), [B.astype(float), C.astype(float)], F32, F16, F16)
            assert np.array_equal(got16, want)
            count += 1
    # every 1x1x1 chain over {-1,0,1}^3 exhaustively
    for a, b, c in itertools.product(vals, repeat=3):
        got = oracle.chain(np.array([[[a]]], float), [np.array([[b]], float), np.array([[c]], float)],
                           F32, BF16, BF16)
        assert got[0, 0, 0] == a * b * c
    assert count == 162


def test_fp64_matches_numpy_matmul():
    A = RNG.normal(size=(2, 33, 20))
    B = RNG.normal(size=(2, 20, 17))
    C = RNG.normal(size=(2, 17, 9))
    F = RNG.normal(size=(2, 9, 5))
    got = oracle.chain(A, [B, C, F], NONE, NONE, NONE)
    want = A @ B @ C @ F
    assert np.max(np.abs(got - want)) <= 1e-13 * np.max(np.abs(want))


def test_fp16_chain_matches_stepwise_numpy():
    # a different route to the same definition: numpy fp64 matmul, then casts
    A = RNG.normal(size=(2, 40, 32)).astype(np.float16).astype(np.float64)
    B = RNG.normal(size=(2, 32, 24)).astype(np.float16).astype(np.float64)
    C = RNG.normal(size=(2, 24, 16)).astype(np.float16).astype(np.float64)
    P = (A @ B).astype(np.float32).astype(np.float16).astype(np.float64)
    want = (P @ C).astype(np.float32).astype(np.float16).astype(np.float64)
    got = oracle.chain(A, [B, C], F32, F16, F16)
    # numpy's pairwise sums may differ in the last fp64 bit; allow a final-ulp flip
    diff = np.abs(got - want)
    ulp = np.spacing(np.abs(want).astype(np.float16)).astype(np.float64)
    assert np.all(diff <= ulp)
    assert np.mean(diff == 0) > 0.999


def test_threads_do_not_change_results():
    A = RNG.normal(size=(3, 50, 16))
    B = RNG.normal(size=(3, 16, 8))
    C = RNG.normal(size=(3, 8, 8))
    one = oracle.chain(A, [B, C], F32, BF16, BF16, n_threads=1)
    many = oracle.chain(A, [B, C], F32, BF16, BF16, n_threads=4)
    assert np.array_equal(one, many)


def test_rejects_mismatched_shapes():
    with pytest.raises(ValueError):
        oracle.chain(np.zeros((1, 2, 3)), [np.zeros((1, 4, 2))], F32, F16, F16)


# ------------------------------------------ rounding after later GEMMs --
# Every intermediate is the operand of the next GEMM, so it is rounded to the
# operand type after every GEMM but the last, not only after the first one
# (three or more cascaded operators: patent Detailed description para. 41;
# the operand data types: para. 28).  The pins below fix that placement for
# the second and later hand-overs, and for the output of chains of three and
# four GEMMs.

THREE_STAGE_KINDS = ["f16_f32out", "f16", "bf16", "tf32"]


@pytest.mark.parametrize("kind", THREE_STAGE_KINDS)
def test_three_stage_diagonal_closed_form(kind):
    # with diagonal weights every entry is one product per stage:
    # E[m][n] = r_out(r32(r_mid(r32(r_mid(r32(A b)) c)) f))
    acc, mid, out = CHAIN_KINDS[kind]
    A = oracle.round_to(mid, RNG.uniform(-1, 1, size=(2, 11, 6)))
    b, c, f = (oracle.round_to(mid, RNG.uniform(-1, 1, size=6)) for _ in range(3))
    got = oracle.chain(A, [np.diag(b), np.diag(c), np.diag(f)], acc, mid, out)
    p = oracle.round_to(mid, oracle.round_to(acc, A * b))
    q = oracle.round_to(mid, oracle.round_to(acc, p * c))
    want = oracle.round_to(out, oracle.round_to(acc, q * f))
    assert np.array_equal(got, want)
    # the pin has power: leaving the second intermediate unrounded changes
    # the result
    q_raw = oracle.round_to(acc, p * c)
    assert not np.array_equal(oracle.round_to(out, oracle.round_to(acc, q_raw * f)), want)


def _eighths(shape):
    """Entries k/8 with integer |k| <= 8: every product and sum below is exact in fp64."""
    return RNG.integers(-8, 9, size=shape).astype(np.float64) / 8.0


def _cast_f16(x):
    return x.astype(np.float32).astype(np.float16).astype(np.float64)


def _cast_bf16(x):
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def _cast_tf32(x):
    return _tf32_rna_bits(x.astype(np.float32))


@pytest.mark.parametrize("kind,cast", [("f16", _cast_f16), ("bf16", _cast_bf16), ("tf32", _cast_tf32)])
def test_three_and_four_stage_chains_match_stepwise_casts(kind, cast):
    # another route to the definition: numpy fp64 matmul (exact here: the
    # operands are k/8, or operand-type values of at most 11 significant
    # bits, and the sums stay far inside 53 bits), then the library casts of
    # numpy / torch / the tf32 bit rule
    acc, mid, out = CHAIN_KINDS[kind]
    A = _eighths((2, 20, 24))
    Ws = [_eighths((2, 24, 16)), _eighths((2, 16, 12)), _eighths((2, 12, 16)), _eighths((2, 16, 8))]
    f32 = lambda x: x.astype(np.float32).astype(np.float64)  # noqa: E731
    out_cast = cast if out == mid else f32
    for stages in (3, 4):
        x = A
        rounded_mid = 0
        for s in range(stages):
            y = f32(x @ Ws[s])
            if s < stages - 1:
                x = cast(y)
                rounded_mid += int(np.sum(x != y))
            else:
                x = out_cast(y)
        got = oracle.chain(A, Ws[:stages], acc, mid, out)
        assert np.array_equal(got, x), (kind, stages)
        # the intermediates are not all representable before rounding: the
        # rounding placement decides the result
        assert rounded_mid > 0


@pytest.mark.parametrize("stage", [0, 1, 2])
def test_accumulator_is_rounded_to_fp32_before_the_operand_type(stage):
    # Three GEMMs of 3x3 weights, identities except GEMM `stage`, whose ones
    # put the sum of the row in every column.
    eye, ones = np.eye(3), np.ones((3, 3))
    Ws = [eye, eye, eye]
    Ws[stage] = ones
    # bf16: a sum above a tie by less than half an fp32 ulp.  Rounded to fp32
    # first it lands on the tie and goes to even (1.0); rounded directly it
    # would go up (1 + 2^-7).  After the last GEMM the output rounding does
    # the same.
    got = oracle.chain(np.array([[[1.0, 2.0 ** -8, 2.0 ** -30]]]), Ws, F32, BF16, BF16)
    assert np.array_equal(got[0, 0], [1.0, 1.0, 1.0])
    # tf32 (ties away from zero): a sum below a tie by less than half an fp32
    # ulp lands on the tie in fp32 and then goes away (1 + 2^-10); directly it
    # would go down (1.0).  After the last GEMM only the fp32 rounding is left.
    got = oracle.chain(np.array([[[1.0, 2.0 ** -11, -(2.0 ** -30)]]]), Ws, F32, TF32, F32)
    want = 1.0 + (2.0 ** -11 if stage == 2 else 2.0 ** -10)
    assert np.array_equal(got[0, 0], [want] * 3)


# ------------------------------------------------------ planted mistakes --
# Each mutant is oracle.c with one plausible mistake planted in a copy (the
# oracle itself is untouched), compiled with the host compiler and put in
# place of the real library; at least one of the pins above must then fail.

MUTANTS = {
    "later intermediates left unrounded": (
        "cur[n] = oracle_round1(last ? out_kind : interm_kind, nxt[n]);",
        "cur[n] = oracle_round1(last ? out_kind : (s == 0 ? interm_kind : ORC_NONE), nxt[n]);"),
    "later accumulators not rounded to fp32": (
        "nxt[n] = oracle_round1(acc_kind, acc);", "nxt[n] = oracle_round1(s == 0 ? acc_kind : ORC_NONE, acc);"),
    "accumulators never rounded to fp32": ("nxt[n] = oracle_round1(acc_kind, acc);", "nxt[n] = acc;"),
    "output rounded to the intermediate type": ("last ? out_kind : interm_kind", "interm_kind"),
    "output left unrounded": ("last ? out_kind : interm_kind", "last ? ORC_NONE : interm_kind"),
    "first term of every sum dropped": ("for (int64_t k = 0; k < kin; ++k)", "for (int64_t k = 1; k < kin; ++k)"),
    "weight read transposed": ("w[k * n_out + n]", "w[n * kin + k]"),
    "batch 0's weights for every batch": ("W[s] + b * kin * n_out", "W[s]"),
    "tf32 ties to even": ("round_binary(x, 10, -126, 127, 1)", "round_binary(x, 10, -126, 127, 0)"),
    "fp16 ties away from zero": ("round_binary(x, 10, -14, 15, 0)", "round_binary(x, 10, -14, 15, 1)"),
    "fp16 subnormal bound off by one": ("round_binary(x, 10, -14, 15, 0)", "round_binary(x, 10, -15, 15, 0)"),
    "bf16 with the fp16 exponent range": ("round_binary(x, 7, -126, 127, 0)", "round_binary(x, 7, -14, 15, 0)"),
    "overflow kept finite": ("r = INFINITY;", "r = maxv;"),
}


def _pins():
    """Every pin of this module as a zero-argument call."""
    calls = [test_f16_every_pattern_round_trips, test_bf16_every_pattern_round_trips, test_f16_matches_numpy_cast,
             test_bf16_matches_torch_cast, test_f32_matches_numpy_cast,
             test_tf32_round_half_away_matches_bit_definition, test_tf32_ties_away_vs_even,
             test_intermediate_is_rounded_to_operand_type, test_brute_force_tiny_shapes,
             test_fp64_matches_numpy_matmul, test_fp16_chain_matches_stepwise_numpy]
    for kind in CHAIN_KINDS:
        calls += [lambda k=kind: test_identity(k), lambda k=kind: test_permutation(k),
                  lambda k=kind: test_diagonal_closed_form(k)]
    calls += [lambda n=n: test_associativity_exact_integers(n) for n in (2, 3)]
    calls += [lambda k=k: test_three_stage_diagonal_closed_form(k) for k in THREE_STAGE_KINDS]
    calls += [lambda k=k, c=c: test_three_and_four_stage_chains_match_stepwise_casts(k, c)
              for k, c in (("f16", _cast_f16), ("bf16", _cast_bf16), ("tf32", _cast_tf32))]
    calls += [lambda s=s: test_accumulator_is_rounded_to_fp32_before_the_operand_type(s) for s in (0, 1, 2)]
    return calls


def _load_mutant(path):
    import ctypes
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    lib.oracle_round1.restype = ctypes.c_double
    lib.oracle_round1.argtypes = [ctypes.c_int, ctypes.c_double]
    lib.oracle_round.restype = None
    lib.oracle_round.argtypes = [ctypes.c_int, dp, dp, ctypes.c_int64]
    lib.oracle_chain.restype = ctypes.c_int
    lib.oracle_chain.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                 ctypes.POINTER(ctypes.c_int64), dp, ctypes.POINTER(dp), ctypes.c_int,
                                 ctypes.c_int, ctypes.c_int, dp, ctypes.c_int]
    lib.oracle_max_threads.restype = ctypes.c_int
    lib.oracle_max_threads.argtypes = []
    return lib


@pytest.mark.parametrize("name", list(MUTANTS))
def test_a_planted_mistake_fails_a_pin(name, tmp_path, monkeypatch):
    import os
    import subprocess
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"the mutation site {old!r} is not unique in oracle.c"
    c_file = tmp_path / "mutant.c"
    c_file.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-fno-fast-math",
                    "-ffp-contract=off", str(c_file), "-o", str(so), "-lm"], check=True)
    monkeypatch.setattr(oracle, "_lib", _load_mutant(str(so)))
    caught = None
    for pin in _pins():
        try:
            pin()
        except AssertionError:
            caught = pin
            break
    assert caught is not None, f"no pin fails when {name}"
