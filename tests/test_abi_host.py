"""Host-side checks of the C ABI (no GPU needed).

The library must load on a machine without a GPU, export every function the
header declares, reject bad arguments before touching a device, and its
coordination-matrix generator must satisfy the patent's facts about the
coordination matrix and realise the rearrangement relation of the oracle.
"""
import ctypes
import os
import re

import pytest

import fusion_b2b_gemm_gb300 as b2b
from oracle import relation as rel

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


def _declared_functions():
    with open(os.path.join(ROOT, "include", "b2b.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(b2b_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    names = _declared_functions()
    assert len(names) >= 10
    lib = ctypes.CDLL(b2b.library_path())
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings():
    for code in range(8):
        s = b2b.b2b_status_string(code).decode()
        assert s and s != "unknown status"
    assert b2b.b2b_status_string(99).decode() == "unknown status"


def _create(dtype, batch, M, K, N1, N2, N3=0):
    h = ctypes.c_void_p()
    code = b2b.b2b_plan_create(ctypes.byref(h), dtype, batch, M, K, N1, N2, N3)
    return code, h


@pytest.mark.parametrize("args,code", [
    ((1, 1, 64, 64, 64, 64), 0),          # valid: fails only on the device check below
    ((1, -1, 64, 64, 64, 64), 1),         # negative batch
    ((1, 1, 64, 0, 64, 64), 1),           # K = 0
    ((1, 1, 64, 64, 0, 64), 1),           # N1 = 0
    ((1, 1, 64, 60, 64, 64), 2),          # K not a multiple of 8 for fp16
    ((1, 1, 64, 64, 520, 64), 2),         # N1 > 512
    ((1, 1, 64, 64, 264, 64), 0),         # 256 < N1 <= 512: the paired kernel
    ((3, 1, 64, 64, 264, 64), 2),         # tf32 N1 > 256
    ((3, 1, 64, 64, 64, 64, 64), 2),      # tf32 three-stage
    ((4, 1, 64, 64, 48, 64), 2),          # fp64 N1 not in {16, 32, 64}
    ((9, 1, 64, 64, 64, 64), 1),          # unknown dtype
])
def test_plan_create_validates_before_device(args, code):
    got, h = _create(*args)
    if code == 0:
        # No GPU here: a valid request is refused only by the device check.
        import torch
        if torch.cuda.is_available():
            pytest.skip("a GPU is present")
        assert got in (5, 6)
    else:
        assert got == code
    assert not h.value


def _create_chain(dtype, batch, M, K, widths, n=None):
    h = ctypes.c_void_p()
    arr = (ctypes.c_int64 * max(1, len(widths)))(*widths)
    code = b2b.b2b_chain_plan_create(ctypes.byref(h), dtype, batch, M, K,
                                     len(widths) if n is None else n, arr)
    return code, h


@pytest.mark.parametrize("args,code", [
    ((1, 1, 64, 64, (64, 64, 64, 64, 64)), 0),       # five stages
    ((2, 1, 64, 64, (512,) * 7 + (4096,)), 0),       # eight stages at the width limits
    ((1, 1, 64, 64, (64,) * 9), 1),                  # more than eight stages
    ((1, 1, 64, 64, ()), 1),                         # no stage
    ((1, 1, 64, 64, (64, 64, 520, 64)), 2),          # an intermediate wider than 512
    ((1, 1, 64, 64, (64, 64, 64, 4104)), 2),         # last width above 4096
    ((1, 1, 64, 64, (64, 60, 64, 64)), 2),           # width not a multiple of 8
    ((3, 1, 64, 64, (64, 64, 64)), 2),               # tf32 three stages
    ((4, 1, 64, 64, (16, 16, 16)), 2),               # fp64 three stages
    ((6, 1, 64, 64, (64, 64, 64)), 0),               # tf32 first GEMM, fp16 after it
    ((7, 2, 64, 96, (512, 64)), 0),                  # tf32 then bf16, wide intermediate
    ((6, 1, 64, 64, (64,)), 2),                      # a mixed cascade needs two stages
    ((7, 1, 64, 66, (64, 64)), 2),                   # fp32 rows not 16-byte aligned
    ((6, 1, 64, 64, (68, 64)), 2),                   # 16-bit width not a multiple of 8
    ((8, 1, 64, 64, (64, 64)), 1),                   # unknown dtype
])
def test_chain_plan_create_validates_before_device(args, code):
    got, h = _create_chain(*args)
    if code == 0:
        import torch
        if torch.cuda.is_available():
            pytest.skip("a GPU is present")
        assert got in (5, 6)
    else:
        assert got == code
    assert not h.value


def test_null_arguments():
    assert b2b.b2b_run(None, None, None, None, None, None, None) == 1
    assert b2b.b2b_chain_run(None, None, None, None, None) == 1
    assert b2b.b2b_chain_plan_create(None, 1, 1, 64, 64, 2, None) == 1
    h = ctypes.c_void_p()
    assert b2b.b2b_chain_plan_create(ctypes.byref(h), 1, 1, 64, 64, 2, None) == 1
    assert b2b.b2b_plan_destroy(None) == 0
    assert b2b.b2b_plan_device_status(None, None) == 1
    assert b2b.b2b_plan_info(None, None, None, None, None, None, None, None) == 1
    assert b2b.b2b_plan_create(None, 1, 1, 1, 64, 64, 64, 0) == 1


# ------------------------------------------------- coordination matrix --

def _golden_matrix():
    with open(os.path.join(GOLDEN, "coordination_matrix.txt"), encoding="utf-8") as f:
        text = f.read()
    row0 = [tuple(int(x) for x in m) for m in re.findall(r"\((\d+),(\d+),(\d+)\)",
                                                         re.search(r"^row0:(.*)$", text, re.M).group(1))]
    f0 = [int(x) for x in re.search(r"^f0:(.*)$", text, re.M).group(1).split()]
    return row0, f0


def _sources(relation, n, m):
    st = [[relation[(i, r)][0] for r in range(m)] for i in range(n)]
    sr = [[relation[(i, r)][1] for r in range(m)] for i in range(n)]
    return st, sr


def test_tf32_example_coordination_matrix():
    row0, f0 = _golden_matrix()
    r = rel.relation(rel.m16n8k8_tf32_c, rel.m16n8k8_tf32_a, lanes=4, regs=4)
    st, sr = _sources(r, 4, 4)
    H = b2b.coordination_matrix(st, sr)
    assert H[0] == row0
    assert [H[i][0][0] for i in range(4)] == f0
    # f0 is the patent's bit expression
    assert f0 == [((i & 2) >> 1) + ((i & 1) << 1) for i in range(4)]
    cols = [[H[i][j] for i in range(4)] for j in range(4)]
    assert rel.is_conflict_free(cols)
    vals = [[(lane, e) for e in range(4)] for lane in range(4)]
    out = rel.apply_rounds(vals, cols)
    for i in range(4):
        assert out[i] == [r[(i, k)] for k in range(4)]


def test_f64_relation_schedule_realises_the_oracle_relation():
    prod = rel.tiled(rel.m8n8k4_f64_c, 2, 1, 8)
    cons = rel.tiled(rel.m8n8k4_f64_a, 1, 2, 4)
    r = rel.relation(prod, cons, lanes=4, regs=2)
    st, sr = _sources(r, 4, 2)
    H = b2b.coordination_matrix(st, sr)
    cols = [[H[i][j] for i in range(4)] for j in range(2)]
    assert rel.is_conflict_free(cols)
    vals = [[(lane, e) for e in range(2)] for lane in range(4)]
    out = rel.apply_rounds(vals, cols)
    for i in range(4):
        assert out[i] == [r[(i, k)] for k in range(2)]
    # round 0 of the fp64 schedule is the patent's f0 as well
    assert [H[i][0][0] for i in range(4)] == [((i & 2) >> 1) + ((i & 1) << 1) for i in range(4)]


def test_generator_falls_back_when_greedy_gets_stuck():
    # A relation on which the in-order greedy choice blocks a later receiver:
    # every receiver's first source is thread 0 or 1, so the greedy order
    # uses both in round 0 for receivers 0 and 1 and strands receiver 2.
    n, m = 3, 3
    st = [[0, 1, 2], [1, 0, 2], [0, 1, 2]]
    sr = [[0, 0, 0], [1, 1, 1], [2, 2, 2]]
    H = b2b.coordination_matrix(st, sr)
    cols = [[H[i][j] for i in range(n)] for j in range(m)]
    assert rel.is_conflict_free(cols)
    vals = [[(lane, e) for e in range(m)] for lane in range(n)]
    out = rel.apply_rounds(vals, cols)
    for i in range(n):
        assert out[i] == [(st[i][k], sr[i][k]) for k in range(m)]


@pytest.mark.parametrize("seed", range(20))
def test_generator_on_random_permutations(seed):
    import random
    rnd = random.Random(seed)
    n, m = rnd.randint(2, 8), rnd.randint(1, 6)
    srcs = [(p, q) for p in range(n) for q in range(m)]
    rnd.shuffle(srcs)
    st = [[srcs[i * m + r][0] for r in range(m)] for i in range(n)]
    sr = [[srcs[i * m + r][1] for r in range(m)] for i in range(n)]
    H = b2b.coordination_matrix(st, sr)
    cols = [[H[i][j] for i in range(n)] for j in range(m)]
    assert rel.is_conflict_free(cols)
    out = rel.apply_rounds([[(l, e) for e in range(m)] for l in range(n)], cols)
    for i in range(n):
        assert out[i] == [(st[i][k], sr[i][k]) for k in range(m)]


def test_generator_rejects_a_source_used_twice():
    with pytest.raises(b2b.B2BError) as e:
        b2b.coordination_matrix([[0, 0], [1, 1]], [[0, 0], [0, 1]])
    assert e.value.code == 1


# ------------------------------------------- operand checks of the binding --

def test_operand_checks_refuse_short_or_mistyped_tensors():
    """The kernels read and write the plan's full sizes, so the binding refuses
    a tensor with fewer elements or of another type before any launch."""
    import torch
    f16, f32 = torch.float16, torch.float32
    N = (64, 32)
    A = torch.zeros(2, 100, 48, dtype=f16)
    W = [torch.zeros(2, 48, 64, dtype=f16), torch.zeros(2, 64, 32, dtype=f16)]
    D = torch.zeros(2, 100, 32, dtype=f16)
    b2b.check_operands("f16", 2, 100, 48, N, A, W, D)           # exact sizes
    b2b.check_operands("f16", 2, 100, 48, N, A, W, torch.zeros(7000, dtype=f16))  # larger is fine
    with pytest.raises(ValueError, match="A"):
        b2b.check_operands("f16", 2, 100, 48, N, A[:, :99], W, D)
    with pytest.raises(ValueError, match=r"W\[1\]"):
        b2b.check_operands("f16", 2, 100, 48, N, A, [W[0], W[1][:1]], D)
    with pytest.raises(ValueError, match="D"):
        b2b.check_operands("f16", 2, 100, 48, N, A, W, D[:1])
    with pytest.raises(TypeError, match="D"):
        b2b.check_operands("f16", 2, 100, 48, N, A, W, D.float())   # f16 out expected
    with pytest.raises(TypeError, match="A"):
        b2b.check_operands("f16_f32out", 2, 100, 48, N, A.bfloat16(), W, D.float())
    # a missing operand is left to the C ABI's argument error
    b2b.check_operands("f16", 2, 100, 48, N, A, [W[0], None], D)
    # a plan without rows reads and writes nothing
    b2b.check_operands("f16", 2, 0, 48, N, A[:, :0], [w[:0] for w in W], D[:, :0])


def test_operand_checks_follow_the_mixed_types():
    """Mixed cascades: fp32 A and first weight, 16-bit later weights, fp32 out."""
    import torch
    N = (64, 32, 16)
    A = torch.zeros(1, 10, 8, dtype=torch.float32)
    W = [torch.zeros(1, 8, 64, dtype=torch.float32), torch.zeros(1, 64, 32, dtype=torch.bfloat16),
         torch.zeros(1, 32, 16, dtype=torch.bfloat16)]
    D = torch.zeros(1, 10, 16, dtype=torch.float32)
    b2b.check_operands("tf32_bf16", 1, 10, 8, N, A, W, D)
    with pytest.raises(TypeError, match=r"W\[1\]"):
        b2b.check_operands("tf32_f16", 1, 10, 8, N, A, W, D)      # fp16 later weights expected
    with pytest.raises(TypeError, match=r"W\[0\]"):
        b2b.check_operands("tf32_bf16", 1, 10, 8, N, A, [W[0].bfloat16()] + W[1:], D)


def test_operand_checks_refuse_tensors_on_another_gpu():
    """A plan runs on the GPU it was created on; a tensor of another GPU would
    be read through a peer address, so the binding refuses it."""
    import torch

    class OnGpu:
        """Stands for a CUDA tensor on device `index` (no GPU here)."""

        def __init__(self, t, index):
            self.t, self.is_cuda, self.dtype = t, True, t.dtype
            self.device = torch.device("cuda", index)

        def numel(self):
            return self.t.numel()

    f16 = torch.float16
    N = (64, 32)
    A = OnGpu(torch.zeros(2, 100, 48, dtype=f16), 1)
    W = [OnGpu(torch.zeros(2, 48, 64, dtype=f16), 1), OnGpu(torch.zeros(2, 64, 32, dtype=f16), 1)]
    D = OnGpu(torch.zeros(2, 100, 32, dtype=f16), 1)
    b2b.check_operands("f16", 2, 100, 48, N, A, W, D, device=1)
    for bad in ("A", "W[1]", "D"):
        args = {"A": A, "W[0]": W[0], "W[1]": W[1], "D": D}
        args[bad] = OnGpu(args[bad].t, 0)
        with pytest.raises(ValueError, match=bad.replace("[", r"\[").replace("]", r"\]")):
            b2b.check_operands("f16", 2, 100, 48, N, args["A"], [args["W[0]"], args["W[1]"]], args["D"], device=1)
