"""The accumulator -> operand rearrangement as a pure index map (needs a GB300).

The converter routine of the fused kernels is run on tagged accumulator
tiles and the operand it produces is compared, bit for bit, with the layout
maps restated in ``oracle.relation`` from the PTX ISA.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import relation as rel

pytestmark = pytest.mark.gpu

b2b = pytest.importorskip("fusion_b2b_gemm_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    torch.cuda.set_device(0)


def _image_values(dtype, img_words: torch.Tensor) -> np.ndarray:
    raw = img_words.cpu().numpy().view(np.uint16)
    if dtype == "f16":
        return raw.view(np.float16).astype(np.float64)
    return (raw.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("width", [64, 128, 256])
def test_operand_image_is_the_swizzled_k_major_layout(dtype, width):
    offsets = np.array([[rel.sw128_kmajor_offset(m, k, 2) for k in range(width)] for m in range(128)])
    assert len(np.unique(offsets)) == 128 * width
    idx = offsets // 2
    rows = np.repeat(np.arange(128.0)[:, None], width, axis=1)
    cols = np.repeat(np.arange(width, dtype=np.float64)[None, :], 128, axis=0)
    for tag in (rows, cols):   # integers below 256: exact in fp16 and bf16
        acc = torch.from_numpy(tag.astype(np.float32)).cuda()
        vals = _image_values(dtype, b2b.probe_operand_image(dtype, acc))
        assert np.array_equal(vals[idx], tag)
    # random values: the image holds each accumulator value rounded to nearest even
    rng = np.random.default_rng(5)
    x = rng.normal(size=(128, width)).astype(np.float32)
    vals = _image_values(dtype, b2b.probe_operand_image(dtype, torch.from_numpy(x).cuda()))
    kind = oracle.F16 if dtype == "f16" else oracle.BF16
    assert np.array_equal(vals[idx], oracle.round_to(kind, x.astype(np.float64)))


@pytest.mark.parametrize("width", [64, 128, 256])
def test_tf32_operand_stays_in_the_accumulator_layout(width):
    rng = np.random.default_rng(6)
    x = (rng.normal(size=(128, width)) * 10.0 ** rng.integers(-3, 4, size=(128, width))).astype(np.float32)
    # include exact ties of the tf32 rounding
    ties = (rng.integers(0x3f800000, 0x40800000, size=64, dtype=np.uint32) & 0xFFFFE000) | 0x1000
    x.reshape(-1)[:64] = ties.view(np.float32)
    out = b2b.probe_operand_image("tf32", torch.from_numpy(x).cuda())
    got = out.cpu().numpy().view(np.float32).astype(np.float64)
    assert np.array_equal(got, oracle.round_to(oracle.TF32, x.astype(np.float64)))


@pytest.mark.parametrize("tiles", [1, 2, 8])
def test_f64_register_rearrangement(tiles):
    prod = rel.tiled(rel.m8n8k4_f64_c, 2, tiles, 8)
    cons = rel.tiled(rel.m8n8k4_f64_a, 1, 2 * tiles, 4)
    r = rel.relation(prod, cons, lanes=32, regs=2 * tiles)
    # tag = lane * 1000 + register: every accumulator value is distinct
    c = np.array([[lane * 1000 + reg for reg in range(2 * tiles)] for lane in range(32)], dtype=np.float64)
    a = b2b.probe_f64_rearrange(torch.from_numpy(c).cuda()).cpu().numpy()
    for lane in range(32):
        for reg in range(2 * tiles):
            src_lane, src_reg = r[(lane, reg)]
            assert a[lane, reg] == c[src_lane, src_reg], (lane, reg)


def _halves_values(dtype, words: np.ndarray) -> np.ndarray:
    """16-bit payloads of 32-bit words, as values: [..., 2] (low half first)."""
    w = words.astype(np.uint32)
    halves = np.stack([w & 0xFFFF, w >> 16], axis=-1).astype(np.uint16)
    if dtype == "f16":
        return halves.view(np.float16).astype(np.float64)
    return (halves.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _tags(width):
    """Row, column-low and column-high tags: integers below 256, exact in
    fp16 and bf16, which together name every element of a 128 x width tile."""
    rows = np.repeat(np.arange(128.0)[:, None], width, axis=1)
    cols = np.repeat(np.arange(width, dtype=np.float64)[None, :], 128, axis=0)
    tags = [rows, cols % 256]
    if width > 256:
        tags.append(np.floor(cols / 256))
    return tags


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("width", [64, 128, 256])
def test_tensor_memory_operand_packs_two_k_per_column(dtype, width):
    # the 16-bit intermediate kept in tensor memory as GEMM2's A operand
    where = [[rel.tmem_operand16(m, k) for k in range(width)] for m in range(128)]
    flat = [(l, c, h) for row in where for (l, c, h) in row]
    assert len(set(flat)) == 128 * width            # a bijection onto the packed columns
    lane = np.array([[x[0] for x in r] for r in where])
    col = np.array([[x[1] for x in r] for r in where])
    half = np.array([[x[2] for x in r] for r in where])
    for tag in _tags(width):
        acc = torch.from_numpy(tag.astype(np.float32)).cuda()
        out = b2b.probe_operand_layout(dtype, b2b.PROBE_TMEM16, acc).cpu().numpy()
        vals = _halves_values(dtype, out.reshape(128, width // 2))
        assert np.array_equal(vals[lane, col, half], tag)
    rng = np.random.default_rng(7)
    x = rng.normal(size=(128, width)).astype(np.float32)
    out = b2b.probe_operand_layout(dtype, b2b.PROBE_TMEM16, torch.from_numpy(x).cuda()).cpu().numpy()
    vals = _halves_values(dtype, out.reshape(128, width // 2))
    kind = oracle.F16 if dtype == "f16" else oracle.BF16
    assert np.array_equal(vals[lane, col, half], oracle.round_to(kind, x.astype(np.float64)))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("width,region", [(128, 0), (256, 1), (384, 0), (512, 1)])
def test_pair_converters_write_the_swizzled_k_major_layout(dtype, width, region):
    # eight converter warps, two per TMEM lane quadrant (64 of every 128
    # columns each), an accumulator starting in either tensor-memory region
    offsets = np.array([[rel.sw128_kmajor_offset(m, k, 2) for k in range(width)] for m in range(128)])
    assert len(np.unique(offsets)) == 128 * width
    idx = offsets // 2
    for tag in _tags(width):
        acc = torch.from_numpy(tag.astype(np.float32)).cuda()
        out = b2b.probe_operand_layout(dtype, b2b.PROBE_PAIR_CONVERTERS, acc, region)
        vals = _image_values(dtype, out)
        assert np.array_equal(vals[idx], tag)
    rng = np.random.default_rng(8)
    x = rng.normal(size=(128, width)).astype(np.float32)
    out = b2b.probe_operand_layout(dtype, b2b.PROBE_PAIR_CONVERTERS, torch.from_numpy(x).cuda(), region)
    kind = oracle.F16 if dtype == "f16" else oracle.BF16
    assert np.array_equal(_image_values(dtype, out)[idx], oracle.round_to(kind, x.astype(np.float64)))
