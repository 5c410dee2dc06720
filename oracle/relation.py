"""Data layouts and the data rearrangement relation -- test infrastructure only.

The patent "数据处理方法、装置、设备及介质" (Alibaba, 2023) calls the way a
computing unit holds a matrix in its thread registers a "data processing
rule" (数据处理规律, Detailed description para. 39, 53).  GEMM1's result
follows rule 1, GEMM2's operand follows rule 2, and when the two differ the
"data rearrangement relation" (数据重排关系) says which register of which
thread each operand element comes from (para. 61-70, Fig. 3).

This module states those rules as plain index maps and derives the relation
from them.  The register layouts are the warp-level ``mma.sync`` fragment
layouts of the public PTX ISA; the on-chip layouts of the tensor-memory
accumulator and of the 128-byte-swizzled shared-memory operand image are the
ones the PTX ISA documents for ``tcgen05``.  Nothing here is imported by the
product; the tests compare the product's kernels and its coordination-matrix
generator against these maps.

Pins: the patent's worked tf32 example (para. 116-125, Fig. 3) and its
offset rule (para. 72-74) are stored under ``tests/golden`` and checked
against :func:`relation` on the m16n8k8 tf32 fragments; the shared-memory
image is checked against the GPU both by the layout probe and, independently,
by the tensor cores consuming it in the parity tests.
"""
from __future__ import annotations

from typing import Callable, Dict, List, Tuple

Coord = Tuple[int, int]                  # (row, col) of the logical matrix
Slot = Tuple[int, int]                   # (lane, register index)
Layout = Callable[[int, int], Coord]     # (lane, register) -> (row, col)


# --------------------------------------------------------------------------
# Register fragment layouts of warp-level MMA (PTX ISA, "Matrix fragments for
# mma.m16n8k8" with .tf32 and "Matrix fragments for mma.m8n8k4" with .f64).
# Lane l is split as g = l // 4 (group) and t = l % 4 (thread in group).
# --------------------------------------------------------------------------

def m16n8k8_tf32_c(lane: int, reg: int) -> Coord:
    """Accumulator C/D of m16n8k8 (fp32): regs 0,1 on row g, 2,3 on row g+8."""
    g, t = divmod(lane, 4)
    return (g + 8 * (reg // 2), 2 * t + (reg % 2))


def m16n8k8_tf32_a(lane: int, reg: int) -> Coord:
    """Operand A of m16n8k8 .tf32: a0=(g,t) a1=(g+8,t) a2=(g,t+4) a3=(g+8,t+4)."""
    g, t = divmod(lane, 4)
    return (g + 8 * (reg % 2), t + 4 * (reg // 2))


def m8n8k4_f64_c(lane: int, reg: int) -> Coord:
    """Accumulator C/D of m8n8k4 .f64: two values per lane on row g."""
    g, t = divmod(lane, 4)
    return (g, 2 * t + reg)


def m8n8k4_f64_a(lane: int, reg: int) -> Coord:
    """Operand A of m8n8k4 .f64: one value per lane, (g, t)."""
    assert reg == 0
    g, t = divmod(lane, 4)
    return (g, t)


def tiled(layout: Layout, regs_per_tile: int, tiles: int, col_step: int) -> Layout:
    """A thread's registers for ``tiles`` tiles side by side along columns.

    Register ``j*regs_per_tile + r`` holds tile ``j``'s register ``r``; tile
    ``j`` starts at column ``j*col_step``.  This is how one thread holds
    c0..c31 of a wide accumulator (para. 58, Fig. 2a).
    """
    def f(lane: int, reg: int) -> Coord:
        j, r = divmod(reg, regs_per_tile)
        if j >= tiles:
            raise IndexError(reg)
        row, col = layout(lane, r)
        return (row, col + j * col_step)
    return f


def relation(producer: Layout, consumer: Layout, lanes: int, regs: int,
             consumer_regs: int | None = None) -> Dict[Slot, Slot]:
    """The data rearrangement relation between two register layouts.

    For every consumer slot (lane, register) it gives the producer slot that
    holds the same matrix element (para. 65-66: the correspondence of matrix
    elements between the first and second rearrangement group matrices).
    Raises if the two layouts do not cover the same elements.
    """
    consumer_regs = regs if consumer_regs is None else consumer_regs
    where: Dict[Coord, Slot] = {}
    for lane in range(lanes):
        for r in range(regs):
            c = producer(lane, r)
            if c in where:
                raise ValueError(f"producer holds {c} twice")
            where[c] = (lane, r)
    rel: Dict[Slot, Slot] = {}
    for lane in range(lanes):
        for r in range(consumer_regs):
            c = consumer(lane, r)
            if c not in where:
                raise ValueError(f"consumer needs {c}, which the producer lacks")
            rel[(lane, r)] = where[c]
    if len(rel) != len(where):
        raise ValueError("layouts do not cover the same elements")
    return rel


def relation_table(rel: Dict[Slot, Slot], lanes: List[int], regs: int) -> List[List[Slot]]:
    """Rows new_t -> [(old lane, old register) for each new register]."""
    return [[rel[(l, r)] for r in range(regs)] for l in lanes]


def is_conflict_free(rounds: List[List[Tuple[int, int, int]]]) -> bool:
    """Para. 90: in each round no two receivers ask the same sender.

    ``rounds[j][i] = (p, q, r)`` -- receiver i takes element q of lane p into
    its register r during round j.
    """
    for col in rounds:
        ps = [p for (p, _, _) in col]
        if len(set(ps)) != len(ps):
            return False
    return True


def apply_rounds(values: List[List[object]], rounds: List[List[Tuple[int, int, int]]]):
    """Carry out exchange rounds on per-lane register lists (a plain model).

    Each round every receiver i copies ``values[p][q]`` into its result
    register ``r``; the inputs never change during the exchange.
    """
    n = len(values)
    out: List[List[object]] = [[None] * len(values[0]) for _ in range(n)]
    for col in rounds:
        for i, (p, q, r) in enumerate(col):
            out[i][r] = values[p][q]
    return out


# --------------------------------------------------------------------------
# tcgen05 layouts (PTX ISA: "Tensor Memory" data-path layout for M = 128 with
# one CTA, and "Shared memory descriptor" canonical K-major layout with the
# 128-byte swizzle).
# --------------------------------------------------------------------------

def tmem_accumulator(row: int, col: int) -> Tuple[int, int]:
    """fp32 accumulator of a 128-row tcgen05.mma: row -> lane, col -> column."""
    if not (0 <= row < 128):
        raise IndexError(row)
    return (row, col)


def sw128_kmajor_offset(row: int, k: int, elem_bytes: int, rows: int = 128) -> int:
    """Byte offset of element (row, k) in a K-major 128B-swizzled operand image.

    The image is split along K into 128-byte-wide panels (64 16-bit or 32
    32-bit elements) of ``rows`` rows each; row r of a panel starts at
    r * 128 bytes, and inside it the 16-byte unit u is stored at unit
    u XOR (r mod 8).  This is also the layout the TMA engine reads and writes
    for a box whose inner extent is 128 bytes with CU_TENSOR_MAP_SWIZZLE_128B.
    """
    per_row = 128 // elem_bytes
    panel, kk = divmod(k, per_row)
    unit, within = divmod(kk * elem_bytes, 16)
    return panel * rows * 128 + row * 128 + ((unit ^ (row % 8)) << 4) + within


def sw128_inverse(rows: int, cols: int, elem_bytes: int) -> Dict[int, Coord]:
    """Map from byte offset (element start) back to (row, k)."""
    inv: Dict[int, Coord] = {}
    for r in range(rows):
        for k in range(cols):
            off = sw128_kmajor_offset(r, k, elem_bytes, rows)
            if off in inv:
                raise ValueError("not a bijection")
            inv[off] = (r, k)
    return inv


def tmem_operand16(row: int, k: int) -> Tuple[int, int, int]:
    """Where element (row, k) of a 16-bit A operand sits in tensor memory.

    A tcgen05.mma of kind::f16 whose A operand (M = 128 rows, one CTA) comes
    from tensor memory reads row m from lane m, and two consecutive K elements
    from each 32-bit column: K elements 2c and 2c + 1 share column c, the even
    one in the low 16 bits.  Returns (lane, column, half), half 0 = bits 0-15.
    """
    if not (0 <= row < 128) or k < 0:
        raise IndexError((row, k))
    return (row, k // 2, k % 2)
