"""Pins of the layout maps and the rearrangement relation (no GPU needed).

The patent's worked tf32 example (Fig. 3) and its offset rule are read from
``tests/golden`` and compared with the relation derived from the PTX ISA
fragment layouts.
"""
import os
import re

import pytest

from oracle import relation as rel

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_example():
    table = {}
    with open(os.path.join(GOLDEN, "tf32_group_example.txt"), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, rest = line.split(":", 1)
            new_t = int(head.replace("newt", ""))
            slots = []
            for tok in rest.split():
                t, c = tok.split(":")
                slots.append((int(t[1:]), int(c[1:])))
            table[new_t] = slots
    return table


def test_worked_example_is_the_m16n8k8_tf32_relation():
    table = _read_example()
    r = rel.relation(rel.m16n8k8_tf32_c, rel.m16n8k8_tf32_a, lanes=32, regs=4)
    for new_t, slots in table.items():
        assert [r[(new_t, j)] for j in range(4)] == slots


def test_example_repeats_for_every_group_of_four_lanes():
    r = rel.relation(rel.m16n8k8_tf32_c, rel.m16n8k8_tf32_a, lanes=32, regs=4)
    table = _read_example()
    for base in range(0, 32, 4):
        for new_t, slots in table.items():
            assert [r[(base + new_t, j)] for j in range(4)] == [(base + t, c) for t, c in slots]


def test_offset_rule_for_wide_accumulators():
    # c0..c31 per thread (8 tiles of n8, Fig. 2a); the operand holds 8 k8 steps
    with open(os.path.join(GOLDEN, "coordination_matrix.txt"), encoding="utf-8") as f:
        offset = int(re.search(r"^offset:\s*(\d+)", f.read(), re.M).group(1))
    prod = rel.tiled(rel.m16n8k8_tf32_c, 4, 8, 8)
    cons = rel.tiled(rel.m16n8k8_tf32_a, 4, 8, 8)
    r = rel.relation(prod, cons, lanes=32, regs=32)
    for lane in range(32):
        for j in range(8):
            for s in range(4):
                src_lane, src_reg = r[(lane, offset * j + s)]
                base_lane, base_reg = r[(lane, s)]
                assert (src_lane, src_reg) == (base_lane, base_reg + offset * j)


def test_f64_relation_stays_inside_four_lane_groups():
    prod = rel.tiled(rel.m8n8k4_f64_c, 2, 8, 8)           # 8 rows x 64 cols
    cons = rel.tiled(rel.m8n8k4_f64_a, 1, 16, 4)          # 16 k4 steps
    r = rel.relation(prod, cons, lanes=32, regs=16)
    for (lane, reg), (src_lane, src_reg) in r.items():
        assert lane // 4 == src_lane // 4                  # same row g
        # k-step s needs column 4s + t, which n8 tile s//2 holds in lane 2(s%2) + t//2
        s, t = reg, lane % 4
        assert src_lane % 4 == 2 * (s % 2) + t // 2
        assert src_reg == 2 * (s // 2) + (t % 2)


def test_relation_rejects_mismatched_layouts():
    with pytest.raises(ValueError):
        rel.relation(rel.m8n8k4_f64_c, rel.m16n8k8_tf32_a, lanes=32, regs=2, consumer_regs=4)


def test_apply_rounds_and_conflicts():
    rounds = [[(0, 0, 0), (2, 1, 1), (1, 0, 0), (3, 1, 1)],
              [(2, 0, 1), (0, 1, 0), (3, 0, 1), (1, 1, 0)]]
    assert rel.is_conflict_free(rounds)
    vals = [[(lane, e) for e in range(2)] for lane in range(4)]
    out = rel.apply_rounds(vals, rounds)
    assert out[0] == [(0, 0), (2, 0)]
    assert out[1] == [(0, 1), (2, 1)]
    assert not rel.is_conflict_free([[(0, 0, 0), (0, 1, 0), (1, 0, 0), (2, 0, 0)]])


@pytest.mark.parametrize("elem", [2, 4])
def test_sw128_is_a_bijection_within_each_panel(elem):
    rows, cols = 128, 256 // elem * 2
    inv = rel.sw128_inverse(rows, cols, elem)
    assert len(inv) == rows * cols
    per_row = 128 // elem
    for (r, k) in [(0, 0), (1, 0), (7, per_row - 1), (8, 3), (127, cols - 1)]:
        off = rel.sw128_kmajor_offset(r, k, elem)
        assert off // (rows * 128) == k // per_row          # panel
        assert (off % (rows * 128)) // 128 == r              # row inside the panel
    # row 0 is not swizzled; row r moves 16-byte unit u to u ^ (r % 8)
    assert rel.sw128_kmajor_offset(0, 8 // (elem // 2) if elem == 2 else 4, elem) == 16
    assert rel.sw128_kmajor_offset(3, 0, elem) == 3 * 128 + 3 * 16
