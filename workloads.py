"""Seeded synthetic workloads for the fused cascaded GEMM.

This module holds the shapes and the random-input recipes only -- none of
the method's arithmetic.  Both the CUDA path (tests, benchmark) and the CPU
oracle take their inputs from here, and this module imports neither.

Recipe: numpy PCG64 (``default_rng(seed)``), values drawn in fp64 and cast
to the storage type with round-to-nearest-even.  "N(0, s)" means standard
deviation s; "fan_in" is the contraction length of the GEMM that consumes the
matrix (A and W1 -> K, W2 -> N1, W3 -> N2).  Weights are distinct per batch.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Tuple

import numpy as np

# Storage / compute types of a chain.  The names match the C enum b2b_dtype_t.
DTYPES = ("f16_f32out", "f16", "bf16", "tf32", "f64", "bf16_f32out", "tf32_f16", "tf32_bf16")

# torch dtypes for (inputs, output); resolved lazily so that this module
# imports without torch.
_IO = {
    "f16_f32out": ("float16", "float32"),
    "f16": ("float16", "float16"),
    "bf16": ("bfloat16", "bfloat16"),
    "bf16_f32out": ("bfloat16", "float32"),
    "tf32": ("float32", "float32"),
    "f64": ("float64", "float64"),
    # mixed: fp32 A and first weight (tf32 operands), 16-bit later weights
    "tf32_f16": ("float32", "float32"),
    "tf32_bf16": ("float32", "float32"),
}
# storage type of the weights after the first, where it differs from A's
_LATER = {"tf32_f16": "float16", "tf32_bf16": "bfloat16"}


def io_dtypes(dtype: str):
    import torch
    a, b = _IO[dtype]
    return getattr(torch, a), getattr(torch, b)


def input_dtypes(dtype: str, stages: int):
    """torch storage types of [A, W1, ..., W_stages]."""
    import torch
    a, _ = _IO[dtype]
    later = _LATER.get(dtype, a)
    return [getattr(torch, a), getattr(torch, a)] + [getattr(torch, later)] * (stages - 1)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dtype: str
    batch: int
    M: int
    K: int
    N: Tuple[int, ...]          # N1, N2[, N3]
    dist: str                    # "uniform" | "normal" | "normal_fanin" | "int"
    scale: float = 1.0
    seed: int = 0
    note: str = ""

    @property
    def stages(self) -> int:
        return len(self.N)

    def flops(self) -> int:
        kin, total = self.K, 0
        for n in self.N:
            total += 2 * self.batch * self.M * kin * n
            kin = n
        return total

    def shapes(self) -> List[Tuple[int, int, int]]:
        out = [(self.batch, self.M, self.K)]
        kin = self.K
        for n in self.N:
            out.append((self.batch, kin, n))
            kin = n
        return out

    def out_shape(self) -> Tuple[int, int, int]:
        return (self.batch, self.M, self.N[-1])

    def elem_bytes(self) -> Tuple[int, int]:
        import torch
        i, o = io_dtypes(self.dtype)
        return (torch.empty((), dtype=i).element_size(), torch.empty((), dtype=o).element_size())

    def input_elem_bytes(self) -> List[int]:
        import torch
        return [torch.empty((), dtype=t).element_size() for t in input_dtypes(self.dtype, self.stages)]

    def unique_bytes(self) -> int:
        """Inputs and output, each once; the intermediates are not counted."""
        _, eo = self.elem_bytes()
        n_in = sum(int(np.prod(s)) * e for s, e in zip(self.shapes(), self.input_elem_bytes()))
        return n_in + int(np.prod(self.out_shape())) * eo

    def intermediate_bytes(self) -> int:
        """Bytes an unfused chain writes and reads back for its intermediates."""
        ei = self.input_elem_bytes()[-1]
        return sum(2 * self.batch * self.M * n * ei for n in self.N[:-1])

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads of the fused cascaded GEMM (seed = position 0..4).
WORKLOADS: Dict[str, Workload] = {
    "tiny_f16": Workload("tiny_f16", "f16_f32out", 1, 256, 64, (64, 64), "uniform", 1.0, 0,
                         "fp16 in, fp16 intermediate, fp32 out"),
    "batched_f16": Workload("batched_f16", "f16", 64, 4096, 128, (128, 128), "normal_fanin", 1.0, 1,
                            "fp16 in/out, weights distinct per batch"),
    "tf32": Workload("tf32", "tf32", 1, 16384, 256, (256, 256), "normal", 1.0 / 16, 2,
                     "fp32 storage, tf32 operands, tf32 intermediate, fp32 out"),
    "f64": Workload("f64", "f64", 8, 8192, 64, (64, 64), "uniform", 1.0, 3,
                    "fp64 throughout"),
    "three_stage_bf16": Workload("three_stage_bf16", "bf16", 1, 65536, 512, (256, 256, 512),
                                 "normal_fanin", 1.0, 4, "bf16 in/out, two bf16 intermediates"),
}

# Longer cascades and wider intermediates than the five workloads above (the
# general form of the method: each operator's output is the next one's
# input).  Measured beside them; not part of the published comparison.
EXTRA_WORKLOADS: Dict[str, Workload] = {
    "four_stage_bf16": Workload("four_stage_bf16", "bf16", 1, 65536, 256, (256, 256, 256, 256),
                                "normal_fanin", 1.0, 5, "bf16 in/out, three bf16 intermediates"),
    "wide_f16": Workload("wide_f16", "f16", 8, 8192, 128, (512, 128), "normal_fanin", 1.0, 6,
                         "fp16 in/out, one 512-column fp16 intermediate"),
    "mixed_tf32_bf16": Workload("mixed_tf32_bf16", "tf32_bf16", 1, 65536, 256, (256, 256, 256),
                                "normal_fanin", 1.0, 7,
                                "fp32 A and first weight (tf32 GEMM), bf16 intermediates and later "
                                "weights, fp32 out"),
    "tf32_batched": Workload("tf32_batched", "tf32", 4, 16384, 256, (256, 256), "normal", 1.0 / 16, 8,
                             "the tf32 workload over four batches, weights distinct per batch "
                             "(more 128-row tiles than SMs)"),
}

ALL_WORKLOADS: Dict[str, Workload] = {**WORKLOADS, **EXTRA_WORKLOADS}

BENCH_WORKLOAD = "batched_f16"


def _draw(rng: np.random.Generator, shape, dist: str, scale: float, fan_in: int) -> np.ndarray:
    if dist == "uniform":
        return rng.uniform(-scale, scale, size=shape)
    if dist == "normal":
        return rng.normal(0.0, scale, size=shape)
    if dist == "normal_fanin":
        return rng.normal(0.0, 1.0 / np.sqrt(fan_in), size=shape)
    if dist == "int":
        # integers in [-scale, scale]: every product and partial sum is exact
        s = int(scale)
        return rng.integers(-s, s + 1, size=shape).astype(np.float64)
    raise ValueError(dist)


def make_inputs(w: Workload, seed: Optional[int] = None):
    """Seeded CPU tensors [A, W1, W2(, W3)] in the workload's storage type."""
    import torch
    rng = np.random.default_rng(w.seed if seed is None else seed)
    dts = input_dtypes(w.dtype, w.stages)
    out = []
    fan = [w.K, w.K] + list(w.N[:-1])        # A, W1, W2, W3 consumers' K
    for idx, shp in enumerate(w.shapes()):
        in_dt = dts[idx]
        x = _draw(rng, shp, w.dist, w.scale, fan[idx])
        if in_dt == torch.float64:
            t = torch.from_numpy(x)
        elif in_dt == torch.float16:
            t = torch.from_numpy(x.astype(np.float16))
        elif in_dt == torch.float32:
            t = torch.from_numpy(x.astype(np.float32))
        else:  # bfloat16: fp64 -> fp32 (RNE) -> bf16 (RNE)
            t = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
        out.append(t.contiguous())
    return out


def small(w: Workload, M: int, batch: Optional[int] = None) -> Workload:
    """The same workload with fewer rows (for the oracle's quick cases)."""
    return w.with_(M=M, batch=w.batch if batch is None else batch)
