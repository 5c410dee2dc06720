"""CPU oracle for the fused cascaded GEMM -- test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or calls it, and this package imports
nothing from the product.

The arithmetic lives in ``oracle.c`` (plain C, fp64 loops); this module only
compiles it with the host compiler and marshals numpy arrays.  The
rearrangement relation between the accumulator layout and the operand layout
is restated separately in :mod:`oracle.relation`.

Source: patent "数据处理方法、装置、设备及介质" (Alibaba, 2023), Detailed
description para. 28-31 (GEMM, cascaded GEMM), para. 41 (three cascaded
operators), para. 70 and 79 (rearrangement keeps every element).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

__all__ = [
    "NONE", "F32", "F16", "BF16", "TF32", "TF32_RNE",
    "build", "round_to", "chain", "max_threads", "widen",
]

NONE, F32, F16, BF16, TF32, TF32_RNE = 0, 1, 2, 3, 4, 5

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``oracle/_build/liboracle.so`` (gcc, OpenMP)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            lib.oracle_round1.restype = ctypes.c_double
            lib.oracle_round1.argtypes = [ctypes.c_int, ctypes.c_double]
            lib.oracle_round.restype = None
            lib.oracle_round.argtypes = [ctypes.c_int, dp, dp, ctypes.c_int64]
            lib.oracle_chain.restype = ctypes.c_int
            lib.oracle_chain.argtypes = [
                ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.POINTER(ctypes.c_int64), dp, ctypes.POINTER(dp),
                ctypes.c_int, ctypes.c_int, ctypes.c_int, dp, ctypes.c_int]
            lib.oracle_max_threads.restype = ctypes.c_int
            lib.oracle_max_threads.argtypes = []
            _lib = lib
    return _lib


def _dptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def round_to(kind: int, x) -> np.ndarray:
    """Round every element of ``x`` (read as fp64) to the format ``kind``."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    y = np.empty_like(x)
    _load().oracle_round(int(kind), _dptr(x), _dptr(y), x.size)
    return y


def widen(t) -> np.ndarray:
    """Exact fp64 copy of a stored input (numpy array or torch CPU tensor).

    bfloat16 is read through its bit pattern (the top half of a binary32),
    so no rounding happens anywhere on the way to fp64.
    """
    try:
        import torch  # only for tensors handed in by the caller
        if isinstance(t, torch.Tensor):
            t = t.detach().cpu()
            if t.dtype == torch.bfloat16:
                bits = t.contiguous().view(torch.int16).numpy().astype(np.uint16)
                return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            t = t.numpy()
    except ImportError:  # pragma: no cover - torch is always present here
        pass
    return np.asarray(t).astype(np.float64)


def chain(A, weights, acc: int, interm: int, out: int, n_threads: int = 0) -> np.ndarray:
    """Cascaded product ``round_out(...round_interm(A.W1)...W_last)``.

    ``A`` is [batch, M, K]; ``weights[s]`` is [batch, K_s, N_s] with
    K_0 = K and K_s = N_{s-1}.  Every product is accumulated in fp64 and
    rounded once to ``acc`` (F32, or NONE for an fp64 chain); intermediates
    are then rounded to ``interm`` and the last product to ``out``.
    """
    A = np.ascontiguousarray(np.asarray(A, dtype=np.float64))
    if A.ndim == 2:
        A = A[None]
    Ws = []
    for w in weights:
        w = np.ascontiguousarray(np.asarray(w, dtype=np.float64))
        if w.ndim == 2:
            w = np.broadcast_to(w, (A.shape[0],) + w.shape).copy()
        Ws.append(w)
    batch, M, K = A.shape
    ns = []
    kin = K
    for w in Ws:
        if w.shape[0] != batch or w.shape[1] != kin:
            raise ValueError(f"weight shape {w.shape} does not follow {kin}")
        ns.append(w.shape[2])
        kin = w.shape[2]
    res = np.empty((batch, M, ns[-1]), dtype=np.float64)
    n_arr = (ctypes.c_int64 * len(ns))(*ns)
    w_arr = (ctypes.POINTER(ctypes.c_double) * len(Ws))(*[_dptr(w) for w in Ws])
    rc = _load().oracle_chain(len(Ws), batch, M, K, n_arr, _dptr(A), w_arr,
                              int(acc), int(interm), int(out), _dptr(res), int(n_threads))
    if rc != 0:
        raise RuntimeError("oracle_chain rejected its arguments")
    return res
