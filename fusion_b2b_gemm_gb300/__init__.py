"""Python binding of the fused cascaded GEMM library (``libb2b.so``).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/b2b.h``.  PyTorch supplies
device memory and streams.  There is no fallback: if the library is missing
this module raises on import, telling how to build it.

Low-level functions carry the C names (``b2b_plan_create``, ``b2b_run``,
...); :class:`Plan`, :class:`ChainPlan` and :class:`GemmPlan` wrap them for
torch tensors.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

__all__ = [
    "B2BError", "DTYPES", "MAX_STAGES", "Plan", "ChainPlan", "GemmPlan", "library_path",
    "b2b_plan_create", "b2b_chain_plan_create", "b2b_gemm_plan_create", "b2b_run", "b2b_chain_run",
    "b2b_plan_destroy",
    "b2b_plan_device_status", "b2b_plan_set_wait_budget", "b2b_plan_set_debug", "b2b_plan_info",
    "b2b_status_string", "b2b_coordination_matrix", "b2b_probe_operand_image",
    "b2b_probe_operand_layout", "b2b_schedule_table", "b2b_probe_f64_rearrange", "b2b_run_tf32_noalloc", "coordination_matrix",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_lib", "libb2b.so")

# b2b_dtype_t
DTYPES = {"f16_f32out": 0, "f16": 1, "bf16": 2, "tf32": 3, "f64": 4, "bf16_f32out": 5,
          "tf32_f16": 6, "tf32_bf16": 7}
MAX_STAGES = 8  # B2B_MAX_STAGES
STATUS = {0: "B2B_OK", 1: "B2B_ERR_INVALID_ARG", 2: "B2B_ERR_UNSUPPORTED", 3: "B2B_ERR_ALIGNMENT",
          4: "B2B_ERR_ALIAS", 5: "B2B_ERR_DEVICE", 6: "B2B_ERR_CUDA", 7: "B2B_ERR_TIMEOUT"}


class B2BError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        super().__init__(f"{where}: {STATUS.get(self.code, self.code)} ({_lib.b2b_status_string(code).decode()})")


def library_path() -> str:
    return _LIB_PATH


def _load() -> ctypes.CDLL:
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            f"{_LIB_PATH} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()' or "
            "python fusion_b2b_gemm_gb300/_build.py)")
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.c_void_p
    i64, i32, u64 = ctypes.c_int64, ctypes.c_int, ctypes.c_uint64
    ip = ctypes.POINTER(ctypes.c_int)
    sig = {
        "b2b_plan_create": [ctypes.POINTER(P), i32, i64, i64, i64, i64, i64, i64],
        "b2b_chain_plan_create": [ctypes.POINTER(P), i32, i64, i64, i64, i32, ctypes.POINTER(i64)],
        "b2b_chain_run": [P, P, ctypes.POINTER(P), P, P],
        "b2b_gemm_plan_create": [ctypes.POINTER(P), i32, i64, i64, i64, i64],
        "b2b_run": [P, P, P, P, P, P, P],
        "b2b_plan_destroy": [P],
        "b2b_plan_device_status": [P, P],
        "b2b_plan_set_wait_budget": [P, u64],
        "b2b_plan_set_debug": [P, ctypes.c_uint32],
        "b2b_plan_info": [P, ip, ip, ip, ip, ip, ip, ip],
        "b2b_coordination_matrix": [i32, i32, ip, ip, ip, ip, ip],
        "b2b_probe_operand_image": [i32, i32, P, P, P],
        "b2b_probe_operand_layout": [i32, i32, i32, i32, P, P, P],
        "b2b_schedule_table": [i32, ctypes.POINTER(i64), i32, ctypes.POINTER(i64), i32],
        "b2b_probe_f64_rearrange": [i32, P, P, P],
        "b2b_run_tf32_noalloc": [i64, i64, i64, i64, i64, P, P, P, P, P],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.b2b_status_string.argtypes = [ctypes.c_int]
    lib.b2b_status_string.restype = ctypes.c_char_p
    return lib


_lib = _load()

# -- raw C entry points (same names as the C ABI) ---------------------------
b2b_plan_create = _lib.b2b_plan_create
b2b_chain_plan_create = _lib.b2b_chain_plan_create
b2b_chain_run = _lib.b2b_chain_run
b2b_gemm_plan_create = _lib.b2b_gemm_plan_create
b2b_run = _lib.b2b_run
b2b_plan_destroy = _lib.b2b_plan_destroy
b2b_plan_device_status = _lib.b2b_plan_device_status
b2b_plan_set_wait_budget = _lib.b2b_plan_set_wait_budget
b2b_plan_set_debug = _lib.b2b_plan_set_debug
b2b_plan_info = _lib.b2b_plan_info
b2b_status_string = _lib.b2b_status_string
b2b_coordination_matrix = _lib.b2b_coordination_matrix
b2b_probe_operand_image = _lib.b2b_probe_operand_image
b2b_probe_operand_layout = _lib.b2b_probe_operand_layout
b2b_schedule_table = _lib.b2b_schedule_table
b2b_probe_f64_rearrange = _lib.b2b_probe_f64_rearrange
b2b_run_tf32_noalloc = _lib.b2b_run_tf32_noalloc


def _check(code: int, where: str) -> None:
    if code != 0:
        raise B2BError(code, where)


def _stream_handle(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream or None


def _torch_types(dtype: str):
    """(type of A, type of each weight by stage, type of the output) of a chain type."""
    import torch
    f16, bf16, f32, f64 = torch.float16, torch.bfloat16, torch.float32, torch.float64
    a, later, out = {"f16_f32out": (f16, f16, f32), "f16": (f16, f16, f16), "bf16": (bf16, bf16, bf16),
                     "bf16_f32out": (bf16, bf16, f32), "tf32": (f32, f32, f32), "f64": (f64, f64, f64),
                     "tf32_f16": (f32, f16, f32), "tf32_bf16": (f32, bf16, f32)}[dtype]
    # mixed types: fp32 A and first weight (tf32 operands), 16-bit later weights
    return a, (lambda s: a if s == 0 else later), out


def check_operands(dtype: str, batch: int, M: int, K: int, N: Sequence[int], A, Ws: Sequence, D,
                   device: Optional[int] = None) -> None:
    """Check the tensors of one run against the plan's sizes, types and device.

    The kernels read and write exactly the plan's sizes (A [batch][M][K], W_s
    [batch][K_s][N_s], D [batch][M][N_last], dense), so a tensor with fewer
    elements, or of another type, would let them reach past its end: refused
    here.  A plan is bound to the GPU that was current when it was created
    (``device``), and its kernels run there: a tensor on another GPU would be
    read through a peer address, so it is refused too.  A plan without rows
    reads and writes nothing.
    """
    if device is not None:
        for name, t in [("A", A), ("D", D)] + [(f"W[{s}]", w) for s, w in enumerate(Ws)]:
            if t is not None and t.is_cuda and t.device.index != device:
                raise ValueError(f"{name} is on cuda:{t.device.index}, the plan on cuda:{device}")
    if batch * M == 0:
        return
    ta, tw, to = _torch_types(dtype)
    kin = K
    need = [("A", A, ta, batch * M * K)]
    for s, (n, w) in enumerate(zip(N, Ws)):
        need.append((f"W[{s}]", w, tw(s), batch * kin * n))
        kin = n
    need.append(("D", D, to, batch * M * N[-1]))
    for name, t, want, count in need:
        if t is None:
            continue  # a missing operand is the C ABI's argument error
        if t.dtype != want:
            raise TypeError(f"{name}: {t.dtype} given, {want} expected for a {dtype} chain")
        if t.numel() < count:
            raise ValueError(f"{name}: {t.numel()} elements given, the plan reads or writes {count}")


def _current_device() -> int:
    """The CUDA device a new plan binds to (the current one)."""
    import torch
    return torch.cuda.current_device()


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to b2b_run must live on the GPU")
    if not t.is_contiguous():
        raise ValueError("tensors passed to b2b_run must be contiguous (row-major)")
    return t.data_ptr()


class Plan:
    """A fused chain D = (A.B).C, or E = ((A.B).C).F when ``N3 > 0``."""

    _single = False

    def __init__(self, dtype: str, batch: int, M: int, K: int, N1: int, N2: int = 0, N3: int = 0):
        if dtype not in DTYPES:
            raise ValueError(f"unknown dtype {dtype!r}; one of {sorted(DTYPES)}")
        self.dtype = dtype
        self.batch, self.M, self.K = batch, M, K
        self.N = (N1,) if self._single else ((N1, N2, N3) if N3 else (N1, N2))
        h = ctypes.c_void_p()
        if self._single:
            code = _lib.b2b_gemm_plan_create(ctypes.byref(h), DTYPES[dtype], batch, M, K, N1)
        else:
            code = _lib.b2b_plan_create(ctypes.byref(h), DTYPES[dtype], batch, M, K, N1, N2, N3)
        _check(code, "b2b_plan_create")
        self._h = h
        self.device_index = _current_device()

    # -- torch helpers ---------------------------------------------------
    def io_dtypes(self):
        import torch
        # (type of A, type of the output); the mixed types' later weights are
        # 16-bit (weight_dtypes)
        table = {"f16_f32out": (torch.float16, torch.float32), "f16": (torch.float16, torch.float16),
                 "bf16": (torch.bfloat16, torch.bfloat16), "bf16_f32out": (torch.bfloat16, torch.float32),
                 "tf32": (torch.float32, torch.float32), "f64": (torch.float64, torch.float64),
                 "tf32_f16": (torch.float32, torch.float32), "tf32_bf16": (torch.float32, torch.float32)}
        return table[self.dtype]

    def out_shape(self) -> Tuple[int, int, int]:
        return (self.batch, self.M, self.N[-1])

    def empty_out(self, device="cuda"):
        import torch
        return torch.empty(self.out_shape(), dtype=self.io_dtypes()[1], device=device)

    def run(self, A, B, C=None, F=None, D=None, stream=None):
        """Launch on ``stream`` (default: torch's current stream); returns D."""
        if D is None:
            D = self.empty_out(A.device)
        check_operands(self.dtype, self.batch, self.M, self.K, self.N, A, [B, C, F][:len(self.N)], D,
                       self.device_index)
        code = _lib.b2b_run(self._h, _ptr(A), _ptr(B), _ptr(C), _ptr(F), _ptr(D), _stream_handle(stream))
        _check(code, "b2b_run")
        return D

    def run_from_host(self, host_inputs: Sequence, host_out, dev_inputs: Sequence, dev_out, stream=None,
                      chunks: Optional[int] = None, graph: bool = True):
        """One end-to-end call from pinned host buffers.

        Copies the inputs host->device, runs the chain, copies the result
        device->host; returns (h2d_bytes, d2h_bytes).  The device buffers are
        the caller's.  The call starts and ends on ``stream``.

        With ``chunks`` > 1 (default: 2 when the call moves more than 16 MB,
        4 above 64 MB; on a GB300 more chunks cost more host time per call
        than they overlap)
        the work is cut along the batch, or along the rows of A when there is
        one batch: the upload of chunk i+1, the chain on chunk i (on
        ``stream``) and the download of chunk i-1 overlap, the copies on two
        side streams of this plan.  Every row tile is computed as in one call,
        so the result is the same.  With ``graph`` (default) the chunked
        pipeline is captured in a CUDA graph on its first call for a set of
        buffers and replayed afterwards (host memory must be pinned).
        """
        import torch
        s = stream or torch.cuda.current_stream()
        h2d = sum(h.numel() * h.element_size() for h in host_inputs)
        d2h = host_out.numel() * host_out.element_size()
        pieces = self._host_chunks(chunks, h2d + d2h)
        if len(pieces) <= 1:
            with torch.cuda.stream(s):
                for h, d in zip(host_inputs, dev_inputs):
                    d.copy_(h, non_blocking=True)
                self._run_inputs(list(dev_inputs), dev_out, s)
                host_out.copy_(dev_out, non_blocking=True)
            return h2d, d2h
        for lo, hi in pieces:  # every chunk's plan exists before any capture
            self._sub_plan(hi - lo, self.M) if self.batch > 1 else self._sub_plan(1, hi - lo)
        s_in, s_out = self._side_streams(s.device)
        if not graph:
            self._pipeline(pieces, host_inputs, host_out, dev_inputs, dev_out, s, s_in, s_out)
            return h2d, d2h
        # The chunked pipeline is captured once per set of buffers and
        # replayed: a replay costs the host a few microseconds where the
        # eager form spends tens per chunk.
        key = (tuple(t.data_ptr() for t in host_inputs), host_out.data_ptr(),
               tuple(t.data_ptr() for t in dev_inputs), dev_out.data_ptr(), tuple(pieces),
               tuple(tuple(t.shape) for t in host_inputs), s.device.index)
        graphs = self.__dict__.setdefault("_graphs", {})
        g = graphs.get(key)
        if g is None:
            if len(graphs) >= 4:
                graphs.pop(next(iter(graphs)))
            g = torch.cuda.CUDAGraph()
            cap = torch.cuda.Stream(device=s.device)
            cap.wait_stream(s)
            with torch.cuda.graph(g, stream=cap):
                self._pipeline(pieces, host_inputs, host_out, dev_inputs, dev_out, cap, s_in, s_out)
            s.wait_stream(cap)
            graphs[key] = g
        with torch.cuda.stream(s):
            g.replay()
        return h2d, d2h

    def _pipeline(self, pieces, host_inputs, host_out, dev_inputs, dev_out, s, s_in, s_out):
        """Upload chunk i+1 on s_in, run chunk i on s, download chunk i-1 on s_out."""
        import torch
        start = torch.cuda.Event()
        start.record(s)
        s_in.wait_event(start)
        s_out.wait_event(start)
        by_batch = self.batch > 1
        loaded = []
        with torch.cuda.stream(s_in):
            if not by_batch:  # one batch: the weights go up once, before the first rows
                for h, d in zip(host_inputs[1:], dev_inputs[1:]):
                    d.copy_(h, non_blocking=True)
            for lo, hi in pieces:
                for i, (h, d) in enumerate(zip(host_inputs, dev_inputs)):
                    if by_batch:
                        d[lo:hi].copy_(h[lo:hi], non_blocking=True)
                    elif i == 0:
                        d[:, lo:hi].copy_(h[:, lo:hi], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(s_in)
                loaded.append(ev)
        for (lo, hi), ev in zip(pieces, loaded):
            s.wait_event(ev)
            if by_batch:
                sub_in = [d[lo:hi] for d in dev_inputs]
                sub_out = dev_out[lo:hi]
                plan = self._sub_plan(hi - lo, self.M)
            else:
                sub_in = [dev_inputs[0][:, lo:hi]] + list(dev_inputs[1:])
                sub_out = dev_out[:, lo:hi]
                plan = self._sub_plan(1, hi - lo)
            plan._run_inputs(sub_in, sub_out, s)
            done = torch.cuda.Event()
            done.record(s)
            s_out.wait_event(done)
            with torch.cuda.stream(s_out):
                if by_batch:
                    host_out[lo:hi].copy_(sub_out, non_blocking=True)
                else:
                    host_out[:, lo:hi].copy_(sub_out, non_blocking=True)
        s.wait_stream(s_out)

    def _host_chunks(self, chunks, nbytes):
        """[(lo, hi)] along the batch, or along the rows (multiples of 256) of one batch."""
        if chunks is None:
            chunks = 4 if nbytes > (64 << 20) else (2 if nbytes > (16 << 20) else 1)
        n = chunks
        if n <= 1 or self.batch == 0 or self.M == 0:
            return [(0, self.batch)]
        if self.batch > 1:
            n = min(n, self.batch)
            edges = [self.batch * i // n for i in range(n + 1)]
        else:
            units = (self.M + 255) // 256
            n = min(n, units)
            edges = [min(self.M, 256 * (units * i // n)) for i in range(n + 1)]
        return [(lo, hi) for lo, hi in zip(edges, edges[1:]) if hi > lo]

    def _side_streams(self, device):
        import torch
        st = getattr(self, "_streams", None)
        if st is None or st[0] != device:
            st = (device, torch.cuda.Stream(device=device), torch.cuda.Stream(device=device))
            self._streams = st
        return st[1], st[2]

    def _sub_plan(self, batch: int, M: int):
        cache = self.__dict__.setdefault("_subs", {})
        key = (batch, M)
        if key not in cache:
            cache[key] = self._make_like(batch, M)
        return cache[key]

    def _make_like(self, batch: int, M: int):
        if self._single:
            return GemmPlan(self.dtype, batch, M, self.K, self.N[0])
        return ChainPlan(self.dtype, batch, M, self.K, self.N)

    def _run_inputs(self, inputs, D, stream):
        args = inputs + [None] * (4 - len(inputs))
        self.run(args[0], args[1], args[2], args[3], D, stream=stream)

    def status(self, stream=None) -> int:
        """Synchronise and return the device status word (0 = OK)."""
        return int(_lib.b2b_plan_device_status(self._h, _stream_handle(stream)))

    def set_wait_budget(self, ns: int) -> None:
        _check(_lib.b2b_plan_set_wait_budget(self._h, int(ns)), "b2b_plan_set_wait_budget")

    def set_debug(self, flags: int) -> None:
        """Test support (see b2b_plan_set_debug in include/b2b.h)."""
        _check(_lib.b2b_plan_set_debug(self._h, int(flags)), "b2b_plan_set_debug")

    def info(self) -> dict:
        vals = [ctypes.c_int() for _ in range(7)]
        _check(_lib.b2b_plan_info(self._h, *[ctypes.byref(v) for v in vals]), "b2b_plan_info")
        keys = ("launches_per_run", "grid", "threads", "smem_bytes", "tmem_cols", "ring_stages", "passes")
        return {k: v.value for k, v in zip(keys, vals)}

    def close(self) -> None:
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            _lib.b2b_plan_destroy(h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class ChainPlan(Plan):
    """A cascade of GEMMs E = (..((A.W[0]).W[1])..).W[S-1], 1 <= S <= MAX_STAGES.

    ``widths`` are the output widths N[0..S-1] of the GEMMs.
    """

    def __init__(self, dtype: str, batch: int, M: int, K: int, widths: Sequence[int]):
        if dtype not in DTYPES:
            raise ValueError(f"unknown dtype {dtype!r}; one of {sorted(DTYPES)}")
        widths = tuple(int(w) for w in widths)
        self.dtype = dtype
        self.batch, self.M, self.K = batch, M, K
        self.N = widths
        h = ctypes.c_void_p()
        arr = (ctypes.c_int64 * max(1, len(widths)))(*widths)
        _check(_lib.b2b_chain_plan_create(ctypes.byref(h), DTYPES[dtype], batch, M, K, len(widths), arr),
               "b2b_chain_plan_create")
        self._h = h
        self.device_index = _current_device()

    def run(self, A, Ws: Sequence, D=None, stream=None):
        """Launch on ``stream`` (default: torch's current stream); returns D."""
        if D is None:
            D = self.empty_out(A.device)
        check_operands(self.dtype, self.batch, self.M, self.K, self.N, A, list(Ws)[:len(self.N)], D,
                       self.device_index)
        ptrs = (ctypes.c_void_p * max(1, len(Ws)))(*[_ptr(w) for w in Ws])
        _check(_lib.b2b_chain_run(self._h, _ptr(A), ptrs, _ptr(D), _stream_handle(stream)), "b2b_chain_run")
        return D

    def _run_inputs(self, inputs, D, stream):
        self.run(inputs[0], inputs[1:], D, stream=stream)


class GemmPlan(Plan):
    """A single GEMM D = A.B (one operator; the unfused chain is built from these)."""

    _single = True

    def __init__(self, dtype: str, batch: int, M: int, K: int, N: int):
        super().__init__(dtype, batch, M, K, N)

    def run(self, A, B, C=None, F=None, D=None, stream=None):
        return super().run(A, B, None, None, D, stream)


def coordination_matrix(src_thread: Sequence[Sequence[int]], src_reg: Sequence[Sequence[int]]):
    """H as a list of rows [(p, q, r), ...] (one triple per round)."""
    n, m = len(src_thread), len(src_thread[0])
    flat_t = (ctypes.c_int * (n * m))(*[x for row in src_thread for x in row])
    flat_r = (ctypes.c_int * (n * m))(*[x for row in src_reg for x in row])
    P, Q, R = [(ctypes.c_int * (n * m))() for _ in range(3)]
    _check(_lib.b2b_coordination_matrix(n, m, flat_t, flat_r, P, Q, R), "b2b_coordination_matrix")
    return [[(P[i * m + j], Q[i * m + j], R[i * m + j]) for j in range(m)] for i in range(n)]


def probe_operand_image(dtype: str, acc):
    """Run the converter routine on acc (torch fp32 [128, width] on the GPU)."""
    import torch
    width = acc.shape[1]
    if dtype == "tf32":
        out = torch.empty((128, width), dtype=torch.int32, device=acc.device)
    else:
        out = torch.empty((width * 256 // 4,), dtype=torch.int32, device=acc.device)
    _check(_lib.b2b_probe_operand_image(DTYPES[dtype], width, _ptr(acc.contiguous()), _ptr(out),
                                        _stream_handle(None)), "b2b_probe_operand_image")
    return out


PROBE_TMEM16, PROBE_PAIR_CONVERTERS = 1, 2  # B2B_PROBE_*
TABLE_REGION_USE, TABLE_PAIR_UNITS, TABLE_PAIR_REGIONS, TABLE_PAIR_TMEM_INTERMEDIATES = 1, 2, 3, 4  # B2B_TABLE_*


def schedule_table(table: int, args: Sequence[int], nout: int):
    """One of the kernels' scheduling tables, evaluated on the host (test support)."""
    a = (ctypes.c_int64 * max(1, len(args)))(*args)
    out = (ctypes.c_int64 * nout)()
    _check(_lib.b2b_schedule_table(table, a, len(args), out, nout), "b2b_schedule_table")
    return list(out)


def probe_operand_layout(dtype: str, form: int, acc, region: int = 0):
    """Run another form of the 16-bit rearrangement on acc (torch fp32 [128, width] on the GPU)."""
    import torch
    width = acc.shape[1]
    words = 128 * width // 2 if form == PROBE_TMEM16 else width * 256 // 4
    out = torch.empty((words,), dtype=torch.int32, device=acc.device)
    _check(_lib.b2b_probe_operand_layout(DTYPES[dtype], form, width, region, _ptr(acc.contiguous()), _ptr(out),
                                         _stream_handle(None)), "b2b_probe_operand_layout")
    return out


def probe_f64_rearrange(cfrag):
    """cfrag: torch fp64 [32, tiles*2] on the GPU -> afrag of the same shape."""
    import torch
    tiles = cfrag.shape[1] // 2
    out = torch.empty_like(cfrag)
    _check(_lib.b2b_probe_f64_rearrange(tiles, _ptr(cfrag.contiguous()), _ptr(out), _stream_handle(None)),
           "b2b_probe_f64_rearrange")
    return out
