"""Operator determination on a model graph (step 101 of the method).

Patent "数据处理方法、装置、设备及介质" (Alibaba, 2023), Detailed description
para. 35 and 46-47, claim 2: the operators to fuse are found in the machine
learning model itself -- a first operator whose output is the input of a
second operator, with no conversion step between them.  Here the model is a
``torch.fx.GraphModule`` and the operators are GEMMs:

* ``find_chains(gm)`` returns every maximal run of GEMM nodes g1 -> g2 -> ...
  in which each GEMM's output feeds only the next GEMM, as its left operand,
  with no node (activation, cast, transpose, bias add, ...) in between;
* ``fuse_chains(gm)`` replaces each such run by one
  :class:`FusedGemmChain` module, which runs the whole run as one cascade on
  the GPU through this package's C ABI (``b2b_chain_plan_create`` /
  ``b2b_chain_run``).

A GEMM node is ``torch.matmul`` / ``torch.mm`` / ``torch.bmm`` /
``operator.matmul`` / ``Tensor.matmul`` with a 2-D or 3-D right operand, or an
``nn.Linear`` without bias (its right operand is the transposed weight).  The
graph analysis is plain Python and needs no GPU; the fused module has no CPU
path and raises on tensors it cannot run.
"""
from __future__ import annotations

import operator
from typing import Dict, List, Optional, Sequence, Tuple

import torch
import torch.fx as fx

__all__ = ["GemmNode", "find_chains", "fuse_chains", "FusedGemmChain"]

_MATMUL_FUNCS = (torch.matmul, torch.mm, torch.bmm, operator.matmul)
# torch dtype of the activations -> library dtype of a chain
_DTYPE_NAMES = {torch.float16: "f16", torch.bfloat16: "bf16"}


class GemmNode:
    """One GEMM of the graph: ``node`` computes ``left @ right``.

    ``right`` is an fx node producing the right operand, or ``None`` for an
    ``nn.Linear``, whose right operand is ``linear.weight`` transposed.
    """

    def __init__(self, node: fx.Node, left: fx.Node, right: Optional[fx.Node], linear=None):
        self.node, self.left, self.right, self.linear = node, left, right, linear

    def __repr__(self) -> str:
        return f"GemmNode({self.node.name})"


def _as_gemm(gm: fx.GraphModule, node: fx.Node) -> Optional[GemmNode]:
    if node.op == "call_function" and node.target in _MATMUL_FUNCS and len(node.args) == 2 and not node.kwargs:
        a, b = node.args
        if isinstance(a, fx.Node) and isinstance(b, fx.Node):
            return GemmNode(node, a, b)
    if node.op == "call_method" and node.target == "matmul" and len(node.args) == 2 and not node.kwargs:
        a, b = node.args
        if isinstance(a, fx.Node) and isinstance(b, fx.Node):
            return GemmNode(node, a, b)
    if node.op == "call_module":
        mod = gm.get_submodule(node.target)
        if isinstance(mod, torch.nn.Linear) and mod.bias is None and len(node.args) == 1 and not node.kwargs:
            a = node.args[0]
            if isinstance(a, fx.Node):
                return GemmNode(node, a, None, mod)
    return None


def find_chains(gm: fx.GraphModule, min_len: int = 2, max_len: int = 8) -> List[List[GemmNode]]:
    """Maximal runs of cascaded GEMMs with nothing between them (para. 46-47).

    A run continues from GEMM g to GEMM h when g's output has exactly one
    user, h, and h takes it as its left operand (and not also as its right
    one).  Runs longer than ``max_len`` are cut into pieces of at most
    ``max_len``; pieces shorter than ``min_len`` are dropped.
    """
    gemms: Dict[fx.Node, GemmNode] = {}
    for node in gm.graph.nodes:
        g = _as_gemm(gm, node)
        if g is not None:
            gemms[node] = g

    def successor(g: GemmNode) -> Optional[GemmNode]:
        users = list(g.node.users)
        if len(users) != 1:
            return None
        h = gemms.get(users[0])
        if h is None or h.left is not g.node or h.right is g.node:
            return None
        return h

    has_pred = set()
    for g in gemms.values():
        h = successor(g)
        if h is not None:
            has_pred.add(h.node)
    chains: List[List[GemmNode]] = []
    for node in gm.graph.nodes:  # topological order
        if node not in gemms or node in has_pred:
            continue
        run = [gemms[node]]
        while True:
            h = successor(run[-1])
            if h is None:
                break
            run.append(h)
        for i in range(0, len(run), max_len):
            piece = run[i:i + max_len]
            if len(piece) >= min_len:
                chains.append(piece)
    return chains


class FusedGemmChain(torch.nn.Module):
    """``x @ W[0] @ W[1] ... @ W[S-1]`` as one fused cascade on the GPU.

    ``forward(x, *dynamic)`` takes the chain's left input and, in order, the
    right operands that are graph values (``None`` placeholders stand for the
    ``nn.Linear`` weights, held transposed here).  Right operands are
    [K_s, N_s] (shared by every leading index of x, which are folded into the
    rows) or [B, K_s, N_s] with x [B, M, K] (one matrix per batch).  The
    activations' dtype picks the chain type: fp16 or bf16 (fp32 accumulation,
    every intermediate rounded to the operand type, as the unfused chain of
    16-bit GEMMs stores it).  Inference only: the ``nn.Linear`` weights are
    copied (transposed) when the chain is fused, and the output carries no
    gradient, so inputs that require one are refused.
    """

    def __init__(self, linear_weights: Sequence[Optional[torch.Tensor]]):
        super().__init__()
        self.n_stages = len(linear_weights)
        self.static = [w is not None for w in linear_weights]
        for s, w in enumerate(linear_weights):
            if w is not None:
                # nn.Linear computes x @ weight.T: keep weight.T row-major
                self.register_buffer(f"w{s}", w.detach().t().contiguous(), persistent=False)
        self._plans: Dict[Tuple, object] = {}

    def _plan(self, key):
        # (the plan binds to the device that is current when it is created:
        # the caller makes it the activations' device)
        plan = self._plans.get(key)
        if plan is None:
            from . import ChainPlan
            dt, batch, M, K, widths, _device = key
            plan = ChainPlan(dt, batch, M, K, widths)
            self._plans[key] = plan
        return plan

    def forward(self, x: torch.Tensor, *dynamic):
        if not x.is_cuda:
            raise RuntimeError("FusedGemmChain runs on the GPU only (the fused kernels have no CPU path)")
        dt = _DTYPE_NAMES.get(x.dtype)
        if dt is None:
            raise TypeError(f"FusedGemmChain: activations of dtype {x.dtype} (fp16 or bf16 expected)")
        ws, it = [], iter(dynamic)
        for s in range(self.n_stages):
            w = getattr(self, f"w{s}") if self.static[s] else next(it)
            if w.dtype != x.dtype or w.device != x.device:
                raise TypeError("FusedGemmChain: every right operand must match the activations' dtype and device")
            ws.append(w.contiguous())
        if torch.is_grad_enabled() and (x.requires_grad or any(w.requires_grad for w in ws)):
            raise RuntimeError("FusedGemmChain is inference-only: its output has no gradient "
                               "(run it under torch.no_grad())")
        if all(w.dim() == 2 for w in ws):
            lead = x.shape[:-1]
            a = x.reshape(1, -1, x.shape[-1]).contiguous()
            batch = 1
        elif all(w.dim() == 3 for w in ws) and x.dim() == 3:
            lead = x.shape[:-1]
            a = x.contiguous()
            batch = x.shape[0]
            if any(w.shape[0] != batch for w in ws):
                raise ValueError("FusedGemmChain: batched right operands must have the batch of x")
        else:
            raise ValueError("FusedGemmChain: right operands must be all 2-D, or all 3-D with a 3-D x")
        if batch == 1 and all(w.dim() == 3 for w in ws):
            ws = [w[0] for w in ws]
        ws = [w.reshape(batch, w.shape[-2], w.shape[-1]) for w in ws]
        M, K = a.shape[1], a.shape[2]
        widths = tuple(int(w.shape[-1]) for w in ws)
        kin = K
        for w in ws:
            if w.shape[-2] != kin:
                raise ValueError(f"FusedGemmChain: right operand {tuple(w.shape)} does not follow width {kin}")
            kin = w.shape[-1]
        # plans are per device: create and run this one on the activations' GPU
        with torch.cuda.device(x.device):
            plan = self._plan((dt, batch, M, K, widths, x.device.index))
            out = plan.run(a, ws)
        return out.reshape(*lead, widths[-1])


def fuse_chains(gm: fx.GraphModule, min_len: int = 2, max_len: int = 8) -> Tuple[fx.GraphModule, int]:
    """Replace every chain found by :func:`find_chains` by a :class:`FusedGemmChain`.

    Returns the (recompiled, modified in place) graph module and the number of
    chains fused.  The fused module's right operands are the original graph
    values (for matmuls) or the transposed ``nn.Linear`` weights (held by the
    fused module).
    """
    chains = find_chains(gm, min_len, max_len)
    for idx, chain in enumerate(chains):
        name = f"b2b_fused_chain_{idx}"
        while hasattr(gm, name):
            name += "_"
        mod = FusedGemmChain([g.linear.weight if g.linear is not None else None for g in chain])
        gm.add_submodule(name, mod)
        last = chain[-1].node
        dynamic = [g.right for g in chain if g.linear is None]
        with gm.graph.inserting_after(last):
            new = gm.graph.call_module(name, args=(chain[0].left, *dynamic))
        last.replace_all_uses_with(new)
        for g in reversed(chain):
            gm.graph.erase_node(g.node)
    gm.graph.lint()
    gm.recompile()
    return gm, len(chains)
