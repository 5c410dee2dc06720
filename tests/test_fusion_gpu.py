"""A model whose GEMM cascades were found and fused on its fx graph runs them
through the fused kernels (needs a GB300).

The fused model is checked element by element against the CPU oracle applied
to the same pieces (each fused cascade: fp32 accumulation, every intermediate
and the output rounded to the activations' 16-bit type; the graph's other
nodes, here a ReLU, applied exactly between them), and, as a second check,
against the unfused model run by torch.
"""
import numpy as np
import pytest
import torch
import torch.fx as fx

import oracle

pytestmark = pytest.mark.gpu

b2b = pytest.importorskip("fusion_b2b_gemm_gb300")
from fusion_b2b_gemm_gb300 import fusion  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    torch.cuda.set_device(0)


class Mlp(torch.nn.Module):
    def __init__(self, dims, act_after=()):
        super().__init__()
        self.layers = torch.nn.ModuleList(torch.nn.Linear(a, b, bias=False) for a, b in zip(dims, dims[1:]))
        self.act_after = set(act_after)

    def forward(self, x):
        for i, layer in enumerate(self.layers):
            x = layer(x)
            if i in self.act_after:
                x = torch.relu(x)
        return x


def rel(a, b):
    a, b = a.detach().float(), b.detach().float()
    return float((a - b).abs().max() / b.abs().max())


def rel_oracle(got, want: np.ndarray) -> float:
    g = got.detach().double().cpu().numpy()
    return float(np.max(np.abs(g - want)) / max(np.max(np.abs(want)), 1e-300))


def oracle_chain(x: torch.Tensor, weights, dtype) -> np.ndarray:
    """One fused cascade on the CPU oracle: rows of x (leading indices folded)
    through the weights ([K_s, N_s], or [B, K_s, N_s] per batch)."""
    mid = oracle.F16 if dtype == torch.float16 else oracle.BF16
    a = oracle.widen(x)
    if weights[0].dim() == 2:
        a = a.reshape(1, -1, a.shape[-1])
    out = oracle.chain(a, [oracle.widen(w) for w in weights], oracle.F32, mid, mid)
    return out.reshape(*x.shape[:-1], out.shape[-1])


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_fused_mlp_matches_the_unfused_model(dtype):
    torch.manual_seed(0)
    model = Mlp([256, 512, 256, 128, 256, 64], act_after=(2,)).to("cuda", dtype)
    for layer in model.layers:
        torch.nn.init.normal_(layer.weight, 0.0, layer.in_features ** -0.5)
    x = torch.randn(4, 300, 256, device="cuda", dtype=dtype)
    want = model(x)
    gm, n = fusion.fuse_chains(fx.symbolic_trace(model))
    assert n == 2
    got = gm(x)
    torch.cuda.synchronize()
    assert got.shape == want.shape and got.dtype == dtype
    # the oracle on the fused pieces: layers 0-2, ReLU (exact), layers 3-4
    wt = [layer.weight.detach().t() for layer in model.layers]
    h = oracle_chain(x, wt[:3], dtype)
    h = torch.from_numpy(np.maximum(h, 0.0)).to(dtype)        # exact: h is already 16-bit
    want_oracle = oracle_chain(h, wt[3:], dtype)
    assert rel_oracle(got, want_oracle) <= 1e-2
    # and the unfused model run by torch
    assert rel(got, want) <= 1e-2
    for name, mod in gm.named_modules():
        if isinstance(mod, fusion.FusedGemmChain):
            assert all(p.status() == 0 for p in mod._plans.values())


def test_batched_matmul_chain():
    class M(torch.nn.Module):
        def forward(self, x, w0, w1, w2):
            return torch.bmm(torch.bmm(x, w0), w1) @ w2
    torch.manual_seed(1)
    B, Mr, K, N = 3, 200, 128, (256, 128, 192)
    x = torch.randn(B, Mr, K, device="cuda", dtype=torch.float16)
    ws, kin = [], K
    for n in N:
        ws.append(torch.randn(B, kin, n, device="cuda", dtype=torch.float16) / kin ** 0.5)
        kin = n
    gm = fx.symbolic_trace(M())
    want = gm(x, *ws)
    gm, n = fusion.fuse_chains(gm)
    assert n == 1
    got = gm(x, *ws)
    torch.cuda.synchronize()
    assert rel_oracle(got, oracle_chain(x, ws, torch.float16)) <= 1e-2
    assert rel(got, want) <= 1e-2


def test_fused_module_rejects_fp32_activations_and_gradients():
    gm, _ = fusion.fuse_chains(fx.symbolic_trace(Mlp([64, 64, 64]).cuda()))
    with pytest.raises(TypeError):
        gm(torch.randn(2, 64, device="cuda"))
    gm = gm.half()
    x = torch.randn(2, 64, device="cuda", dtype=torch.float16, requires_grad=True)
    with pytest.raises(RuntimeError, match="inference-only"):
        gm(x)
    with torch.no_grad():
        assert gm(x).shape == (2, 64)
