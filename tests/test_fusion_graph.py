"""Operator determination on a model graph (patent para. 46-47, claim 2): which
GEMM nodes of a torch.fx graph form a fusable cascade.  Host only."""
import pytest
import torch
import torch.fx as fx

from fusion_b2b_gemm_gb300 import fusion


class Mlp(torch.nn.Module):
    def __init__(self, dims, bias=False, act_after=()):
        super().__init__()
        self.layers = torch.nn.ModuleList(torch.nn.Linear(a, b, bias=bias) for a, b in zip(dims, dims[1:]))
        self.act_after = set(act_after)

    def forward(self, x):
        for i, layer in enumerate(self.layers):
            x = layer(x)
            if i in self.act_after:
                x = torch.relu(x)
        return x


class Weights(torch.nn.Module):
    def __init__(self, *shapes):
        super().__init__()
        for i, s in enumerate(shapes):
            self.register_buffer(f"w{i}", torch.randn(*s))


def names(chains):
    return [[g.node.name for g in c] for c in chains]


def test_linear_stack_is_one_chain():
    gm = fx.symbolic_trace(Mlp([64, 128, 64, 32]))
    chains = fusion.find_chains(gm)
    assert names(chains) == [["layers_0", "layers_1", "layers_2"]]
    assert all(g.linear is not None and g.right is None for g in chains[0])


def test_an_activation_splits_the_stack():
    gm = fx.symbolic_trace(Mlp([64, 128, 64, 32, 16], act_after=(0,)))
    assert names(fusion.find_chains(gm)) == [["layers_1", "layers_2", "layers_3"]]
    gm = fx.symbolic_trace(Mlp([64, 128, 64, 32, 16], act_after=(1,)))
    assert names(fusion.find_chains(gm)) == [["layers_0", "layers_1"], ["layers_2", "layers_3"]]


def test_bias_is_not_a_plain_gemm():
    gm = fx.symbolic_trace(Mlp([64, 64, 64], bias=True))
    assert fusion.find_chains(gm) == []


def test_matmul_chain_with_buffer_weights():
    class M(Weights):
        def forward(self, x):
            return torch.matmul(x @ self.w0, self.w1).matmul(self.w2)
    gm = fx.symbolic_trace(M((64, 32), (32, 16), (16, 8)))
    chains = fusion.find_chains(gm)
    assert len(chains) == 1 and len(chains[0]) == 3
    assert [g.right.op for g in chains[0]] == ["get_attr"] * 3


def test_an_intermediate_with_two_users_is_not_fused():
    class M(Weights):
        def forward(self, x):
            y = x @ self.w0
            return (y @ self.w1) + y.sum()
    gm = fx.symbolic_trace(M((8, 8), (8, 8)))
    assert fusion.find_chains(gm) == []


def test_a_conversion_between_gemms_breaks_the_chain():
    class T(Weights):
        def forward(self, x):
            return (x @ self.w0).transpose(-1, -2) @ self.w1

    class C(Weights):
        def forward(self, x):
            return (x @ self.w0).float() @ self.w1

    for cls in (T, C):
        gm = fx.symbolic_trace(cls((8, 8), (8, 8)))
        assert fusion.find_chains(gm) == []


def test_the_intermediate_must_be_the_left_operand():
    class M(Weights):
        def forward(self, x):
            return self.w1 @ (x @ self.w0)
    gm = fx.symbolic_trace(M((8, 8), (8, 8)))
    assert fusion.find_chains(gm) == []


def test_long_stacks_are_cut_at_eight():
    gm = fx.symbolic_trace(Mlp([16] * 12))
    chains = fusion.find_chains(gm)
    assert [len(c) for c in chains] == [8, 3]
    assert [len(c) for c in fusion.find_chains(gm, max_len=4)] == [4, 4, 3]


def test_fuse_rewrites_the_graph():
    torch.manual_seed(0)
    model = Mlp([64, 128, 64, 32, 16], act_after=(1,))
    gm = fx.symbolic_trace(model)
    gm, n = fusion.fuse_chains(gm)
    assert n == 2
    kinds = [(node.op, str(node.target)) for node in gm.graph.nodes]
    assert sum(1 for op, t in kinds if op == "call_module" and t.startswith("b2b_fused_chain")) == 2
    assert not any(op == "call_module" and t.startswith("layers") for op, t in kinds)
    # the relu between the two chains stays
    assert any(op == "call_function" and "relu" in t for op, t in kinds)
    # the fused module holds the transposed Linear weights
    mod = gm.get_submodule("b2b_fused_chain_0")
    assert torch.equal(mod.w0, model.layers[0].weight.t())


def test_fused_module_has_no_cpu_path():
    gm, n = fusion.fuse_chains(fx.symbolic_trace(Mlp([16, 16, 16])))
    assert n == 1
    with pytest.raises(RuntimeError, match="GPU only"):
        gm(torch.randn(4, 16))
