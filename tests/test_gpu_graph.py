"""The verify calls captured in a CUDA graph and replayed with new inputs give
the eager results (the library allocates nothing and its launches read only
their arguments, so a captured step is a reusable step)."""
import numpy as np
import pytest

from speculative_decoding_verification_64_gb300 import workloads as W

pytestmark = pytest.mark.gpu

LIN = ("n_accepted", "out_tokens", "final_token", "is_bonus", "row_status", "p_draft")
TREE = ("n_accepted", "path_nodes", "out_tokens", "final_token", "is_bonus", "row_status", "p_node")


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    from speculative_decoding_verification_64_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def same(a, b, keys):
    for k in keys:
        x, y = getattr(a, k), getattr(b, k)
        if x is None:
            continue
        assert np.array_equal(x.cpu().numpy(), y.cpu().numpy(), equal_nan=True), k


@pytest.mark.parametrize("name,B,V", [("linear_b1_g4_v32000_f32", None, None),
                                      ("linear_b64_g5_v32000_bf16", 24, None),
                                      ("mixed_b512_g4_v152064_bf16", 32, 12347)])
def test_linear_graph_replay(name, B, V):
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    cases = [W.make_workload(name, B=B, V=V, seed_offset=i) for i in range(3)]
    static = [t.clone() for t in binding.linear_inputs_to_device(cases[0])]
    ws = binding.alloc_workspace(cases[0].B, cases[0].gamma + 1, cases[0].V,
                                 binding.dtype_code(static[0]))
    out = binding.LinearOut.empty(cases[0].B, cases[0].gamma, "cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):       # warm-up outside capture (first-call set-up)
        binding.verify_linear(*static, out=out, workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        binding.verify_linear(*static, out=out, workspace=ws)
    for w in cases[1:] + cases[:1]:
        for dst, src in zip(static, binding.linear_inputs_to_device(w)):
            dst.copy_(src)
        g.replay()
        eager = binding.verify_linear(*binding.linear_inputs_to_device(w))
        torch.cuda.synchronize()
        same(out, eager, LIN)


def test_tree_graph_replay():
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    cases = [W.make_workload("tree_b32_n64_v128256_bf16", B=6, V=8011, seed_offset=i)
             for i in range(3)]
    w0 = cases[0]
    static = [t.clone() for t in binding.tree_inputs_to_device(w0)]
    ws = binding.alloc_workspace(w0.B, w0.N, w0.V, binding.dtype_code(static[0]))
    out = binding.TreeOut.empty(w0.B, w0.N, w0.max_depth, "cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        binding.verify_tree(*static, w0.max_depth, out=out, workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        binding.verify_tree(*static, w0.max_depth, out=out, workspace=ws)
    for w in cases[1:] + cases[:1]:
        for dst, src in zip(static, binding.tree_inputs_to_device(w)):
            dst.copy_(src)
        g.replay()
        eager = binding.verify_tree(*binding.tree_inputs_to_device(w), w.max_depth)
        torch.cuda.synchronize()
        same(out, eager, TREE)
