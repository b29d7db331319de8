"""The one-launch path of specdec_verify_linear for large batches (one
cooperative launch: the stats pass, a grid barrier, the decisions, then the
draw dealt round robin over the CTAs) against the two-kernel path
(specdec_row_stats, then specdec_linear_finalize) and the oracle: outputs,
p_draft, the draw normaliser and the workspace's stage partials bit for bit;
and its replay from a CUDA graph."""
import numpy as np
import pytest

from parity import compare_linear
from speculative_decoding_verification_64_gb300 import workloads as W

pytestmark = pytest.mark.gpu

KEYS = ("n_accepted", "out_tokens", "final_token", "is_bonus", "row_status", "p_draft")


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    from speculative_decoding_verification_64_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def both_paths(w):
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    x = binding.linear_inputs_to_device(w)
    logits, q, toks, temp, uni = x
    R = w.gamma + 1
    dt = binding.dtype_code(logits)
    ws1 = binding.alloc_workspace(w.B, R, w.V, dt)
    ws2 = binding.alloc_workspace(w.B, R, w.V, dt)
    ws1.fill_(0x5A)                       # no initialisation needed by either path
    assert binding.verify_linear_path(logits, q) == binding.PATH_LARGE_ONE_LAUNCH
    one = binding.verify_linear(*x, workspace=ws1)
    m1 = binding.final_mass(ws1, w.B, R, w.V, dt)
    two = binding.LinearOut.empty(w.B, w.gamma, "cuda")
    binding.row_stats(logits, temp, ws2, q=q, draft_tokens=toks)
    binding.linear_finalize(logits, q, toks, temp, uni, two, ws2)
    m2 = binding.final_mass(ws2, w.B, R, w.V, dt)
    torch.cuda.synchronize()
    g1 = {k: getattr(one, k).cpu().numpy() for k in KEYS}
    g2 = {k: getattr(two, k).cpu().numpy() for k in KEYS}
    for k in KEYS:
        assert np.array_equal(g1[k], g2[k], equal_nan=(k == "p_draft")), k
    assert np.array_equal(m1.cpu().numpy(), m2.cpu().numpy(), equal_nan=True)
    # the stage partials (16 bytes per row and 8 KB stage) at the workspace's start
    es = 4 if w.dtype == "f32" else 2
    spr = -(-w.V * es // 8192)
    nb = w.B * R * spr * 16
    assert torch.equal(ws1[:nb], ws2[:nb])
    g1["final_mass"] = m1.cpu().numpy()
    return g1


@pytest.mark.parametrize("name,B,V", [
    ("linear_b256_g8_v128256_bf16", None, None),     # the benchmark workload itself
    ("mixed_b512_g4_v152064_bf16", None, None),      # greedy rows, several temperatures
    ("linear_b256_g8_v128256_bf16", 100, 65536),     # fewer requests than SMs
    ("linear_b1_g4_v32000_f32", 600, 20000),         # float32 rows, 4 requests per CTA
])
def test_cooperative_launch_equals_two_and_the_oracle(oracle_lib, name, B, V):
    w = W.make_workload(name, B=B, V=V)
    g = both_paths(w)
    rep = compare_linear(w, g, oracle_lib.verify_linear_workload(w))
    print(w.name, rep)


def test_cooperative_launch_edges(oracle_lib):
    w = W.make_linear("normal2_tq08", B=160, gamma=6, V=24576, dtype="bf16", seed=71)
    w.temperature[[1, 50]] = 0.0                 # greedy
    w.draft_tokens[2, 0] = w.V                   # a token out of range: malformed
    w.temperature[3] = float("nan")              # a bad temperature: malformed
    g = both_paths(w)
    compare_linear(w, g, oracle_lib.verify_linear_workload(w))


def test_cooperative_launch_graph_replay():
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    cases = [W.make_workload("mixed_b512_g4_v152064_bf16", B=200, V=40000, seed_offset=i)
             for i in range(3)]
    static = [t.clone() for t in binding.linear_inputs_to_device(cases[0])]
    assert binding.verify_linear_path(static[0], static[1]) == binding.PATH_LARGE_ONE_LAUNCH
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
        for k in KEYS:
            assert np.array_equal(getattr(out, k).cpu().numpy(), getattr(eager, k).cpu().numpy(),
                                  equal_nan=True), k
