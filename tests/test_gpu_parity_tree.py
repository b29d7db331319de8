"""Token-tree verify: CUDA path (through the C ABI) against the float64 oracle."""
import numpy as np
import pytest

from parity import compare_tree, gpu_linear, gpu_tree
from speculative_decoding_verification_64_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    from speculative_decoding_verification_64_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def run(w, oracle_lib, **kw):
    g = gpu_tree(w, **kw)
    o = oracle_lib.verify_tree_workload(w)
    rep = compare_tree(w, g, o)
    print(w.name, rep)
    return g, o, rep


# Small cases: unaligned and aligned rows; V = 8 and 12 leave seven of the
# eight CTA slices empty; float32 rows take two tiles a load batch.
@pytest.mark.parametrize("dtype,V", [("bf16", 10007), ("f32", 4099), ("bf16", 10008),
                                     ("f32", 4100), ("bf16", 8), ("f32", 12)])
def test_tree_parity_small(oracle_lib, dtype, V):
    w = W.make_tree(B=12, N=64, V=V, dtype=dtype, seed=3)
    g, o, rep = run(w, oracle_lib)


def test_tree_many_nodes_large_vocabulary(oracle_lib):
    # 1024 nodes over an 80000-token vocabulary: three tiles a CTA slice (one
    # partial), deep walks
    w = W.make_tree(B=3, N=1024, V=80000, dtype="bf16", seed=9, max_depth=12, branching=3)
    run(w, oracle_lib)


def test_tree_aligned_and_unaligned_rows_agree():
    # one stats pass, then the walk twice on it: on the aligned rows (vector
    # loads) and on copies of them one element off a 16-byte boundary
    # (element loads): identical results
    import torch
    from parity import _offset_copy
    from speculative_decoding_verification_64_gb300 import binding
    w = W.make_tree(B=24, N=64, V=20000, dtype="bf16", seed=8)
    logits, q, toks, par, temp, uni = binding.tree_inputs_to_device(w)
    dt = binding.dtype_code(logits)
    ws = binding.alloc_workspace(w.B, w.N, w.V, dt)
    binding.row_stats(logits, temp, ws)
    res = []
    for lg, qq in ((logits, q), (_offset_copy(logits, 1), _offset_copy(q, 1))):
        out = binding.TreeOut.empty(w.B, w.N, w.max_depth, "cuda")
        binding.tree_finalize(lg, qq, toks, par, temp, uni, w.max_depth, out, ws)
        mass = binding.final_mass(ws, w.B, w.N, w.V, dt)
        torch.cuda.synchronize()
        r = {k: v.cpu().numpy() for k, v in vars(out).items() if v is not None}
        r["final_mass"] = mass.cpu().numpy()
        res.append(r)
    assert (res[0]["row_status"] == 0).all()
    for key in ("n_accepted", "path_nodes", "out_tokens", "final_token", "is_bonus",
                "row_status", "p_node", "final_mass"):
        assert np.array_equal(res[0][key], res[1][key]), key


def test_tree_full_size(oracle_lib):
    w = W.make_workload("tree_b32_n64_v128256_bf16")
    g, o, rep = run(w, oracle_lib)
    assert g["n_accepted"].max() >= 1


def test_tree_duplicate_siblings_small_vocab(oracle_lib):
    # V = 5: siblings drawn i.i.d. from q repeat tokens often
    w = W.make_tree(B=200, N=40, V=5, dtype="f32", seed=11, max_depth=4)
    g, o, rep = run(w, oracle_lib)


def test_tree_root_only_is_a_bonus_draw(oracle_lib):
    w = W.make_tree(B=9, N=1, V=3000, dtype="bf16", seed=2, max_depth=0)
    g, o, rep = run(w, oracle_lib)
    assert (g["is_bonus"] == 1).all() and (g["n_accepted"] == 0).all()


def test_tree_many_nodes(oracle_lib):
    w = W.make_tree(B=4, N=1024, V=2003, dtype="bf16", seed=6, max_depth=12, branching=3)
    run(w, oracle_lib)


def test_tree_greedy_with_ties(oracle_lib):
    w = W.make_tree(B=40, N=30, V=200, dtype="f32", seed=7, max_depth=4)
    rng = np.random.default_rng(1)
    lg = rng.integers(-3, 3, size=w.logits.shape).astype(np.float32)
    w.logits = lg
    amax = lg.argmax(-1)
    for b in range(w.B):
        for n in range(1, w.N):
            if rng.random() < 0.5:
                w.node_tokens[b, n] = amax[b, w.parent[b, n]]
    w.temperature[:] = 0.0
    run(w, oracle_lib)


def test_tree_malformed(oracle_lib):
    w = W.make_tree(B=6, N=16, V=300, dtype="f32", seed=4, max_depth=3)
    w.parent[1, 0] = 0
    w.parent[2, 7] = 9
    w.node_tokens[3, 4] = 300
    w.logits[4, 15, 2] = np.inf
    w.temperature[5] = -2.0
    g, o, rep = run(w, oracle_lib)
    assert (g["row_status"][1:6] != 0).all() and g["row_status"][0] == 0


def test_chain_tree_matches_linear_on_gpu():
    w = W.make_linear("normal2_tq08", B=40, gamma=5, V=6007, dtype="bf16", seed=21)
    B, g, V = w.B, w.gamma, w.V
    N = g + 1
    q = np.zeros((B, N, V), dtype=w.q.dtype)
    q[:, :g] = w.q
    q[:, g] = w.q[:, g - 1]
    toks = np.zeros((B, N), np.int32)
    toks[:, 1:] = w.draft_tokens
    uni = np.empty((B, N), np.float32)
    uni[:, 1:] = w.uniforms[:, :g]
    uni[:, 0] = w.uniforms[:, g]
    t = W.TreeWorkload("chain", w.dtype, B, N, V, g, w.logits, q, toks,
                       np.tile(np.arange(-1, N - 1, dtype=np.int32), (B, 1)),
                       w.temperature, uni)
    lin = gpu_linear(w)
    tr = gpu_tree(t)
    for key in ("n_accepted", "final_token", "is_bonus", "row_status", "out_tokens"):
        assert np.array_equal(lin[key], tr[key]), key
