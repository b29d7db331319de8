"""Calls on several streams at once, each with its own workspace and outputs.

The library keeps no state between calls but per-device set-up, so verify
calls enqueued on different streams, free to overlap on the GPU, must give
exactly what each gives alone: the two-launch linear step (bulk-copy draw),
the one-launch small batch (a cluster of 16 or 8 CTAs), the chunked draw on
unaligned rows and the tree walk, interleaved call by call with no
synchronisation in between.  No kernel of the library waits on another
CTA outside its own cluster, so sharing the SMs with other grids can delay a
call but not stall it.
"""
import pytest

from speculative_decoding_verification_64_gb300 import workloads as W

pytestmark = pytest.mark.gpu

KEYS_LIN = ("n_accepted", "out_tokens", "final_token", "is_bonus", "row_status", "p_draft")
KEYS_TREE = ("n_accepted", "path_nodes", "out_tokens", "final_token", "is_bonus", "row_status",
             "p_node")
N_CALLS = 8


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    from speculative_decoding_verification_64_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def test_interleaved_calls_on_four_streams():
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    lin = [W.make_linear("zipf_t07", B=160, gamma=3, V=8192, dtype="bf16", seed=61),
           W.make_linear("normal2_q05", B=2, gamma=4, V=4096, dtype="f32", seed=62),
           W.make_linear("normal2_tq08", B=40, gamma=4, V=8191, dtype="bf16", seed=63)]
    tree = W.make_tree(B=4, N=16, V=5000, dtype="bf16", seed=64, max_depth=4)
    xl = [binding.linear_inputs_to_device(w) for w in lin]
    xt = binding.tree_inputs_to_device(tree)

    def run_linear(i, stream):
        w, x = lin[i], xl[i]
        ws = binding.alloc_workspace(w.B, w.gamma + 1, w.V, binding.dtype_code(x[0]))
        return binding.verify_linear(*x, workspace=ws, stream=stream)

    def run_tree(stream):
        ws = binding.alloc_workspace(tree.B, tree.N, tree.V, binding.dtype_code(xt[0]))
        return binding.verify_tree(*xt, tree.max_depth, workspace=ws, stream=stream)

    # each call alone, on the default stream
    ref_l = [run_linear(i, None) for i in range(len(lin))]
    ref_t = run_tree(None)
    torch.cuda.synchronize()
    # the same calls interleaved on four streams (workspaces and outputs
    # allocated up front on the default stream, so no allocation reuse races)
    streams = [torch.cuda.Stream() for _ in range(4)]
    torch.cuda.synchronize()
    outs_l = [[None] * N_CALLS for _ in lin]
    outs_t = [None] * N_CALLS
    wss_l = [[binding.alloc_workspace(w.B, w.gamma + 1, w.V, binding.dtype_code(x[0]))
              for _ in range(N_CALLS)] for w, x in zip(lin, xl)]
    wss_t = [binding.alloc_workspace(tree.B, tree.N, tree.V, binding.dtype_code(xt[0]))
             for _ in range(N_CALLS)]
    res_l = [[binding.LinearOut.empty(w.B, w.gamma, "cuda") for _ in range(N_CALLS)] for w in lin]
    res_t = [binding.TreeOut.empty(tree.B, tree.N, tree.max_depth, "cuda") for _ in range(N_CALLS)]
    torch.cuda.synchronize()
    for c in range(N_CALLS):
        for i in range(len(lin)):
            s = streams[i]
            with torch.cuda.stream(s):
                outs_l[i][c] = binding.verify_linear(*xl[i], out=res_l[i][c], workspace=wss_l[i][c],
                                                     stream=s)
        s = streams[3]
        with torch.cuda.stream(s):
            outs_t[c] = binding.verify_tree(*xt, tree.max_depth, out=res_t[c], workspace=wss_t[c],
                                            stream=s)
    torch.cuda.synchronize()
    for i in range(len(lin)):
        for c in range(N_CALLS):
            for k in KEYS_LIN:
                a, b = getattr(ref_l[i], k), getattr(outs_l[i][c], k)
                assert torch.equal(a, b) or (k == "p_draft" and torch.equal(a.isnan(), b.isnan())
                                             and torch.equal(a.nan_to_num(), b.nan_to_num())), (i, c, k)
    for c in range(N_CALLS):
        for k in KEYS_TREE:
            a, b = getattr(ref_t, k), getattr(outs_t[c], k)
            assert torch.equal(a, b) or (k == "p_node" and torch.equal(a.isnan(), b.isnan())
                                         and torch.equal(a.nan_to_num(), b.nan_to_num())), (c, k)
