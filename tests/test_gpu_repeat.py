"""Back-to-back verify calls with no synchronisation between them, as a
serving loop (and the benchmark) issues them: every call must produce
bit-identical outputs.  A race in a kernel's handshakes (rings of shared
memory slots, tickets, programmatically dependent launches) shows up here
as a call that differs from the others."""
import numpy as np
import pytest

from speculative_decoding_verification_64_gb300 import workloads as W

pytestmark = pytest.mark.gpu

N_CALLS = 200


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    from speculative_decoding_verification_64_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def snapshot(out):
    return {k: v.clone() for k, v in vars(out).items() if v is not None}


def check_same(outs):
    first = outs[0]
    for i, o in enumerate(outs[1:], 1):
        for k, v in first.items():
            a, b = v.cpu().numpy(), o[k].cpu().numpy()
            assert np.array_equal(a, b, equal_nan=True), (i, k)


@pytest.mark.parametrize("V", [128256, 128255])   # the bulk-copy draw; the chunked draw
def test_linear_calls_repeat_exactly(V):
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    w = W.make_workload("linear_b256_g8_v128256_bf16", V=V)
    x = binding.linear_inputs_to_device(w)
    assert binding.verify_linear_path(x[0], x[1]) == binding.PATH_TWO_LAUNCHES
    ws = binding.alloc_workspace(w.B, w.gamma + 1, w.V, binding.dtype_code(x[0]))
    outs = [binding.LinearOut.empty(w.B, w.gamma, "cuda") for _ in range(N_CALLS)]
    for o in outs:
        binding.verify_linear(*x, out=o, workspace=ws)
    torch.cuda.synchronize()
    check_same([snapshot(o) for o in outs])


def test_one_launch_calls_repeat_exactly():
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    w = W.make_workload("linear_b1_g4_v32000_f32", B=8)
    x = binding.linear_inputs_to_device(w)
    assert binding.verify_linear_launches(x[0], x[1]) == 1
    ws = binding.alloc_workspace(w.B, w.gamma + 1, w.V, binding.dtype_code(x[0]))
    outs = [binding.LinearOut.empty(w.B, w.gamma, "cuda") for _ in range(N_CALLS)]
    for o in outs:
        binding.verify_linear(*x, out=o, workspace=ws)
    torch.cuda.synchronize()
    check_same([snapshot(o) for o in outs])


def test_topk_calls_repeat_exactly():
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    w = W.make_workload("linear_b256_g8_v128256_bf16")
    x = binding.linear_inputs_to_device(w)
    ws = binding.alloc_workspace(w.B, w.gamma + 1, w.V, binding.dtype_code(x[0]))
    outs = [binding.LinearOut.empty(w.B, w.gamma, "cuda") for _ in range(N_CALLS // 4)]
    for o in outs:
        binding.verify_linear_topk(*x, 64, out=o, workspace=ws)
    torch.cuda.synchronize()
    check_same([snapshot(o) for o in outs])


def test_tree_calls_repeat_exactly():
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    w = W.make_workload("tree_b32_n64_v128256_bf16")
    x = binding.tree_inputs_to_device(w)
    ws = binding.alloc_workspace(w.B, w.N, w.V, binding.dtype_code(x[0]))
    outs = [binding.TreeOut.empty(w.B, w.N, w.max_depth, "cuda") for _ in range(N_CALLS // 2)]
    for o in outs:
        binding.verify_tree(*x, w.max_depth, out=o, workspace=ws)
    torch.cuda.synchronize()
    check_same([snapshot(o) for o in outs])
