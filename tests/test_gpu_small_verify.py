"""The one-launch path of specdec_verify_linear for small batches (one cluster
of 16, 8, 4 or 2 CTAs per request, rows held in shared memory; the q rows too
when they fit, else q row k copied in after the decision) against the
two-kernel path (specdec_row_stats, then specdec_linear_finalize) and the
oracle: outputs, p_draft and the workspace's stage partials bit for bit.

The cluster size is the largest of which the device holds all B clusters at
once: on a GB300 the smallest batches below take clusters of 16, the others
clusters of 8, 4 or 2 as B grows; the q rows are resident except in the cases
marked "q row k after the decision"."""
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
    ws1 = binding.alloc_workspace(w.B, R, w.V, binding.dtype_code(logits))
    ws2 = binding.alloc_workspace(w.B, R, w.V, binding.dtype_code(logits))
    assert binding.verify_linear_launches(logits, q) == 1
    one = binding.verify_linear(*x, workspace=ws1)
    two = binding.LinearOut.empty(w.B, w.gamma, "cuda")
    binding.row_stats(logits, temp, ws2, q=q, draft_tokens=toks)
    binding.linear_finalize(logits, q, toks, temp, uni, two, ws2)
    torch.cuda.synchronize()
    g1 = {k: getattr(one, k).cpu().numpy() for k in KEYS}
    g2 = {k: getattr(two, k).cpu().numpy() for k in KEYS}
    for k in KEYS:
        assert np.array_equal(g1[k], g2[k], equal_nan=(k == "p_draft")), k
    # the stage partials (16 bytes per row and 8 KB stage) at the workspace's start
    es = 4 if w.dtype == "f32" else 2
    spr = -(-w.V * es // 8192)
    nb = w.B * R * spr * 16
    assert torch.equal(ws1[:nb], ws2[:nb])
    return g1


@pytest.mark.parametrize("name,B,V,gamma", [
    ("linear_b1_g4_v32000_f32", 1, None, None),       # the B = 1 workload itself
    ("linear_b256_g8_v128256_bf16", 1, None, None),   # one request of the benchmark's rows
    ("linear_b1_g4_v32000_f32", 8, 20000, None),
    ("linear_b64_g5_v32000_bf16", 19, None, None),    # the largest batch of one wave
    ("linear_b64_g5_v32000_bf16", 3, 4104, None),     # a last stage of 16 bytes
    ("mixed_b512_g4_v152064_bf16", 12, 30000, None),  # greedy rows, several temperatures
    ("linear_b64_g5_v32000_bf16", 24, None, None),    # clusters of 4
    ("linear_b64_g5_v32000_bf16", 64, None, None),    # the B = 64 workload: q row k after the decision
    ("mixed_b512_g4_v152064_bf16", 40, 30000, None),  # greedy rows; q row k after the decision
    ("linear_b1_g4_v32000_f32", 50, 16000, None),     # float32; q row k after the decision
])
def test_one_launch_equals_two_and_the_oracle(oracle_lib, name, B, V, gamma):
    w = W.make_workload(name, B=B, V=V)
    g = both_paths(w)
    compare_linear(w, g, oracle_lib.verify_linear_workload(w))


@pytest.mark.parametrize("B,gamma,V,dtype", [(4, 1, 8, "f32"), (4, 8, 64, "bf16"),
                                             (4, 12, 2048, "f32"), (4, 5, 12288, "bf16"),
                                             (40, 4, 32768, "bf16")])  # q row k after the decision
def test_one_launch_edges(oracle_lib, B, gamma, V, dtype):
    w = W.make_linear("normal2_tq08", B=B, gamma=gamma, V=V, dtype=dtype, seed=60 + gamma)
    w.temperature[1] = 0.0                       # greedy
    w.draft_tokens[2, 0] = V                     # a token out of range: malformed
    g = both_paths(w)
    compare_linear(w, g, oracle_lib.verify_linear_workload(w))
