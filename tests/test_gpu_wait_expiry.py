"""Bounded waits that give up: the give-up paths of the kernels that wait on bulk copies.

Every wait of a kernel on a bulk copy is bounded.  When a consumer's wait gives
up, the kernel marks what it could not read (the stage partials, or the
request's draw) SPECDEC_ROW_INTERNAL, keeps the CTA until every copy it issued
has landed (those waits keep their full limit), and returns.  The "shortwait"
test build of the library makes the consumers' waits give up without looking,
every time, while the copies they would have read are still issued: every
request of a call must come back with SPECDEC_ROW_INTERNAL and the
malformed-request outputs, and the call must return 0.  The device must stay
usable: the regular library then verifies the same inputs in agreement with
the oracle.  No wait is left unbounded and no copy can land in a CTA that has
left, so a give-up cannot fault the GPU.
"""
import contextlib

import numpy as np
import pytest

from parity import compare_linear, compare_tree, gpu_linear, gpu_tree
from speculative_decoding_verification_64_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def shortwait():
    import torch
    from speculative_decoding_verification_64_gb300 import binding, build
    build.build()
    path = build.build(variant="shortwait")
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return binding.load_library(path)


@contextlib.contextmanager
def using(lib):
    from speculative_decoding_verification_64_gb300 import binding
    saved = binding.load_library()
    binding._lib = lib
    try:
        yield
    finally:
        binding._lib = saved


def _all_internal(g):
    from speculative_decoding_verification_64_gb300.binding import ROW_INTERNAL
    assert (g["row_status"] & ROW_INTERNAL).all(), g["row_status"]
    assert (g["n_accepted"] == 0).all() and (g["final_token"] == -1).all()
    assert (g["out_tokens"] == -1).all() and (g["is_bonus"] == 0).all()


LINEAR = [
    # (workload, the path the call takes)
    (lambda: W.make_workload("linear_b256_g8_v128256_bf16", B=64), "two launches, bulk-copy draw"),
    (lambda: W.make_linear("normal2_tq08", B=16, gamma=4, V=20003, dtype="bf16", seed=3),
     "two launches, chunked draw"),
    (lambda: W.make_workload("linear_b1_g4_v32000_f32", B=2), "one launch, clusters of 16"),
    (lambda: W.make_workload("linear_b1_g4_v32000_f32", B=12), "one launch, clusters of 8"),
    (lambda: W.make_workload("linear_b64_g5_v32000_bf16"), "one launch, clusters of 2"),
]


@pytest.mark.parametrize("case", range(len(LINEAR)), ids=[c[1] for c in LINEAR])
def test_linear_waits_give_up(shortwait, oracle_lib, case):
    # the stats pass's (or the one-launch kernel's) consumers give up
    w = LINEAR[case][0]()
    with using(shortwait):
        g = gpu_linear(w)
    _all_internal(g)
    g = gpu_linear(w)  # the context is intact: the regular library on the same inputs
    compare_linear(w, g, oracle_lib.verify_linear_workload(w))
    assert (g["row_status"] == 0).all()


def test_draw_waits_give_up(shortwait, oracle_lib):
    # a regular stats pass, then the bulk-copy draw of the test build on its
    # workspace: the draw's consumers give up, every request's search reports
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    w = W.make_workload("linear_b256_g8_v128256_bf16", B=64)
    x = binding.linear_inputs_to_device(w)
    ws = binding.alloc_workspace(w.B, w.gamma + 1, w.V, binding.dtype_code(x[0]))
    binding.row_stats(x[0], x[3], ws, q=x[1], draft_tokens=x[2])
    out = binding.LinearOut.empty(w.B, w.gamma, "cuda")
    with using(shortwait):
        binding.linear_finalize(*x, out, ws)
    torch.cuda.synchronize()
    g = {k: (None if v is None else v.cpu().numpy()) for k, v in vars(out).items()}
    _all_internal(g)
    # the same workspace, the regular draw: the step's own outputs
    binding.linear_finalize(*x, out, ws)
    torch.cuda.synchronize()
    g = {k: (None if v is None else v.cpu().numpy()) for k, v in vars(out).items()}
    g["final_mass"] = binding.final_mass(ws, w.B, w.gamma + 1, w.V, binding.dtype_code(x[0])).cpu().numpy()
    compare_linear(w, g, oracle_lib.verify_linear_workload(w))
    assert (g["row_status"] == 0).all()


def test_tree_waits_give_up(shortwait, oracle_lib):
    w = W.make_tree(B=6, N=16, V=20000, dtype="bf16", seed=5, max_depth=4)
    with using(shortwait):
        g = gpu_tree(w)
    _all_internal(g)
    g = gpu_tree(w)
    compare_tree(w, g, oracle_lib.verify_tree_workload(w))
    assert (g["row_status"] == 0).all()
