"""The no-allocation linear verify entry point against the workspace one.

specdec_verify_linear_static serves callers that cannot allocate device memory
for a workspace (a runtime that forbids allocation once it is running, or a
plug-in interface whose calls carry only inputs and outputs): its scratch is a
fixed array inside the library.  Its results must be those of
specdec_verify_linear with a caller workspace -- the same kernels on the same
data -- on calls in a row, whatever the previous call left in the array.
This file is collected last so that a run stopping at the first failure has
run every other test before it.
"""
import ctypes

import numpy as np
import pytest

from speculative_decoding_verification_64_gb300 import workloads as W

pytestmark = pytest.mark.gpu

P_TOL = {"f32": 2e-5, "bf16": 2e-3}   # the parity tolerance of the other GPU tests


@pytest.fixture(scope="module")
def lib():
    import torch
    from speculative_decoding_verification_64_gb300 import binding, build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return binding.load_library()


def _static(lib, w):
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    logits, q, toks, temp, uni = binding.linear_inputs_to_device(w)
    out = binding.LinearOut.empty(w.B, w.gamma, "cuda")
    P = ctypes.c_void_p
    rc = lib.specdec_verify_linear_static(
        P(logits.data_ptr()), P(q.data_ptr()), binding.dtype_code(logits), P(toks.data_ptr()),
        P(temp.data_ptr()), P(uni.data_ptr()), w.B, w.gamma, w.V,
        P(out.n_accepted.data_ptr()), P(out.out_tokens.data_ptr()), P(out.final_token.data_ptr()),
        P(out.is_bonus.data_ptr()), P(out.row_status.data_ptr()), P(out.p_draft.data_ptr()),
        P(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, binding.status_string(rc)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in vars(out).items()}


def _with_workspace(w):
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    out = binding.verify_linear(*binding.linear_inputs_to_device(w))
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in vars(out).items()}


def test_static_entry_point_matches_the_workspace_one(lib):
    from speculative_decoding_verification_64_gb300 import binding
    cases = [
        # the one-launch path of small batches (clusters of 16 and of 2 CTAs)
        (W.make_workload("linear_b1_g4_v32000_f32", B=2), binding.PATH_SMALL_ONE_LAUNCH),
        (W.make_workload("mixed_b512_g4_v152064_bf16", B=40, V=20000, seed_offset=7),
         binding.PATH_SMALL_ONE_LAUNCH),
        # the two launches: the chunked draw (odd V), the bulk-copy draw
        (W.make_workload("linear_b256_g8_v128256_bf16", B=48, V=30011), binding.PATH_TWO_LAUNCHES),
        (W.make_workload("mixed_b512_g4_v152064_bf16", B=100, V=20000, seed_offset=7),
         binding.PATH_TWO_LAUNCHES),
        # the benchmark's batch, whose scratch (1.2 MB) sits well inside the array
        (W.make_workload("linear_b256_g8_v128256_bf16"), binding.PATH_TWO_LAUNCHES),
    ]
    for w, path in cases:                 # calls in a row on the shared array
        x = binding.linear_inputs_to_device(w)
        assert binding.verify_linear_path(x[0], x[1]) == path, w.name
        assert lib.specdec_workspace_size(w.B, w.gamma + 1, w.V,
                                          binding.dtype_code(x[0])) <= (4 << 20)
        got = _static(lib, w)
        want = _with_workspace(w)
        for key in ("n_accepted", "out_tokens", "final_token", "is_bonus", "row_status"):
            assert np.array_equal(got[key], want[key]), (w.name, key)
        assert np.max(np.abs(got["p_draft"] - want["p_draft"])) <= P_TOL[w.dtype]
        assert (got["row_status"] == 0).all() and got["n_accepted"].max() <= w.gamma


def test_static_entry_point_rejects_sizes_beyond_its_array(lib):
    from speculative_decoding_verification_64_gb300 import binding
    N = None
    cap = lib.specdec_workspace_size(4096, 9, 128256, binding.BF16)
    assert cap > (4 << 20)
    # refused before any launch (all pointers null would otherwise be invalid)
    rc = lib.specdec_verify_linear_static(N, N, binding.BF16, N, N, N, 4096, 8, 128256,
                                          N, N, N, N, N, N, N)
    assert rc == 5
    assert "fixed array" in binding.status_string(rc)
