"""Row entropies and path log-probabilities (specdec_row_entropy,
specdec_path_logprob) against the float64 oracle, after linear and tree
verify calls, on the outputs the GPU emitted."""
import numpy as np
import pytest

from speculative_decoding_verification_64_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    from speculative_decoding_verification_64_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def close(got, want, atol, rtol):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    inf = np.isinf(want)
    assert np.array_equal(got[inf], want[inf])
    ok = ~nan & ~inf
    err = np.abs(got[ok] - want[ok])
    assert (err <= atol + rtol * np.abs(want[ok])).all(), float(err.max()) if err.size else 0.0


def linear_case(w, oracle_lib):
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    logits, q, toks, temp, uni = binding.linear_inputs_to_device(w)
    ws = binding.alloc_workspace(w.B, w.gamma + 1, w.V, binding.dtype_code(logits))
    out = binding.LinearOut.empty(w.B, w.gamma, "cuda")
    binding.row_stats(logits, temp, ws, q=q, draft_tokens=toks, entropy=True)
    binding.linear_finalize(logits, q, toks, temp, uni, out, ws)
    ref = binding.verify_linear(logits, q, toks, temp, uni)      # same outputs without the sums
    h = binding.row_entropy(logits, temp, ws)
    lp = binding.path_logprob(logits, temp, out.out_tokens, out.n_accepted, ws,
                              row_status=out.row_status)
    torch.cuda.synchronize()
    for k in ("n_accepted", "out_tokens", "final_token", "is_bonus", "row_status", "p_draft"):
        assert np.array_equal(getattr(out, k).cpu().numpy(), getattr(ref, k).cpu().numpy(),
                              equal_nan=(k == "p_draft")), k
    close(h.cpu().numpy(), oracle_lib.row_entropy(w.logits, w.dtype, w.temperature), 2e-4, 2e-5)
    want = oracle_lib.path_logprob(w.logits, w.dtype, w.temperature, out.out_tokens.cpu().numpy(),
                                   out.n_accepted.cpu().numpy(),
                                   row_status=out.row_status.cpu().numpy())
    close(lp.cpu().numpy(), want, 1e-3, 2e-5)
    # a verify call keeps no entropy sums: its workspace gives NaN entropies
    ws2 = binding.alloc_workspace(w.B, w.gamma + 1, w.V, binding.dtype_code(logits))
    binding.verify_linear(logits, q, toks, temp, uni, workspace=ws2)
    h2 = binding.row_entropy(logits, temp, ws2).cpu().numpy()
    greedy = (w.temperature == 0)
    assert np.isnan(h2[~greedy]).all()
    return h.cpu().numpy(), lp.cpu().numpy()


@pytest.mark.parametrize("name,B,V", [
    ("linear_b1_g4_v32000_f32", None, None),
    ("linear_b64_g5_v32000_bf16", 16, None),
    ("linear_b256_g8_v128256_bf16", 12, 20011),
    ("mixed_b512_g4_v152064_bf16", 40, 9001),    # greedy rows and temperatures 0.3 .. 1.5
])
def test_linear_entropy_and_logprob(oracle_lib, name, B, V):
    linear_case(W.make_workload(name, B=B, V=V), oracle_lib)


def test_masked_and_malformed_rows(oracle_lib):
    w = W.make_linear("normal2_tq08", B=8, gamma=3, V=777, dtype="f32", seed=31)
    w.logits[0, 1, :400] = -np.inf               # masked tokens: valid
    w.logits[1, 2, 5] = np.nan                   # malformed
    w.temperature[2] = 0.0                       # greedy
    w.temperature[3] = -2.0                      # invalid temperature
    w.draft_tokens[4, 0] = w.V                   # bad token
    h, lp = linear_case(w, oracle_lib)
    assert np.isnan(h[1, 2]) and np.isnan(h[3]).all() and (h[2] == 0).all()
    assert np.isnan(lp[[1, 3, 4]]).all() and np.isfinite(lp[[0, 2, 5]]).all()


def test_tree_entropy_and_logprob(oracle_lib):
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    w = W.make_workload("tree_b32_n64_v128256_bf16", B=8, V=10007)
    logits, q, toks, par, temp, uni = binding.tree_inputs_to_device(w)
    ws = binding.alloc_workspace(w.B, w.N, w.V, binding.dtype_code(logits))
    out = binding.TreeOut.empty(w.B, w.N, w.max_depth, "cuda")
    binding.row_stats(logits, temp, ws, entropy=True)
    binding.tree_finalize(logits, q, toks, par, temp, uni, w.max_depth, out, ws)
    h = binding.row_entropy(logits, temp, ws)
    lp = binding.path_logprob(logits, temp, out.out_tokens, out.n_accepted, ws,
                              path_nodes=out.path_nodes, row_status=out.row_status)
    torch.cuda.synchronize()
    close(h.cpu().numpy(), oracle_lib.row_entropy(w.logits, w.dtype, w.temperature), 2e-4, 2e-5)
    want = oracle_lib.path_logprob(w.logits, w.dtype, w.temperature, out.out_tokens.cpu().numpy(),
                                   out.n_accepted.cpu().numpy(),
                                   path_nodes=out.path_nodes.cpu().numpy(),
                                   row_status=out.row_status.cpu().numpy())
    close(lp.cpu().numpy(), want, 1e-3, 2e-5)
