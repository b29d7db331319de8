"""Per-position acceptance rates, sum_v min(p_i, q_i) of every drafted row
(specdec_row_alpha), against the float64 oracle."""
import numpy as np
import pytest

from speculative_decoding_verification_64_gb300 import workloads as W

pytestmark = pytest.mark.gpu

# float32 sums of up to ~V/256 terms per thread, a float32 reciprocal of S and
# ex2.approx (relative error ~2^-22) per element; alpha <= 1
ATOL = 2e-5


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    from speculative_decoding_verification_64_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def gpu_alpha(w, verify=True):
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    logits, q, toks, temp, uni = binding.linear_inputs_to_device(w)
    ws = binding.alloc_workspace(w.B, w.gamma + 1, w.V, binding.dtype_code(logits))
    if verify:  # the workspace of a whole verify call
        binding.verify_linear(logits, q, toks, temp, uni, workspace=ws)
    else:
        binding.row_stats(logits, temp, ws, q=q, draft_tokens=toks)
    a = binding.row_alpha(logits, q, temp, ws)
    torch.cuda.synchronize()
    return a.cpu().numpy()


def check(got, want):
    assert got.shape == want.shape
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    err = np.abs(got[~nan].astype(np.float64) - want[~nan])
    assert (err <= ATOL).all(), float(err.max())
    return float(err.max()) if err.size else 0.0


@pytest.mark.parametrize("name,B,V", [
    ("linear_b256_g8_v128256_bf16", None, None),        # the bench workload, full size
    ("mixed_b512_g4_v152064_bf16", 64, 20011),          # greedy rows, several temperatures, ragged V
    ("linear_b1_g4_v32000_f32", 8, None),
    ("linear_b64_g5_v32000_bf16", 16, 999),             # rows not 16-byte aligned
])
def test_alpha_parity(oracle_lib, name, B, V):
    w = W.make_workload(name, B=B, V=V)
    got = gpu_alpha(w)
    want = oracle_lib.row_alpha(w.logits, w.q, w.dtype, w.temperature)
    err = check(got, want)
    print(name, "max |alpha - oracle| %.2e, mean alpha %.3f" % (err, float(np.nanmean(want))))


def test_alpha_special_rows(oracle_lib):
    w = W.make_linear("normal2_tq08", B=6, gamma=3, V=257, dtype="bf16", seed=44)
    w.logits[1, 0, 9] = 0x7FC0            # NaN in a drafted row: unusable
    w.temperature[2] = 0.0                # greedy: min(1, q(argmax))
    w.temperature[3] = -1.0               # invalid temperature
    w.q[4, 1] = w.q[4, 1] * 0             # q row of zeros: alpha 0
    got = gpu_alpha(w, verify=False)
    want = oracle_lib.row_alpha(w.logits, w.q, w.dtype, w.temperature)
    check(got, want)
    assert np.isnan(got[1, 0]) and np.isnan(got[3]).all() and got[4, 1] == 0.0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V,gamma", [(1, 1), (2, 32), (7, 3), (4097, 32)])
def test_alpha_vocabulary_and_gamma_edges(oracle_lib, dtype, V, gamma):
    w = W.make_linear("normal2_tq08", B=5, gamma=gamma, V=V, dtype=dtype, seed=45 + V)
    w.temperature[1] = 0.0                # one greedy request
    got = gpu_alpha(w, verify=(V > 1))
    want = oracle_lib.row_alpha(w.logits, w.q, w.dtype, w.temperature)
    check(got, want)
