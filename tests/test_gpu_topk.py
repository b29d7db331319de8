"""The top-k residual approximation (specdec_verify_linear_topk) against its
float64 oracle statement, and its distance from the exact step."""
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


def gpu_topk(w, topk):
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    x = binding.linear_inputs_to_device(w)
    dt = binding.dtype_code(x[0])
    ws = binding.alloc_workspace(w.B, w.gamma + 1, w.V, dt)
    out = binding.verify_linear_topk(*x, topk, workspace=ws)
    mass = binding.final_mass(ws, w.B, w.gamma + 1, w.V, dt)
    torch.cuda.synchronize()
    g = {k: getattr(out, k).cpu().numpy() for k in KEYS}
    g["final_mass"] = mass.cpu().numpy()
    return g


@pytest.mark.parametrize("name,B,V,topk", [
    ("linear_b256_g8_v128256_bf16", 32, 128256, 32),
    ("linear_b256_g8_v128256_bf16", 32, 128256, 1024),
    ("mixed_b512_g4_v152064_bf16", 48, 20011, 64),     # greedy rows, several temperatures
    ("linear_b64_g5_v32000_bf16", 24, None, 8),
    ("linear_b1_g4_v32000_f32", 24, None, 100),          # float32 keys: four radix passes
])
def test_topk_parity(oracle_lib, name, B, V, topk):
    w = W.make_workload(name, B=B, V=V)
    g = gpu_topk(w, topk)
    o = oracle_lib.verify_linear_topk_workload(w, topk)
    rep = compare_linear(w, g, o)
    tv = o["tv"][np.isfinite(o["tv"])]
    print(name, topk, rep, "mean TV %.3g max TV %.3g over %d corrections"
          % (tv.mean() if tv.size else 0, tv.max() if tv.size else 0, tv.size))


def test_topk_with_the_whole_vocabulary_is_the_exact_step(oracle_lib):
    w = W.make_workload("linear_b64_g5_v32000_bf16", B=16, V=700)
    g = gpu_topk(w, 1024)
    compare_linear(w, g, oracle_lib.verify_linear_workload(w))


def test_topk_ties_small_vocabularies_and_statuses(oracle_lib):
    w = W.make_linear("normal2_tq08", B=12, gamma=3, V=300, dtype="bf16", seed=41)
    w.logits[:, :, 10:40] = w.logits[0, 0, 7]      # ties among large logits
    w.logits[2, 1, 5] = 0x7FC0                     # NaN: malformed
    w.temperature[3] = 0.0                         # greedy
    for topk in (1, 5, 31, 300):
        g = gpu_topk(w, topk)
        compare_linear(w, g, oracle_lib.verify_linear_topk_workload(w, topk))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_topk_rows_without_a_usable_sample_threshold(oracle_lib, dtype):
    """Rows whose candidate count a sampled threshold cannot bound: constant rows
    (every key ties), and rows whose large logits sit on a regular comb of
    positions (a strided sample sees mostly them, so its estimate keeps too few
    candidates).  Both take the full radix select; results stay the oracle's."""
    V = 20011
    w = W.make_linear("normal2_tq08", B=10, gamma=3, V=V, dtype=dtype, seed=57)
    x = W.decode(w.logits, dtype)
    x[0:3] = 0.25                                   # constant rows: all ties
    comb = np.arange(V)[(np.arange(V) % 40) < 8]    # every fifth 16-byte vector of bf16
    rng = np.random.default_rng(5)
    x[3:7][:, :, comb] = 6.0 + rng.standard_normal((4, 4, comb.size))
    w.logits = W.encode(x, dtype)
    for topk in (7, 300, 1024):
        g = gpu_topk(w, topk)
        compare_linear(w, g, oracle_lib.verify_linear_topk_workload(w, topk))
