"""Linear verify: CUDA path (through the C ABI) against the float64 oracle.

Tolerances and the boundary-draw rule are in ``parity.py``.
"""
import dataclasses

import numpy as np
import pytest

from parity import compare_linear, gpu_linear
from speculative_decoding_verification_64_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    from speculative_decoding_verification_64_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def run(w, oracle_lib, **kw):
    g = gpu_linear(w, **kw)
    o = oracle_lib.verify_linear_workload(w)
    rep = compare_linear(w, g, o)
    print(w.name, rep)
    return g, o, rep


# --- the four linear workloads: smaller cases spanning several tiles and a ragged tail


@pytest.mark.parametrize("name,B,V", [
    ("linear_b1_g4_v32000_f32", None, None),          # full size
    ("linear_b64_g5_v32000_bf16", None, None),        # full size
    ("linear_b256_g8_v128256_bf16", 24, 20011),
    ("mixed_b512_g4_v152064_bf16", 64, 12347),
])
def test_workload_parity(oracle_lib, name, B, V):
    w = W.make_workload(name, B=B, V=V)
    g, o, rep = run(w, oracle_lib)
    assert 0 <= g["n_accepted"].min() and g["n_accepted"].max() <= w.gamma


# --- full sizes, in the launch configuration the benchmark times


@pytest.mark.parametrize("name", ["linear_b256_g8_v128256_bf16", "mixed_b512_g4_v152064_bf16"])
def test_full_size_parity(oracle_lib, name):
    w = W.make_workload(name)
    g, o, rep = run(w, oracle_lib)
    assert rep["B"] == w.B
    # the statistic the workload is built for: some but not all drafts accepted
    assert 0 < g["n_accepted"].mean() < w.gamma


# --- vocabulary and batch edges


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [1, 2, 7, 8, 9, 1000, 4095, 4097, 32769, 65537])
def test_vocabulary_edges(oracle_lib, dtype, V):
    w = W.make_linear("normal2_tq08", B=6, gamma=3, V=V, dtype=dtype, seed=V)
    run(w, oracle_lib)


@pytest.mark.parametrize("gamma", [1, 2, 31, 32])
def test_gamma_edges(oracle_lib, gamma):
    w = W.make_linear("normal2_tq08", B=5, gamma=gamma, V=3001, dtype="bf16", seed=gamma)
    run(w, oracle_lib)


@pytest.mark.parametrize("offset", [1, 3, 5])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_unaligned_base_pointers(oracle_lib, offset, dtype):
    w = W.make_linear("normal2_tq08", B=7, gamma=4, V=20003, dtype=dtype, seed=offset)
    run(w, oracle_lib, offset_elems=offset)


def test_unaligned_rows_of_many_requests(oracle_lib):
    # odd V (rows off 16-byte boundaries) and runs of more than 8 requests per
    # CTA: the chunked draw with shifted vector loads
    w = W.make_linear("normal2_tq08", B=1200, gamma=4, V=20003, dtype="bf16", seed=31)
    run(w, oracle_lib)


@pytest.mark.parametrize("V,offset", [(128255, 0), (128256, 1), (32001, 7)])
def test_unaligned_rows_benchmark_vocabulary(oracle_lib, V, offset):
    # rows off 16-byte boundaries at the benchmark's vocabulary (odd V or an
    # offset base): the stats pass's plain edge loads and the chunked draw's
    # shifted vectors, the row's last vector partial when V is odd
    w = W.make_linear("zipf_t07", B=24, gamma=8, V=V, dtype="bf16", seed=V + offset)
    run(w, oracle_lib, offset_elems=offset)


def test_batch_zero_is_a_noop():
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    d = "cuda"
    out = binding.verify_linear(torch.empty(0, 3, 10, device=d), torch.empty(0, 2, 10, device=d),
                                torch.empty(0, 2, dtype=torch.int32, device=d),
                                torch.empty(0, device=d), torch.empty(0, 3, device=d))
    assert out.n_accepted.numel() == 0


# --- behaviour cases


def test_greedy_rows_with_ties(oracle_lib):
    w = W.make_linear("normal2_tq08", B=64, gamma=4, V=1000, dtype="bf16", seed=5)
    rng = np.random.default_rng(5)
    lg = rng.integers(-4, 4, size=(w.B, w.gamma + 1, w.V)).astype(np.float32)
    w.logits = W.encode(lg, "bf16")
    amax = lg.argmax(-1)
    w.draft_tokens = np.where(rng.random((w.B, w.gamma)) < 0.7, amax[:, :w.gamma],
                              w.draft_tokens).astype(np.int32)
    w.temperature[:] = 0.0
    w.temperature[::3] = 0.8                      # mixed batch
    g, o, rep = run(w, oracle_lib)
    greedy = w.temperature == 0
    assert np.array_equal(g["final_token"][greedy], o["final_token"][greedy])


@pytest.mark.parametrize("pattern", ["all", "first_half", "last_half", "every_third", "invalid"])
def test_requests_that_draw_nothing(oracle_lib, pattern):
    """Greedy requests and requests with an invalid temperature draw nothing:
    the bulk-copy draw (aligned bf16 rows, B = 300) streams no unit of theirs,
    wherever they sit in the CTAs' runs, all of them included."""
    w = W.make_linear("normal2_tq08", B=300, gamma=4, V=32000, dtype="bf16", seed=17)
    B = w.B
    idx = {"all": np.arange(B), "first_half": np.arange(B // 2),
           "last_half": np.arange(B // 2, B), "every_third": np.arange(0, B, 3),
           "invalid": np.arange(0, B, 7)}[pattern]
    w.temperature[idx] = 0.0
    if pattern == "invalid":
        bad = np.arange(3, B, 11)
        w.temperature[bad] = np.array([-1.0, np.nan, 2.0 ** 21])[np.arange(bad.size) % 3]
    g, o, rep = run(w, oracle_lib)
    greedy = w.temperature == 0
    assert np.array_equal(g["final_token"][greedy], o["final_token"][greedy])
    if pattern == "invalid":
        assert (g["row_status"][bad] == 8).all()


def test_all_accepted_when_q_equals_p(oracle_lib):
    w = W.make_linear("normal2_q05", B=32, gamma=6, V=5000, dtype="f32", seed=8)
    l = w.logits[:, :w.gamma].astype(np.float64)
    p = np.exp(l - l.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    w.q = p.astype(np.float32)
    g, o, rep = run(w, oracle_lib)
    assert (g["n_accepted"] >= w.gamma - 1).mean() > 0.9


def test_first_position_rejects(oracle_lib):
    w = W.make_linear("normal2_tq08", B=32, gamma=4, V=4000, dtype="bf16", seed=9)
    lg = W.decode(w.logits, "bf16")
    worst = lg[:, 0].argmin(-1)                   # the least likely target token
    q = W.decode(w.q, "bf16")
    q[np.arange(w.B), 0] = 0.0
    q[np.arange(w.B), 0, worst] = 1.0
    w.q = W.encode(q, "bf16")
    w.draft_tokens[:, 0] = worst
    g, o, rep = run(w, oracle_lib)
    assert (g["n_accepted"] == 0).all()


def test_malformed_requests_report_status(oracle_lib):
    w = W.make_linear("normal2_tq08", B=10, gamma=3, V=777, dtype="f32", seed=2)
    w.logits[1, 2, 5] = np.nan
    w.logits[2, 0, 3] = np.inf
    w.logits[3, 1, :] = -np.inf
    w.draft_tokens[4, 1] = w.V
    w.draft_tokens[5, 0] = -3
    w.q[6, 0, w.draft_tokens[6, 0]] = 0.0
    w.temperature[7] = -1.0
    w.temperature[8] = np.nan
    w.logits[9, 0, :100] = -np.inf                # partially masked row: valid
    g, o, rep = run(w, oracle_lib)
    assert list(g["row_status"][:9]) == [0, 4, 4, 4, 1, 1, 2, 8, 8]
    assert g["row_status"][9] == 0


def test_input_domain_edges(oracle_lib):
    w = W.make_linear("normal2_tq08", B=8, gamma=2, V=3001, dtype="f32", seed=12)
    w.temperature[0] = 2.0 ** -20
    w.temperature[1] = 2.0 ** -21
    w.temperature[2] = 2.0 ** 20
    w.temperature[3] = 2.0 ** 21
    w.logits[4, 1, 3] = 2.0 ** 101
    w.logits[5, 0, 2] = -(2.0 ** 110)
    w.logits[6, 2, 7] = 2.0 ** 100
    w.logits[7, 0, :] = -(2.0 ** 120)
    g, o, rep = run(w, oracle_lib)
    assert list(g["row_status"]) == [0, 8, 0, 8, 4, 0, 0, 0]


def test_deterministic_and_phase_split_agree(oracle_lib):
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    w = W.make_workload("linear_b256_g8_v128256_bf16", B=16, V=9000)
    logits, q, toks, temp, uni = binding.linear_inputs_to_device(w)
    a = binding.verify_linear(logits, q, toks, temp, uni)
    b = binding.verify_linear(logits, q, toks, temp, uni)
    ws = binding.alloc_workspace(w.B, w.gamma + 1, w.V, binding.BF16)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = binding.LinearOut.empty(w.B, w.gamma, "cuda")
        binding.row_stats(logits, temp, ws, q=q, draft_tokens=toks, stream=s)
        binding.linear_finalize(logits, q, toks, temp, uni, out, ws, stream=s)
    s.synchronize()
    torch.cuda.synchronize()
    for k in ("n_accepted", "out_tokens", "final_token", "is_bonus", "row_status", "p_draft"):
        assert torch.equal(getattr(a, k), getattr(b, k)), k
        assert torch.equal(getattr(a, k), getattr(out, k)), k


@pytest.mark.parametrize("fill", [0x00, 0xFF, 0x5A])
def test_workspace_needs_no_initialisation(oracle_lib, fill):
    """Any workspace contents before a call give the same results, also when a
    workspace sized for one shape is reused for another."""
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    big = W.make_workload("linear_b256_g8_v128256_bf16", B=40, V=30011)
    small = W.make_workload("mixed_b512_g4_v152064_bf16", B=24, V=12347, seed_offset=3)
    ws = binding.alloc_workspace(big.B, big.gamma + 1, big.V, binding.BF16)
    for w in (big, small, big):
        args = binding.linear_inputs_to_device(w)
        want = binding.verify_linear(*args)
        ws.fill_(fill)
        got = binding.verify_linear(*args, workspace=ws)
        torch.cuda.synchronize()
        for k in ("n_accepted", "out_tokens", "final_token", "is_bonus", "row_status", "p_draft"):
            assert torch.equal(getattr(want, k), getattr(got, k)), (w.name, fill, k)


def test_phase_two_reruns_on_one_phase_one_result(oracle_lib):
    """Phase 2 leaves phase 1's result intact: with fresh uniforms it gives what a
    full call with those uniforms gives, and the oracle agrees."""
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    w = W.make_workload("linear_b256_g8_v128256_bf16", B=20, V=20011)
    logits, q, toks, temp, uni = binding.linear_inputs_to_device(w)
    ws = binding.alloc_workspace(w.B, w.gamma + 1, w.V, binding.BF16)
    binding.row_stats(logits, temp, ws, q=q, draft_tokens=toks)
    for seed in (1, 2, 3):
        u2 = W.philox_uniforms(1000 + seed, (w.B, w.gamma + 1))
        w2 = dataclasses.replace(w, uniforms=u2)
        uni2 = torch.from_numpy(u2).to("cuda")
        out = binding.LinearOut.empty(w.B, w.gamma, "cuda")
        binding.linear_finalize(logits, q, toks, temp, uni2, out, ws)
        full = binding.verify_linear(logits, q, toks, temp, uni2)
        torch.cuda.synchronize()
        for k in ("n_accepted", "out_tokens", "final_token", "is_bonus", "row_status", "p_draft"):
            assert torch.equal(getattr(out, k), getattr(full, k)), (seed, k)
        compare_linear(w2, {k: v.cpu().numpy() for k, v in vars(out).items()},
                       oracle_lib.verify_linear_workload(w2))
