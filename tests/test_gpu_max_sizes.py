"""Parity at the library's size limits.

* the largest vocabulary the ABI accepts (SPECDEC_MAX_V = 2^21): rows of 8 MB
  (float32) or 4 MB (bfloat16), thousands of stages per row, fixed-point draw
  totals near their widest;
* batches whose inputs span more than 4 GiB, so that every byte offset past
  32 bits is exercised in the stats pass, both linear draws, the top-k draw
  and the tree walk.

The large batches are built on the device by repeating a small generated
batch, with fresh uniforms for every request, so the host never holds them.
The oracle checks sampled requests one by one: the last requests (their rows
lie past 4 GiB), the first ones and a seeded random sample.  Properties that
hold at any size are checked on every request: copies of one generated
request get bit-identical target probabilities, the statuses are clean and
the emitted tokens are laid out as the call documents.
"""
import dataclasses

import numpy as np
import pytest

from parity import compare_linear, compare_tree, gpu_linear, gpu_tree
from speculative_decoding_verification_64_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_V = 1 << 21          # SPECDEC_MAX_V
FOUR_GIB = 1 << 32


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    from speculative_decoding_verification_64_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield
    torch.cuda.empty_cache()


def _numpy(out):
    return {k: (None if v is None else v.cpu().numpy()) for k, v in vars(out).items()}


def _sample(B, B0, seed):
    rng = np.random.default_rng(seed)
    idx = np.concatenate([np.arange(4), np.arange(B - 8, B), rng.choice(B, 8, replace=False)])
    return np.unique(idx)


def _check_layout(g, gamma, V, tokens):
    """Every request: clean status, n in [0, gamma], accepted drafts, then the
    final token, then -1."""
    assert (g["row_status"] == 0).all()
    n = g["n_accepted"]
    assert n.min() >= 0 and n.max() <= gamma
    assert ((g["final_token"] >= 0) & (g["final_token"] < V)).all()
    pos = np.arange(g["out_tokens"].shape[1])[None, :]
    want = np.where(pos < n[:, None], np.pad(tokens, ((0, 0), (0, 1)), constant_values=-1), -1)
    want[np.arange(n.size), n] = g["final_token"]
    assert np.array_equal(g["out_tokens"], want)
    assert np.array_equal(g["is_bonus"].astype(bool), n == gamma)


# --- the largest vocabulary


@pytest.mark.parametrize("dtype,offset", [("f32", 0), ("bf16", 0), ("bf16", 3)])
def test_linear_at_the_largest_vocabulary(oracle_lib, dtype, offset):
    # offset 0: aligned rows (bulk-copy draw); offset 3: unaligned rows (chunked draw)
    w = W.make_linear("normal2_tq08", B=3, gamma=2, V=MAX_V, dtype=dtype, seed=21)
    g = gpu_linear(w, offset_elems=offset)
    rep = compare_linear(w, g, oracle_lib.verify_linear_workload(w))
    print(dtype, offset, rep)


def test_tree_at_the_largest_vocabulary(oracle_lib):
    w = W.make_tree(B=2, N=10, V=MAX_V, dtype="bf16", seed=22, max_depth=3)
    g = gpu_tree(w)
    rep = compare_tree(w, g, oracle_lib.verify_tree_workload(w))
    print(rep)


# --- inputs past 4 GiB


def _tiled_linear(base, reps, seed):
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    logits, q, toks, temp, _ = binding.linear_inputs_to_device(base)
    B = base.B * reps
    uni = W.philox_uniforms(seed, (B, base.gamma + 1))
    x = (logits.repeat(reps, 1, 1), q.repeat(reps, 1, 1), toks.repeat(reps, 1),
         temp.repeat(reps), torch.from_numpy(uni).to("cuda"))
    assert x[0].numel() * x[0].element_size() > FOUR_GIB
    return x, uni


def _linear_sample(base, uni, idx):
    return dataclasses.replace(base.subset(idx % base.B), uniforms=uni[idx])


@pytest.mark.parametrize("law,V,B0,reps", [
    # 2048 requests: runs of more than 8 requests per CTA take the chunked draw
    ("zipf_t07", 128256, 16, 128),
    # 1024 requests of 512 KB rows: the bulk-copy draw
    ("normal2_tq08", 262144, 16, 64),
])
def test_linear_past_four_gib(oracle_lib, law, V, B0, reps):
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    base = W.make_linear(law, B=B0, gamma=8, V=V, dtype="bf16", seed=23)
    x, uni = _tiled_linear(base, reps, seed=24)
    assert binding.verify_linear_path(x[0], x[1]) == binding.PATH_TWO_LAUNCHES
    out = binding.verify_linear(*x)
    torch.cuda.synchronize()
    g = _numpy(out)
    # the same batch as the call's two phases issued separately: the same
    # outputs bit for bit
    ws = binding.alloc_workspace(x[0].shape[0], base.gamma + 1, V, binding.BF16)
    two = binding.LinearOut.empty(x[0].shape[0], base.gamma, "cuda")
    binding.row_stats(x[0], x[3], ws, q=x[1], draft_tokens=x[2])
    binding.linear_finalize(*x, two, ws)
    torch.cuda.synchronize()
    g2 = _numpy(two)
    for key in g:
        assert np.array_equal(g[key], g2[key], equal_nan=True), key
    del ws, two
    B = B0 * reps
    _check_layout(g, base.gamma, V, np.tile(base.draft_tokens, (reps, 1)))
    # copies of one generated request: bit-identical target probabilities
    pd = g["p_draft"].reshape(reps, B0, base.gamma)
    assert np.array_equal(pd, np.broadcast_to(pd[:1], pd.shape), equal_nan=True)
    idx = _sample(B, B0, seed=25)
    ws = _linear_sample(base, uni, idx)
    gs = {k: v[idx] for k, v in g.items()}
    rep = compare_linear(ws, gs, oracle_lib.verify_linear_workload(ws))
    print(law, V, B, rep)
    del x, out
    torch.cuda.empty_cache()


def test_topk_past_four_gib(oracle_lib):
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    base = W.make_linear("zipf_t07", B=16, gamma=8, V=128256, dtype="bf16", seed=26)
    reps, topk = 128, 32
    x, uni = _tiled_linear(base, reps, seed=27)
    out = binding.verify_linear_topk(*x, topk)
    torch.cuda.synchronize()
    g = _numpy(out)
    _check_layout(g, base.gamma, base.V, np.tile(base.draft_tokens, (reps, 1)))
    idx = _sample(base.B * reps, base.B, seed=28)
    ws = _linear_sample(base, uni, idx)
    gs = {k: v[idx] for k, v in g.items()}
    rep = compare_linear(ws, gs, oracle_lib.verify_linear_topk_workload(ws, topk))
    print(rep)
    del x, out
    torch.cuda.empty_cache()


def test_tree_past_four_gib(oracle_lib):
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    base = W.make_workload("tree_b32_n64_v128256_bf16", B=8, seed_offset=5)
    reps = 34
    B = base.B * reps
    logits, q, toks, par, temp, _ = binding.tree_inputs_to_device(base)
    uni = W.philox_uniforms(29, (B, base.N))
    x = (logits.repeat(reps, 1, 1), q.repeat(reps, 1, 1), toks.repeat(reps, 1),
         par.repeat(reps, 1), temp.repeat(reps), torch.from_numpy(uni).to("cuda"))
    assert x[0].numel() * x[0].element_size() > FOUR_GIB
    out = binding.verify_tree(*x, base.max_depth)
    torch.cuda.synchronize()
    g = _numpy(out)
    assert (g["row_status"] == 0).all()
    assert g["n_accepted"].min() >= 0 and g["n_accepted"].max() <= base.max_depth
    pn = g["p_node"].reshape(reps, base.B, base.N)
    assert np.array_equal(pn, np.broadcast_to(pn[:1], pn.shape), equal_nan=True)
    idx = _sample(B, base.B, seed=30)
    ws = dataclasses.replace(base.subset(idx % base.B), uniforms=uni[idx])
    gs = {k: v[idx] for k, v in g.items()}
    rep = compare_tree(ws, gs, oracle_lib.verify_tree_workload(ws))
    print(B, rep)
    del x, out
    torch.cuda.empty_cache()
