"""Host-side checks of the seeded synthetic inputs (no verify arithmetic)."""
import numpy as np
import pytest

from speculative_decoding_verification_64_gb300 import workloads as W


def test_bf16_encoding_round_to_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 0.0, 3.0e38, 1e-40],
                 np.float32)
    bits = W.f32_to_bf16_bits(x)
    assert list(bits[:5]) == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x0000]
    back = W.bf16_bits_to_f32(bits)
    assert back[0] == 1.0 and back[2] == np.float32(1.0 + 2 ** -6)
    # decode(encode(v)) is idempotent
    assert np.array_equal(W.f32_to_bf16_bits(back), bits)


def test_uniforms_exact_and_open_interval():
    u = W.philox_uniforms(123, (1000, 9))
    assert u.dtype == np.float32 and u.shape == (1000, 9)
    assert (u > 0).all() and (u < 1).all()
    k = u.astype(np.float64) * 2 ** 24
    assert np.array_equal(k, np.round(k)) and (np.round(k) % 2 == 1).all()
    assert np.array_equal(W.philox_uniforms(123, (1000, 9)), u)


@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_workloads_deterministic_and_prefix(name):
    a = W.make_workload(name, B=3, V=700)
    b = W.make_workload(name, B=3, V=700)
    c = W.make_workload(name, B=2, V=700)
    for f in ("logits", "q", "temperature", "uniforms"):
        assert np.array_equal(getattr(a, f), getattr(b, f))
    assert np.array_equal(a.logits[:2], c.logits) and np.array_equal(a.q[:2], c.q)
    assert np.array_equal(a.uniforms[:2], c.uniforms)


@pytest.mark.parametrize("name", [n for n, s in W.WORKLOADS.items() if s["kind"] == "linear"])
def test_linear_shapes_and_drafted_tokens_have_mass(name):
    w = W.make_workload(name, B=4, V=900)
    assert w.logits.shape == (w.B, w.gamma + 1, w.V)
    assert w.q.shape == (w.B, w.gamma, w.V)
    assert w.draft_tokens.shape == (w.B, w.gamma) and w.draft_tokens.dtype == np.int32
    q = W.decode(w.q, w.dtype)
    qx = np.take_along_axis(q, w.draft_tokens[..., None].astype(np.int64), -1)
    assert (qx > 0).all()
    assert np.allclose(q.sum(-1), 1.0, atol=5e-3)


def test_zipf_workload_overlap_at_least_07():
    w = W.make_workload("linear_b256_g8_v128256_bf16", B=3, V=5000)
    T = float(w.temperature[0])
    assert T == np.float32(0.7)
    l = W.decode(w.logits, w.dtype)[:, :w.gamma]
    p = np.exp(l / T - (l / T).max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    q = W.decode(w.q, w.dtype)
    assert (np.minimum(p, q).sum(-1) > 0.69).all()


def test_mixed_workload_temperatures():
    w = W.make_workload("mixed_b512_g4_v152064_bf16", B=512, V=16)
    greedy = w.temperature == 0
    assert greedy.sum() == round(0.1 * 512)
    t = w.temperature[~greedy]
    assert (t >= np.float32(0.3)).all() and (t <= np.float32(1.5)).all()


def test_tree_shape_bounds():
    w = W.make_workload("tree_b32_n64_v128256_bf16", B=8, V=300)
    assert w.N == 64 and w.max_depth == 5
    for b in range(w.B):
        par = w.parent[b]
        assert par[0] == -1
        assert all(0 <= par[n] < n for n in range(1, w.N))
        depth = np.zeros(w.N, int)
        for n in range(1, w.N):
            depth[n] = depth[par[n]] + 1
        assert depth.max() <= 5
        assert (np.diff(depth) >= 0).all()                # breadth-first numbering
        assert np.bincount(par[1:], minlength=w.N).max() <= 3
        q = W.decode(w.q[b], w.dtype)
        assert all(q[par[n], w.node_tokens[b, n]] > 0 for n in range(1, w.N))
