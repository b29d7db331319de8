"""A two-level cascade verify ("Chapter 15: Decoding acceleration", the
multi-level speculation passage): the verify call applied level by level.
Level 1 verifies drafts from d against a middle model m; the tokens it emits
follow m, so they are the drafts of level 2, verified against the target p
with q = m.  The token the cascade emits must follow p.  The levels are the
library's verify call on the GPU; the same cascade through the oracle must
emit the same tokens."""
import numpy as np
import pytest
from scipy import special

from speculative_decoding_verification_64_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    from speculative_decoding_verification_64_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def tile(a, B):
    return np.ascontiguousarray(np.broadcast_to(a, (B,) + a.shape))


def gpu_verify(logits, q, toks, temp, uni):
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    dev = [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in (logits, q, toks, temp, uni)]
    out = binding.verify_linear(*dev)
    torch.cuda.synchronize()
    return out.out_tokens.cpu().numpy(), out.row_status.cpu().numpy()


def test_two_level_cascade_emits_the_target_law(oracle_lib):
    rng = np.random.default_rng(21)
    V, B, g1 = 6, 200_000, 3
    d = rng.dirichlet(np.ones(V)).astype(np.float32)                  # level-1 drafts
    lm = (rng.normal(size=V) * 1.2).astype(np.float32)                 # middle model logits
    lp = (rng.normal(size=V) * 1.2).astype(np.float32)                 # target logits
    m = special.softmax(lm.astype(np.float64))
    p = special.softmax(lp.astype(np.float64))
    dd = d.astype(np.float64)
    T = np.ones(B, np.float32)
    # level 1: g1 drafts from d, verified against m
    x = rng.choice(V, size=(B, g1), p=dd / dd.sum()).astype(np.int32)
    L1 = tile(np.stack([lm] * (g1 + 1)), B)
    Q1 = tile(np.stack([d] * g1), B)
    U1 = W.philox_uniforms(101, (B, g1 + 1))
    y, st1 = gpu_verify(L1, Q1, x, T, U1)
    assert (st1 == 0).all()
    # level 2: the first emitted token, drafted from m, verified against p
    y0 = np.ascontiguousarray(y[:, :1])
    L2 = tile(np.stack([lp, lp]), B)
    Q2 = tile(m.astype(np.float32)[None], B)
    U2 = W.philox_uniforms(102, (B, 2))
    z, st2 = gpu_verify(L2, Q2, y0, T, U2)
    assert (st2 == 0).all()
    # laws: level 1 emits m, the cascade emits p
    for tok, law in ((y0[:, 0], m), (z[:, 0], p)):
        freq = np.bincount(tok, minlength=V) / B
        se = np.sqrt(law * (1 - law) / B)
        assert (np.abs(freq - law) <= 5 * se + 1e-9).all(), (freq, law)
    # the oracle's cascade on the same inputs emits the same tokens
    o1 = oracle_lib.verify_linear(L1, Q1, "f32", x, T, U1, diagnostics=False)
    o2 = oracle_lib.verify_linear(L2, Q2, "f32", np.ascontiguousarray(o1["out_tokens"][:, :1]), T, U2,
                                  diagnostics=False)
    same1 = (o1["out_tokens"] == y).all(axis=1).mean()
    same2 = (o2["out_tokens"][:, 0] == z[:, 0]).mean()
    assert same1 >= 1 - 1e-4 and same2 >= 1 - 1e-4, (same1, same2)
