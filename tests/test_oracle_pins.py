"""Pins of the float64 oracle against what the method description fixes.

Source: "Chapter 15: Decoding acceleration" of the LLM edge inference notes
(zsc.github.io llm_edge_inference/chapter15):
  * section 15.1.2, speculative sampling steps 2-4, the theorem that the
    output law equals p, Lemma 1 (probability conservation), the law of the
    accepted count N and its expectation (i.i.d. and exponential decay);
  * section 15.1.3, the constant-acceptance expectation a(1-a^g)/(1-a);
  * the exercises (basic exercise 2: p = [0.5, 0.3, 0.2], q = [0.6, 0.3, 0.1]).

Each pin is chosen so that a plausible slip in the oracle (wrong row index,
wrong sign or missing clamp in the residual, reversed or strict accept
compare, bonus from the wrong row, non-strict CDF compare, wrong tie rule,
dropped temperature) fails at least one test.  No expected value here comes
from the CUDA path.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
from scipy import special, stats

from speculative_decoding_verification_64_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------
# helpers (input construction only)
# ----------------------------------------------------------------------------

def dyadic_rows(rng, rows, V, denom=1024, floor=16):
    """Probability rows that are exact in float32 and sum to exactly 1."""
    out = np.empty((rows, V))
    for r in range(rows):
        extra = rng.multinomial(denom - floor * V, rng.dirichlet(np.ones(V)))
        out[r] = (floor + extra) / denom
    return out


def target_rows(logits_f32, T):
    """Target distributions the oracle must see: softmax(l/T) of the stored
    float32 logits, by scipy (an independent routine)."""
    return special.softmax(logits_f32.astype(np.float64) / T, axis=-1)


def tile(a, n):
    return np.ascontiguousarray(np.broadcast_to(a, (n,) + a.shape))


# ----------------------------------------------------------------------------
# worked exercise
# ----------------------------------------------------------------------------

def test_exercise2_worked_example(oracle_lib):
    g = json.load(open(os.path.join(GOLDEN, "exercise2_pq.json")))
    p = np.array(g["p"])
    q = np.array(g["q"], dtype=np.float32)
    d = g["derived"]
    logits = np.stack([np.log(p), np.log(p)]).astype(np.float32)   # rows 0 and 1
    p_seen = target_rows(logits, 1.0)
    qf = q.astype(np.float64)
    # every draft token, accepted (u small) and rejected (u large)
    cases = []
    for tok in range(3):
        for u0 in (1e-3, 0.5, 0.999):
            for U in (0.01, 0.5, 0.99):
                cases.append((tok, u0, U))
    B = len(cases)
    out = oracle_lib.verify_linear(
        tile(logits, B), tile(q[None, :], B), "f32",
        np.array([[c[0]] for c in cases], np.int32), np.ones(B, np.float32),
        np.array([[c[1], c[2]] for c in cases], np.float32))
    ratio = out["ratio"][:, 0]
    for i, (tok, u0, U) in enumerate(cases):
        want_r = d["accept_prob_per_draft_token"][tok]
        assert abs(ratio[i] - want_r) < 1e-6
        assert abs(out["row_diag"][i, 0, 0] - d["sum_min_pq"]) < 1e-6
        assert abs(out["row_diag"][i, 0, 1] - d["sum_residual"]) < 1e-6
        # exact reference with the stored (rounded) values
        r_exact = min(1.0, p_seen[0, tok] / qf[tok])
        assert abs(ratio[i] - r_exact) < 1e-15
        if u0 <= r_exact:
            assert out["n_accepted"][i] == 1 and out["is_bonus"][i] == 1
        else:
            assert out["n_accepted"][i] == 0 and out["is_bonus"][i] == 0
            assert out["final_token"][i] == d["corrected_token_after_any_rejection"]
    # the residual is concentrated on token 2 with mass 0.1
    res = np.maximum(p_seen[0] - qf, 0)
    assert np.allclose(res, d["residual"], atol=1e-6)


# ----------------------------------------------------------------------------
# exact enumeration of the output law (the theorem of section 15.1.2)
# ----------------------------------------------------------------------------

def _linear_cells(p, q, gamma, V):
    """All decision cells of the verify step for a fixed set of rows.

    For every draft tuple (weight prod q_i(x_i)) and every stopping point j,
    and every token v of the final draw, returns the probability of that cell
    (accept test passes with probability min(1, p/q); final draw law = w/Z)
    and a uniform vector strictly inside it."""
    cells = []
    for x in itertools.product(range(V), repeat=gamma):
        wt = np.prod([q[i][x[i]] for i in range(gamma)])
        if wt == 0:
            continue
        r = [min(1.0, p[i][x[i]] / q[i][x[i]]) for i in range(gamma)]
        for j in range(gamma + 1):
            pj = wt * np.prod(r[:j]) * ((1.0 - r[j]) if j < gamma else 1.0)
            if pj <= 0:
                continue
            w = np.maximum(p[j] - q[j], 0.0) if j < gamma else p[gamma].copy()
            if w.sum() <= 0:
                w = p[j].copy()
            Z = w.sum()
            C = np.cumsum(w)
            for v in range(V):
                if w[v] <= 0:
                    continue
                U = (C[v] - w[v] / 2) / Z
                u = [r[i] / 2 for i in range(j)]
                if j < gamma:
                    u.append((1.0 + r[j]) / 2)
                u += [0.5] * (gamma - len(u))
                u.append(U)
                checkable = (w[v] / Z > 1e-6) and (j == gamma or 1.0 - r[j] > 1e-6)
                cells.append(dict(x=x, j=j, v=v, prob=pj * w[v] / Z, u=u,
                                  checkable=checkable))
    return cells


@pytest.mark.parametrize("V,gamma,T,seed", [(3, 2, 1.0, 0), (4, 3, 0.7, 1), (4, 2, 1.6, 2)])
def test_enumerated_output_law_is_p(oracle_lib, V, gamma, T, seed):
    rng = np.random.default_rng(seed)
    logits = rng.normal(0, 1.5, size=(gamma + 1, V)).astype(np.float32)
    p = target_rows(logits, T)
    q = dyadic_rows(rng, gamma, V)
    cells = _linear_cells(p, q, gamma, V)
    B = len(cells)
    out = oracle_lib.verify_linear(
        tile(logits, B), tile(q.astype(np.float32), B), "f32",
        np.array([c["x"] for c in cells], np.int32), np.full(B, T, np.float32),
        np.array([c["u"] for c in cells], np.float32))
    assert (out["row_status"] == 0).all()
    checked = 0
    for i, c in enumerate(cells):
        if not c["checkable"]:
            continue
        checked += 1
        assert out["n_accepted"][i] == c["j"], c
        assert out["final_token"][i] == c["v"], c
        assert out["is_bonus"][i] == (c["j"] == gamma)
        want = list(c["x"][:c["j"]]) + [c["v"]] + [-1] * (gamma - c["j"])
        assert list(out["out_tokens"][i]) == want
    assert checked >= 0.95 * B
    probs = np.array([c["prob"] for c in cells])
    assert abs(probs.sum() - 1.0) < 1e-12
    # law of the first emitted token is p_0
    first = np.array([c["x"][0] if c["j"] > 0 else c["v"] for c in cells])
    law = np.bincount(first, weights=probs, minlength=V)
    assert np.max(np.abs(law - p[0])) < 1e-12
    # given the first j drafts were accepted, the next emitted token ~ p_j
    for jc in range(1, gamma + 1):
        sel = [k for k, c in enumerate(cells) if c["j"] >= jc]
        tokj = np.array([cells[k]["x"][jc] if cells[k]["j"] > jc else cells[k]["v"]
                         for k in sel])
        lw = np.bincount(tokj, weights=probs[sel], minlength=V)
        assert np.max(np.abs(lw / probs[sel].sum() - p[jc])) < 1e-12


def test_boundary_conventions(oracle_lib):
    """u == min(1,p/q) accepts (the chapter's "u <= alpha"); the CDF draw is
    strict (first C_v > U Z); ties of the greedy argmax go to the lowest index."""
    V = 4
    logits = np.zeros((2, V), np.float32)           # p = 1/4 each, exactly
    q = np.array([[0.5, 0.5, 0.0, 0.0]], np.float32)  # r(token 0) = 0.5 exactly
    cases = [  # (u0, U, expected n_acc, expected final)
        (0.5, 0.5, 1, 2),          # u == r accepts; bonus U*Z = 0.5 = C_1 -> v = 2
        (0.5000001, 0.25, 0, 2),   # just above r rejects; residual (p-q)+ = [0,0,.25,.25]
        (0.5000001, 0.5, 0, 3),    # residual C = [0,0,.25,.5]; U*Z = .25 = C_2 -> v = 3
        (0.25, 0.25, 1, 1),        # bonus: U*Z = .25 = C_0 -> v = 1
        (0.25, 0.2499999, 1, 0),
    ]
    B = len(cases)
    out = oracle_lib.verify_linear(
        tile(logits, B), tile(q, B), "f32", np.zeros((B, 1), np.int32),
        np.ones(B, np.float32), np.array([[c[0], c[1]] for c in cases], np.float32))
    for i, c in enumerate(cases):
        assert out["n_accepted"][i] == c[2], (i, c)
        assert out["final_token"][i] == c[3], (i, c)


# ----------------------------------------------------------------------------
# Monte Carlo with the Philox uniform buffer (the oracle's u-driven path)
# ----------------------------------------------------------------------------

def _mc_linear(oracle_lib, p_logits, q, T, n, seed):
    gamma = q.shape[0]
    V = q.shape[1]
    rng = np.random.default_rng(seed + 100)
    toks = np.stack([rng.choice(V, size=n, p=q[i] / q[i].sum()) for i in range(gamma)],
                    axis=1).astype(np.int32)
    uni = W.philox_uniforms(seed, (n, gamma + 1))
    out = oracle_lib.verify_linear(tile(p_logits, n), tile(q.astype(np.float32), n), "f32",
                                   toks, np.full(n, T, np.float32), uni, diagnostics=False)
    assert (out["row_status"] == 0).all()
    return out


def _assert_freq(samples, p, V, z=5.0):
    n = samples.size
    f = np.bincount(samples, minlength=V) / n
    sd = np.sqrt(np.maximum(p * (1 - p), 1e-12) / n)
    assert np.all(np.abs(f - p) <= z * sd + 1e-12), (f, p)


def test_mc_output_law_and_count_law(oracle_lib):
    V, gamma, n, T = 4, 3, 400_000, 0.9
    rng = np.random.default_rng(11)
    logits = rng.normal(0, 1.2, size=(gamma + 1, V)).astype(np.float32)
    p = target_rows(logits, T)
    q = dyadic_rows(rng, gamma, V)
    out = _mc_linear(oracle_lib, logits, q, T, n, seed=21)
    _assert_freq(out["out_tokens"][:, 0], p[0], V)
    for j in range(1, gamma + 1):
        m = out["n_accepted"] >= j
        _assert_freq(out["out_tokens"][m, j], p[j], V)
    # law of N: P(N=k) = prod_{i<k} a_i (1 - a_k), a_i = sum_x min(p_i, q_i)
    a = np.minimum(p[:gamma], q).sum(axis=1)
    pk = np.array([np.prod(a[:k]) * (1 - a[k]) for k in range(gamma)] + [np.prod(a)])
    obs = np.bincount(out["n_accepted"], minlength=gamma + 1)
    chi = stats.chisquare(obs, pk * n)
    assert chi.pvalue > 1e-4


def _iid_rows(alphas):
    """V = 2 rows with p_i = (a_i, 1 - a_i) and q_i = (1, 0): the drafted token
    is always 0 and min(1, p/q) = a_i exactly as the rows fix it."""
    gamma = len(alphas)
    p = np.array([[a, 1 - a] for a in alphas] + [[0.5, 0.5]])
    logits = np.log(p).astype(np.float32)
    q = np.tile(np.array([1.0, 0.0]), (gamma, 1))
    return logits, q


@pytest.mark.parametrize("alpha,gamma", [(0.8, 4), (0.6, 8), (0.9, 1)])
def test_expected_accepted_iid(oracle_lib, alpha, gamma):
    n = 500_000
    logits, q = _iid_rows([alpha] * gamma)
    a = target_rows(logits, 1.0)[0, 0]                 # the alpha the rows realise
    out = _mc_linear(oracle_lib, logits, q, 1.0, n, seed=31 + gamma)
    N = out["n_accepted"].astype(np.float64)
    se = N.std() / math.sqrt(n)
    # section 15.1.2: E[N] = sum_{k<g} k a^k (1-a) + g a^g ; section 15.1.3: a(1-a^g)/(1-a)
    by_sum = sum(k * a ** k * (1 - a) for k in range(gamma)) + gamma * a ** gamma
    closed = a * (1 - a ** gamma) / (1 - a)
    assert abs(by_sum - closed) < 1e-12
    assert abs(N.mean() - closed) < 4 * se
    # the law of N itself (section 15.1.2, "distribution of accepted tokens")
    pk = np.array([a ** k * (1 - a) for k in range(gamma)] + [a ** gamma])
    obs = np.bincount(out["n_accepted"], minlength=gamma + 1)
    assert stats.chisquare(obs, pk * n).pvalue > 1e-4
    # the generating-function closed form printed in section 15.1.2,
    # a[1 - (g+1)a^g + g a^(g+1)] / (1-a)^2, is sum_{k=0}^{g} k a^k: it equals
    # E[N] only for g = 1.  The oracle follows the defining sum.
    printed = a * (1 - (gamma + 1) * a ** gamma + gamma * a ** (gamma + 1)) / (1 - a) ** 2
    assert abs(printed - sum(k * a ** k for k in range(gamma + 1))) < 1e-12
    if gamma == 1:
        assert abs(printed - closed) < 1e-12
    else:
        assert abs(N.mean() - printed) > 20 * se
    # second moment: E[N^2] = sum_k (2k-1) P(N >= k) = sum_{k=1}^{g} (2k-1) a^k
    m2 = sum((2 * k - 1) * a ** k for k in range(1, gamma + 1))
    se2 = (N ** 2).std() / math.sqrt(n)
    assert abs((N ** 2).mean() - m2) < 4 * se2


def test_printed_second_moment_is_garbled():
    """The closed form for E[N^2] printed in section 15.1.2 goes negative
    (a = 0.8, g = 2 gives -88.8); the defining sum it starts from does not."""
    a, g = 0.8, 2
    printed = a * (1 + a - (g * g + 2 * g + 1) * a ** g + (g * g + g) * a ** (g + 1)) / (1 - a) ** 3
    assert printed < 0
    by_def = sum(k * k * a ** k * (1 - a) for k in range(g)) + g * g * a ** g
    assert abs(by_def - sum((2 * k - 1) * a ** k for k in range(1, g + 1))) < 1e-12


@pytest.mark.parametrize("alpha,beta,gamma", [(0.9, 0.92, 8), (0.85, 0.95, 6)])
def test_expected_accepted_exponential_decay(oracle_lib, alpha, beta, gamma):
    n = 500_000
    al = [alpha * beta ** i for i in range(gamma)]
    logits, q = _iid_rows(al)
    a = target_rows(logits, 1.0)[:gamma, 0]
    out = _mc_linear(oracle_lib, logits, q, 1.0, n, seed=41 + gamma)
    N = out["n_accepted"].astype(np.float64)
    # section 15.1.2 exponential decay: E[N] = sum_{k=1}^{g} a^k b^(k(k-1)/2)
    closed = sum(alpha ** k * beta ** (k * (k - 1) / 2) for k in range(1, gamma + 1))
    exact = sum(np.prod(a[:k]) for k in range(1, gamma + 1))
    assert abs(closed - exact) < 1e-6
    assert abs(N.mean() - exact) < 4 * N.std() / math.sqrt(n)
    pk = np.array([np.prod(a[:k]) * (1 - a[k]) for k in range(gamma)] + [np.prod(a)])
    obs = np.bincount(out["n_accepted"], minlength=gamma + 1)
    assert stats.chisquare(obs, pk * n).pvalue > 1e-4


# ----------------------------------------------------------------------------
# Lemma 1, softmax, greedy limit
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["linear_b64_g5_v32000_bf16", "linear_b256_g8_v128256_bf16",
                                  "mixed_b512_g4_v152064_bf16"])
def test_lemma1_on_workload_rows(oracle_lib, name):
    w = W.make_workload(name, B=6, V=3000)
    out = oracle_lib.verify_linear_workload(w)
    ok = out["row_status"] == 0
    s = out["row_diag"][ok].sum(axis=-1)
    assert np.max(np.abs(s - 1.0)) < 1e-12


@pytest.mark.parametrize("T", [0.3, 1.0, 1.7])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_target_probability_matches_library_softmax(oracle_lib, T, dtype):
    B, gamma, V = 8, 3, 1000
    rng = np.random.default_rng(5)
    l64 = rng.normal(0, 3, size=(B, gamma + 1, V))
    logits = W.encode(l64, dtype)
    seen = W.decode(logits, dtype)
    q = np.full((B, gamma, V), 1.0 / V)
    toks = rng.integers(0, V, size=(B, gamma)).astype(np.int32)
    out = oracle_lib.verify_linear(logits, W.encode(q, dtype), dtype, toks,
                                   np.full(B, T, np.float32), W.philox_uniforms(9, (B, gamma + 1)))
    Tf = float(np.float32(T))
    p = special.softmax(seen / Tf, axis=-1)
    want = np.take_along_axis(p[:, :gamma], toks[..., None].astype(np.int64), axis=-1)[..., 0]
    assert np.max(np.abs(out["p_draft"] / want - 1)) < 1e-12


def test_greedy_rows_follow_first_argmax(oracle_lib):
    B, gamma, V = 400, 4, 40
    rng = np.random.default_rng(3)
    logits = rng.integers(-3, 4, size=(B, gamma + 1, V)).astype(np.float32)   # many ties
    amax = logits.argmax(axis=-1)                        # numpy: first occurrence
    toks = np.where(rng.random((B, gamma)) < 0.7, amax[:, :gamma],
                    rng.integers(0, V, size=(B, gamma))).astype(np.int32)
    q = np.full((B, gamma, V), 1.0 / V, np.float32)
    out = oracle_lib.verify_linear(logits, q, "f32", toks, np.zeros(B, np.float32),
                                   W.philox_uniforms(4, (B, gamma + 1)))
    for b in range(B):
        k = gamma
        for i in range(gamma):
            if toks[b, i] != amax[b, i]:
                k = i
                break
        assert out["n_accepted"][b] == k
        assert out["final_token"][b] == amax[b, k]
        assert out["is_bonus"][b] == (k == gamma)
        r = out["ratio"][b]
        for i in range(gamma):
            assert r[i] == (1.0 if toks[b, i] == amax[b, i] else 0.0)


def test_small_temperature_tends_to_greedy(oracle_lib):
    B, gamma, V = 200, 3, 64
    rng = np.random.default_rng(8)
    # distinct logits spaced >= 0.25 apart: at T = 1e-3 the softmax is one-hot to e^-250
    base = np.arange(V, dtype=np.float64) * 0.25
    logits = np.stack([np.stack([rng.permutation(base) for _ in range(gamma + 1)])
                       for _ in range(B)]).astype(np.float32)
    amax = logits.argmax(axis=-1)
    toks = np.where(rng.random((B, gamma)) < 0.6, amax[:, :gamma],
                    rng.integers(0, V, size=(B, gamma))).astype(np.int32)
    q = np.full((B, gamma, V), 1.0 / V, np.float32)
    uni = W.philox_uniforms(12, (B, gamma + 1))
    g = oracle_lib.verify_linear(logits, q, "f32", toks, np.zeros(B, np.float32), uni)
    s = oracle_lib.verify_linear(logits, q, "f32", toks, np.full(B, 1e-3, np.float32), uni)
    for key in ("n_accepted", "final_token", "out_tokens", "is_bonus"):
        assert np.array_equal(g[key], s[key]), key


# ----------------------------------------------------------------------------
# malformed requests
# ----------------------------------------------------------------------------

def test_input_domain_edges(oracle_lib):
    """Valid temperatures are 0 or [2^-20, 2^20]; a row whose largest logit
    exceeds 2^100 is not usable (so l/T cannot overflow float32); very
    negative finite logits are valid (zero mass)."""
    B, gamma, V = 6, 1, 8
    logits = np.zeros((B, gamma + 1, V), np.float32)
    q = np.full((B, gamma, V), 1.0 / V, np.float32)
    toks = np.zeros((B, gamma), np.int32)
    temp = np.ones(B, np.float32)
    temp[0] = 2.0 ** -20
    temp[1] = 2.0 ** -21
    temp[2] = 2.0 ** 20
    temp[3] = 2.0 ** 21
    logits[4, 1, 3] = 2.0 ** 101
    logits[5, 0, 2] = -(2.0 ** 110)
    logits[5, 1, 0] = 2.0 ** 100
    out = oracle_lib.verify_linear(logits, q, "f32", toks, temp,
                                   W.philox_uniforms(3, (B, gamma + 1)))
    assert list(out["row_status"]) == [0, oracle_lib.ROW_BAD_TEMP, 0, oracle_lib.ROW_BAD_TEMP,
                                       oracle_lib.ROW_NONFINITE, 0]
    assert out["final_token"][5] >= 0


def test_status_bits_and_sentinels(oracle_lib):
    B, gamma, V = 8, 2, 16
    rng = np.random.default_rng(1)
    logits = rng.normal(size=(B, gamma + 1, V)).astype(np.float32)
    q = np.full((B, gamma, V), 1.0 / V, np.float32)
    toks = rng.integers(0, V, size=(B, gamma)).astype(np.int32)
    temp = np.ones(B, np.float32)
    logits[1, 2, 5] = np.nan
    logits[2, 0, 3] = np.inf
    logits[3, 1, :] = -np.inf
    toks[4, 1] = V
    q[5, 0, toks[5, 0]] = 0.0
    temp[6] = -1.0
    logits[7, 0, :4] = -np.inf                        # partial -inf is a valid row
    out = oracle_lib.verify_linear(logits, q, "f32", toks, temp,
                                   W.philox_uniforms(2, (B, gamma + 1)))
    st = out["row_status"]
    assert list(st) == [0, oracle_lib.ROW_NONFINITE, oracle_lib.ROW_NONFINITE,
                        oracle_lib.ROW_NONFINITE, oracle_lib.ROW_BAD_TOKEN,
                        oracle_lib.ROW_BAD_Q, oracle_lib.ROW_BAD_TEMP, 0]
    bad = st != 0
    assert (out["n_accepted"][bad] == 0).all() and (out["final_token"][bad] == -1).all()
    assert (out["out_tokens"][bad] == -1).all() and (out["is_bonus"][bad] == 0).all()
    assert out["final_token"][7] >= 4                 # -inf logits have zero mass


# ----------------------------------------------------------------------------
# token tree
# ----------------------------------------------------------------------------

def _chain_from_linear(w):
    """The linear workload as a chain tree: node n <-> row n, node n's token
    is draft n-1, tree slot n <-> linear slot n-1, tree slot 0 <-> slot gamma."""
    B, g, V = w.B, w.gamma, w.V
    N = g + 1
    q = np.zeros((B, N, V), dtype=w.q.dtype)
    q[:, :g] = w.q
    q[:, g] = w.q[:, g - 1]                           # leaf row: never read
    toks = np.zeros((B, N), np.int32)
    toks[:, 1:] = w.draft_tokens
    parent = np.tile(np.arange(-1, N - 1, dtype=np.int32), (B, 1))
    uni = np.empty((B, N), np.float32)
    uni[:, 1:] = w.uniforms[:, :g]
    uni[:, 0] = w.uniforms[:, g]
    return q, toks, parent, uni


@pytest.mark.parametrize("dtype,T", [("f32", 0.8), ("bf16", 1.0), ("bf16", 0.0)])
def test_chain_tree_equals_linear(oracle_lib, dtype, T):
    w = W.make_linear("normal2_tq08", B=3000, gamma=5, V=50, dtype=dtype, seed=13)
    w.temperature[:] = T
    lin = oracle_lib.verify_linear_workload(w)
    q, toks, parent, uni = _chain_from_linear(w)
    tr = oracle_lib.verify_tree(w.logits, q, dtype, toks, parent, w.temperature, uni,
                                max_depth=w.gamma)
    for key in ("n_accepted", "final_token", "is_bonus", "row_status", "out_tokens"):
        assert np.array_equal(lin[key], tr[key]), key
    D1 = w.gamma + 1
    for b in range(w.B):
        k = lin["n_accepted"][b]
        assert list(tr["path_nodes"][b]) == list(range(k + 1)) + [-1] * (D1 - k - 1)
    assert 0 < lin["n_accepted"].mean() < w.gamma


def _tree_cells_star(p_root, p_child, q, K, V):
    """Exact cells of a star tree: root with K leaf children whose tokens are
    i.i.d. from q.  Sibling s is tested against the current P (p_root, then
    max(0, P - q)/sum after each rejection); an accepted leaf c draws its bonus
    from p_child[c]; if all are rejected the final token is drawn from P."""
    cells = []
    for t in itertools.product(range(V), repeat=K):
        wt = np.prod([q[x] for x in t])
        if wt == 0:
            continue
        P = p_root.copy()
        reach = wt
        rej_u = []
        for s in range(K):
            r = min(1.0, P[t[s]] / q[t[s]])
            if r > 0:
                pa = reach * r
                w = p_child[s]
                C = np.cumsum(w)
                for v in range(V):
                    if w[v] <= 0:
                        continue
                    u = [0.0] * (K + 1)
                    u[0] = (C[v] - w[v] / 2) / w.sum()
                    for s2, uu in enumerate(rej_u):
                        u[1 + s2] = uu
                    u[1 + s] = r / 2
                    for s2 in range(s + 1, K):
                        u[1 + s2] = 0.5
                    ok = w[v] / w.sum() > 1e-6 and all(x < 1 - 1e-7 for x in rej_u)
                    cells.append(dict(t=t, acc=s + 1, v=v, prob=pa * w[v] / w.sum(),
                                      u=u, checkable=ok, first=t[s]))
            if r >= 1:
                reach = 0
                break
            rej_u.append((1.0 + r) / 2)
            reach *= (1 - r)
            nxt = np.maximum(P - q, 0)
            if nxt.sum() > 0:
                P = nxt / nxt.sum()
        if reach > 0:
            C = np.cumsum(P)
            for v in range(V):
                if P[v] <= 0:
                    continue
                u = [0.0] * (K + 1)
                u[0] = (C[v] - P[v] / 2) / P.sum()
                for s2, uu in enumerate(rej_u):
                    u[1 + s2] = uu
                ok = P[v] / P.sum() > 1e-6 and all(x < 1 - 1e-7 for x in rej_u)
                cells.append(dict(t=t, acc=None, v=v, prob=reach * P[v] / P.sum(), u=u,
                                  checkable=ok, first=v))
    return cells


@pytest.mark.parametrize("V,K,seed", [(3, 2, 0), (4, 3, 1), (3, 3, 2)])
def test_tree_enumerated_law_is_p(oracle_lib, V, K, seed):
    rng = np.random.default_rng(seed + 50)
    N = K + 1
    logits = rng.normal(0, 1.3, size=(N, V)).astype(np.float32)
    p = target_rows(logits, 1.0)
    q_root = dyadic_rows(rng, 1, V)[0]
    cells = _tree_cells_star(p[0], p[1:], q_root, K, V)
    B = len(cells)
    qrows = np.tile(q_root.astype(np.float32), (N, 1))
    toks = np.array([[0] + list(c["t"]) for c in cells], np.int32)
    parent = np.tile(np.array([-1] + [0] * K, np.int32), (B, 1))
    out = oracle_lib.verify_tree(tile(logits, B), tile(qrows, B), "f32", toks, parent,
                                 np.ones(B, np.float32), np.array([c["u"] for c in cells],
                                                                  np.float32), max_depth=1)
    assert (out["row_status"] == 0).all()
    checked = 0
    for i, c in enumerate(cells):
        if not c["checkable"]:
            continue
        checked += 1
        if c["acc"] is None:
            assert out["n_accepted"][i] == 0 and out["is_bonus"][i] == 0, c
            assert out["final_token"][i] == c["v"], c
        else:
            assert out["n_accepted"][i] == 1 and out["is_bonus"][i] == 1, c
            assert out["path_nodes"][i, 1] == c["acc"], c
            assert out["final_token"][i] == c["v"], c
    assert checked >= 0.95 * B
    probs = np.array([c["prob"] for c in cells])
    assert abs(probs.sum() - 1) < 1e-12
    law = np.bincount([c["first"] for c in cells], weights=probs, minlength=V)
    assert np.max(np.abs(law - p[0])) < 1e-12


def test_tree_mc_two_level_law(oracle_lib):
    """Root -> nodes 1, 2; node 1 -> nodes 3, 4; node 2 -> node 5 (all siblings
    i.i.d. from the parent's q).  First emitted token ~ p_0; given the walk
    accepted node c at depth 1, the next emitted token ~ p_c."""
    V, n = 4, 300_000
    parent1 = np.array([-1, 0, 0, 1, 1, 2], np.int32)
    N = parent1.size
    rng = np.random.default_rng(77)
    logits = rng.normal(0, 1.0, size=(N, V)).astype(np.float32)
    p = target_rows(logits, 1.0)
    q = dyadic_rows(rng, N, V)
    toks = np.zeros((n, N), np.int32)
    for node in range(1, N):
        qp = q[parent1[node]]
        toks[:, node] = rng.choice(V, size=n, p=qp)
    out = oracle_lib.verify_tree(tile(logits, n), tile(q.astype(np.float32), n), "f32", toks,
                                 tile(parent1, n), np.ones(n, np.float32),
                                 W.philox_uniforms(66, (n, N)), max_depth=2, diagnostics=False)
    assert (out["row_status"] == 0).all()
    _assert_freq(out["out_tokens"][:, 0], p[0], V)
    for c in (1, 2):
        m = out["path_nodes"][:, 1] == c
        assert m.sum() > 10_000
        _assert_freq(out["out_tokens"][m, 1], p[c], V)


def test_tree_residual_identity():
    """After j rejected siblings the literally renormalised residual equals
    (p - c_j q)+ / N_j with c_0 = 0, N_0 = 1, c_{j+1} = c_j + N_j and
    N_{j+1} = sum (p - c_{j+1} q)+ (derived by induction; lets a kernel keep
    only two scalars instead of a residual row)."""
    rng = np.random.default_rng(4)
    for _ in range(50):
        V = 200
        p = rng.dirichlet(np.ones(V) * 0.5)
        q = rng.dirichlet(np.ones(V) * 0.5)
        P = p.copy()
        c, Nj = 0.0, 1.0
        for _j in range(6):
            lit = np.maximum(P - q, 0)
            if lit.sum() <= 0:
                break
            P = lit / lit.sum()
            c = c + Nj
            Nj = np.maximum(p - c * q, 0).sum()
            ident = np.maximum(p - c * q, 0) / Nj
            assert np.max(np.abs(P - ident)) < 1e-12


def test_tree_greedy_walk(oracle_lib):
    B, N, V = 300, 20, 12
    w = W.make_tree(B, N, V, "f32", seed=5, max_depth=4, branching=3)
    rng = np.random.default_rng(9)
    logits = rng.integers(-2, 3, size=(B, N, V)).astype(np.float32)
    amax = logits.argmax(axis=-1)
    toks = w.node_tokens.copy()
    # make some children carry their parent's argmax token
    for b in range(B):
        for n in range(1, N):
            if rng.random() < 0.4:
                toks[b, n] = amax[b, w.parent[b, n]]
    temp = np.zeros(B, np.float32)
    out = oracle_lib.verify_tree(logits, w.q, "f32", toks, w.parent, temp, w.uniforms,
                                 max_depth=4)
    for b in range(B):
        cur, path = 0, [0]
        while True:
            kids = [n for n in range(N) if w.parent[b, n] == cur]
            hit = [n for n in kids if toks[b, n] == amax[b, cur]]
            if hit:
                cur = hit[0]
                path.append(cur)
                continue
            break
        assert list(out["path_nodes"][b][:len(path)]) == path
        assert out["n_accepted"][b] == len(path) - 1
        assert out["final_token"][b] == amax[b, cur]
        leaf = not any(w.parent[b, n] == cur for n in range(N))
        assert out["is_bonus"][b] == leaf


def test_tree_status_bits(oracle_lib):
    w = W.make_tree(6, 10, 30, "f32", seed=2, max_depth=3, branching=3)
    parent = w.parent.copy()
    toks = w.node_tokens.copy()
    logits = w.logits.copy()
    parent[1, 0] = 0                      # root must have parent -1
    parent[2, 5] = 7                      # forward reference
    toks[3, 4] = -2
    logits[4, 9, 0] = np.nan
    out = oracle_lib.verify_tree(logits, w.q, "f32", toks, parent, w.temperature,
                                 w.uniforms, max_depth=3)
    st = out["row_status"]
    assert st[0] == 0 and st[5] == 0
    assert st[1] & oracle_lib.ROW_BAD_TREE and st[2] & oracle_lib.ROW_BAD_TREE
    assert st[3] == oracle_lib.ROW_BAD_TOKEN and st[4] == oracle_lib.ROW_NONFINITE
    # depth bound: the same trees are too deep for max_depth = 1
    out2 = oracle_lib.verify_tree(w.logits, w.q, "f32", w.node_tokens, w.parent,
                                  w.temperature, w.uniforms, max_depth=1)
    deep = np.array([(np.bincount(np.r_[0, w.parent[b, 1:]]) > 0).sum() > 1 for b in range(6)])
    assert (out2["row_status"][deep] & oracle_lib.ROW_BAD_TREE).all()


# --- Philox4x64-10 uniforms (the device generator's oracle) -----------------
# Pinned against NumPy's Philox bit generator: an independent implementation of
# the same published generator, whose raw words the oracle must reproduce for
# any key, counter (including carries across the 64-bit counter words) and
# starting word.

def _numpy_philox(key, counter):
    import numpy as np
    bg = np.random.Philox(0)
    st = bg.state
    st["state"]["key"] = np.asarray(key, dtype=np.uint64)
    st["state"]["counter"] = np.asarray(counter, dtype=np.uint64)
    st["buffer_pos"] = 4
    bg.state = st
    return bg


@pytest.mark.parametrize("counter", [
    [0, 0, 0, 0],
    [2**64 - 3, 7, 0, 0],                               # carry into word 1
    [2**64 - 1, 2**64 - 1, 2**64 - 1, 2**64 - 5],       # carries through three words
    [123456789, 2**63, 5, 2**64 - 1],
])
@pytest.mark.parametrize("key", [[0, 0], [2**64 - 1, 1], [0x0123456789ABCDEF, 0xFEDCBA9876543210]])
def test_philox_words_match_numpy(oracle_lib, key, counter):
    import numpy as np
    want = _numpy_philox(key, counter).random_raw(64)
    for first, n in [(0, 64), (1, 10), (3, 5), (4, 4), (17, 40)]:
        got = oracle_lib.philox_words(key, counter, first, n)
        assert np.array_equal(got, want[first:first + n]), (first, n)


@pytest.mark.parametrize("seed,shape,offset", [(0, (3, 5), 0), (7, (257,), 6), (2024, (4, 9), 1001)])
def test_philox_uniforms_match_the_workload_stream(oracle_lib, seed, shape, offset):
    import numpy as np
    want = W.philox_uniforms(seed, shape, offset_words=offset).reshape(-1)
    st = np.random.Philox(seed).state["state"]
    got = oracle_lib.philox_uniforms(st["key"], st["counter"], offset, want.size)
    assert got.dtype == np.float32
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    assert (got > 0).all() and (got < 1).all()


# --- per-row entropy and path log-probability -------------------------------

def test_entropy_of_a_uniform_row_is_log_v(oracle_lib):
    for V in (1, 2, 7, 1000):
        lg = np.zeros((1, 2, V), dtype=np.float32)
        h = oracle_lib.row_entropy(lg, "f32", np.array([0.9], dtype=np.float32))
        assert np.allclose(h, math.log(V), atol=1e-12, rtol=0)


def test_entropy_matches_scipy_and_the_binary_closed_form(oracle_lib):
    rng = np.random.default_rng(5)
    lg = (rng.normal(size=(3, 4, 500)) * 2).astype(np.float32)
    T = np.array([1.0, 0.37, 2.5], dtype=np.float32)
    h = oracle_lib.row_entropy(lg, "f32", T)
    for b in range(3):
        for i in range(4):
            p = special.softmax(lg[b, i].astype(np.float64) / float(T[b]))
            assert abs(h[b, i] - stats.entropy(p)) < 1e-10
    # two tokens, logits (0, x): binary entropy of sigmoid(x / T)
    for x, t in ((0.0, 1.0), (1.5, 0.5), (-3.0, 2.0)):
        lg2 = np.array([[[0.0, x]]], dtype=np.float32)
        s = 1.0 / (1.0 + math.exp(-x / t))
        want = -(s * math.log(s) + (1 - s) * math.log(1 - s))
        got = oracle_lib.row_entropy(lg2, "f32", np.array([t], dtype=np.float32))[0, 0]
        assert abs(got - want) < 1e-12


def test_entropy_special_rows(oracle_lib):
    lg = np.zeros((4, 1, 6), dtype=np.float32)
    lg[1, 0, :3] = -np.inf                  # masked half: uniform over the rest
    lg[2, 0, 2] = np.nan
    T = np.array([0.0, 1.0, 1.0, -1.0], dtype=np.float32)
    h = oracle_lib.row_entropy(lg, "f32", T)[:, 0]
    assert h[0] == 0.0                      # greedy: one-hot
    assert abs(h[1] - math.log(3)) < 1e-12
    assert np.isnan(h[2]) and np.isnan(h[3])


def test_path_logprob_matches_log_softmax(oracle_lib):
    rng = np.random.default_rng(6)
    B, R, V = 5, 4, 300
    lg = (rng.normal(size=(B, R, V)) * 2).astype(np.float32)
    T = np.array([1.0, 0.6, 1.7, 1.0, 0.8], dtype=np.float32)
    toks = rng.integers(0, V, size=(B, R)).astype(np.int32)
    nacc = np.array([0, 1, 3, 2, 3], dtype=np.int32)
    got = oracle_lib.path_logprob(lg, "f32", T, toks, nacc)
    for b in range(B):
        want = sum(special.log_softmax(lg[b, j].astype(np.float64) / float(T[b]))[toks[b, j]]
                   for j in range(nacc[b] + 1))
        assert abs(got[b] - want) < 1e-10
    # tree form: rows named by the path, here the nodes 0, 2, 3
    nodes = np.tile(np.array([[0, 2, 3, -1]], dtype=np.int32), (B, 1))
    nacc2 = np.full(B, 2, dtype=np.int32)
    got2 = oracle_lib.path_logprob(lg, "f32", T, toks, nacc2, path_nodes=nodes)
    for b in range(B):
        want = sum(special.log_softmax(lg[b, r].astype(np.float64) / float(T[b]))[toks[b, j]]
                   for j, r in enumerate((0, 2, 3)))
        assert abs(got2[b] - want) < 1e-10


def test_path_logprob_special_cases(oracle_lib):
    lg = np.zeros((4, 2, 5), dtype=np.float32)
    lg[:, :, 3] = 1.0                       # argmax 3 in every row
    T = np.array([0.0, 0.0, 1.0, 1.0], dtype=np.float32)
    toks = np.array([[3, 3], [3, 1], [3, 9], [3, 3]], dtype=np.int32)
    nacc = np.array([1, 1, 1, 1], dtype=np.int32)
    status = np.array([0, 0, 0, 2], dtype=np.int32)
    got = oracle_lib.path_logprob(lg, "f32", T, toks, nacc, row_status=status)
    assert got[0] == 0.0                    # greedy path of arg-maxima
    assert got[1] == -np.inf                # greedy path through a non-maximum
    assert np.isnan(got[2])                 # token out of range
    assert np.isnan(got[3])                 # malformed request


# --- top-k residual (an approximate mode of the correction draw) -------------

def test_topk_residual_with_every_token_is_the_exact_step(oracle_lib):
    w = W.make_workload("linear_b64_g5_v32000_bf16", B=12, V=3001)
    exact = oracle_lib.verify_linear_workload(w)
    approx = oracle_lib.verify_linear_topk_workload(w, topk=w.V)
    for k in ("n_accepted", "out_tokens", "final_token", "is_bonus", "row_status"):
        assert np.array_equal(exact[k], approx[k]), k
    assert np.nanmax(np.abs(approx["tv"])) < 1e-12


def test_topk_tv_is_the_mass_outside_the_candidates(oracle_lib):
    w = W.make_workload("linear_b256_g8_v128256_bf16", B=10, V=4000)
    K = 16
    got = oracle_lib.verify_linear_topk_workload(w, topk=K)
    logits = W.decode(w.logits, w.dtype).astype(np.float64)
    qd = W.decode(w.q, w.dtype).astype(np.float64)
    for b in range(w.B):
        k = got["n_accepted"][b]
        if got["row_status"][b] or k == w.gamma:
            assert np.isnan(got["tv"][b])
            continue
        p = special.softmax(logits[b, k] / float(w.temperature[b]))
        r = np.maximum(p - qd[b, k], 0.0)
        cand = np.lexsort((np.arange(w.V), -p))[:K]          # largest p, ties to the lower index
        assert abs(got["tv"][b] - (1.0 - r[cand].sum() / r.sum())) < 1e-12
        assert got["final_token"][b] in set(cand.tolist())


def test_topk_candidates_break_ties_by_index(oracle_lib):
    # p ties on tokens 1, 2, 3; q puts no mass there, so every residual draw is a candidate
    lg = np.array([[[0.0, 2.0, 2.0, 2.0, 1.0], [0.0] * 5]], dtype=np.float32)
    q = np.array([[[0.97, 0.0, 0.0, 0.0, 0.03]]], dtype=np.float32)
    toks = np.array([[0]], dtype=np.int32)
    seen = set()
    for u1 in np.linspace(0.01, 0.99, 41):
        uni = np.array([[0.9999, u1]], dtype=np.float32)        # reject draft 0
        out = oracle_lib.verify_linear_topk(lg, q, "f32", toks, np.array([1.0], np.float32), uni, 2)
        seen.add(int(out["final_token"][0]))
    assert seen == {1, 2}


def test_topk_law_by_monte_carlo(oracle_lib):
    """gamma = 1: the first emitted token has law min(p, q) + Z * r_K / Z_K."""
    rng = np.random.default_rng(9)
    V, K, n = 6, 2, 200_000
    lg = rng.normal(size=V).astype(np.float32)
    p = special.softmax(lg.astype(np.float64))
    qv = rng.dirichlet(np.ones(V)).astype(np.float32)
    qd = qv.astype(np.float64)
    toks = rng.choice(V, size=n, p=qd / qd.sum()).astype(np.int32)
    logits = np.broadcast_to(np.stack([lg, lg])[None], (n, 2, V)).copy()
    q = np.broadcast_to(qv[None, None], (n, 1, V)).copy()
    uni = W.philox_uniforms(77, (n, 2))
    out = oracle_lib.verify_linear_topk(logits, q, "f32", toks[:, None],
                                        np.ones(n, np.float32), uni, K)
    first = out["out_tokens"][:, 0]
    r = np.maximum(p - qd, 0.0)
    cand = np.argsort(-p, kind="stable")[:K]
    rk = np.zeros(V)
    rk[cand] = r[cand]
    law = np.minimum(p, qd) + r.sum() * rk / rk.sum()
    freq = np.bincount(first, minlength=V) / n
    se = np.sqrt(law * (1 - law) / n)
    assert (np.abs(freq - law) <= 5 * se + 1e-9).all()


# ----------------------------------------------------------------------------
# per-position acceptance rate alpha = sum_v min(p, q)
# ----------------------------------------------------------------------------

def test_alpha_matches_the_absolute_difference_form(oracle_lib):
    """sum min(p, q) = (sum p + sum q - sum |p - q|) / 2 for any nonnegative
    rows, with p from scipy's softmax and q as stored (not summing to 1)."""
    rng = np.random.default_rng(11)
    B, gamma, V = 3, 4, 700
    lg = (rng.normal(size=(B, gamma + 1, V)) * 2).astype(np.float32)
    q = rng.dirichlet(np.ones(V), size=(B, gamma)).astype(np.float32) * 1.03
    T = np.array([1.0, 0.45, 2.2], dtype=np.float32)
    a = oracle_lib.row_alpha(lg, q, "f32", T)
    for b in range(B):
        for i in range(gamma):
            p = special.softmax(lg[b, i].astype(np.float64) / float(T[b]))
            qd = q[b, i].astype(np.float64)
            want = 0.5 * (p.sum() + qd.sum() - np.abs(p - qd).sum())
            assert abs(a[b, i] - want) < 1e-12


def test_alpha_special_rows(oracle_lib):
    V = 8
    lg = np.zeros((4, 2, V), dtype=np.float32)
    q = np.zeros((4, 1, V), dtype=np.float32)
    # q = p: alpha 1 (uniform rows)
    q[0, 0] = 1.0 / V
    # disjoint supports: p on tokens 0..3 (-inf elsewhere), q on 4..7
    lg[1, 0, 4:] = -np.inf
    q[1, 0, 4:] = 0.25
    # greedy row: p one-hot at the first arg-max (token 2), alpha = q(2)
    lg[2, 0] = [0, 1, 3, 3, 0, 0, 0, 0]
    q[2, 0] = np.linspace(0.05, 0.2, V)
    # invalid temperature: NaN
    q[3, 0] = 1.0 / V
    T = np.array([1.0, 0.7, 0.0, -1.0], dtype=np.float32)
    a = oracle_lib.row_alpha(lg, q, "f32", T)[:, 0]
    assert abs(a[0] - 1.0) < 1e-12
    assert a[1] == 0.0
    assert a[2] == np.float64(q[2, 0, 2])
    assert np.isnan(a[3])


def test_alpha_is_the_first_draft_acceptance_rate(oracle_lib):
    """Monte Carlo through the verify step itself: a draft drawn from q is
    accepted with probability sum min(p, q)."""
    rng = np.random.default_rng(12)
    V, n = 9, 100_000
    lg = (rng.normal(size=V) * 1.5).astype(np.float32)
    qv = rng.dirichlet(np.ones(V)).astype(np.float32)
    qd = qv.astype(np.float64)
    toks = rng.choice(V, size=n, p=qd / qd.sum()).astype(np.int32)
    logits = np.broadcast_to(np.stack([lg, lg])[None], (n, 2, V)).copy()
    q = np.broadcast_to(qv[None, None], (n, 1, V)).copy()
    T = np.full(n, 0.8, np.float32)
    out = oracle_lib.verify_linear(logits, q, "f32", toks[:, None], T, W.philox_uniforms(78, (n, 2)),
                                   diagnostics=False)
    freq = float((out["n_accepted"] == 1).mean())
    a = float(oracle_lib.row_alpha(logits[:1], q[:1], "f32", T[:1])[0, 0])
    assert abs(freq - a) <= 5 * math.sqrt(a * (1 - a) / n)


def test_alpha_agrees_with_the_verify_diagnostics(oracle_lib):
    w = W.make_workload("mixed_b512_g4_v152064_bf16", B=6, V=900)
    a = oracle_lib.row_alpha(w.logits, w.q, w.dtype, w.temperature)
    d = oracle_lib.verify_linear_workload(w)["row_diag"][..., 0]
    ok = np.isfinite(a)
    assert ok.any()
    assert np.allclose(a[ok], d[ok], rtol=0, atol=1e-12)


def test_cascade_of_two_verify_levels_emits_the_target_law(oracle_lib):
    """Multi-level speculation: level 1 verifies drafts from d against m, and
    its emitted token, drafted from m, is verified against p; the cascade's
    token follows p (Monte Carlo)."""
    rng = np.random.default_rng(22)
    V, n = 5, 200_000
    d = rng.dirichlet(np.ones(V)).astype(np.float32)
    lm = (rng.normal(size=V) * 1.3).astype(np.float32)
    lp = (rng.normal(size=V) * 1.3).astype(np.float32)
    m = special.softmax(lm.astype(np.float64))
    p = special.softmax(lp.astype(np.float64))
    dd = d.astype(np.float64)
    T = np.ones(n, np.float32)
    x = rng.choice(V, size=(n, 2), p=dd / dd.sum()).astype(np.int32)
    o1 = oracle_lib.verify_linear(tile(np.stack([lm] * 3), n), tile(np.stack([d] * 2), n), "f32", x, T,
                                  W.philox_uniforms(201, (n, 3)), diagnostics=False)
    y0 = np.ascontiguousarray(o1["out_tokens"][:, :1])
    o2 = oracle_lib.verify_linear(tile(np.stack([lp, lp]), n), tile(m.astype(np.float32)[None], n), "f32",
                                  y0, T, W.philox_uniforms(202, (n, 2)), diagnostics=False)
    for tok, law in ((y0[:, 0], m), (o2["out_tokens"][:, 0], p)):
        freq = np.bincount(tok, minlength=V) / n
        se = np.sqrt(law * (1 - law) / n)
        assert (np.abs(freq - law) <= 5 * se + 1e-9).all()


# ----------------------------------------------------------------------------
# the final draw's normaliser Z (section 15.1.2 step 4: the correction is
# drawn from max(0, p - q) / Z)
# ----------------------------------------------------------------------------

def test_final_mass_of_exercise2(oracle_lib):
    """Exercise 2's distributions: after any rejection Z = sum (p - q)+ = 0.1
    (the derivation in the golden file); after an acceptance the bonus draw
    from p has Z = 1."""
    g = json.load(open(os.path.join(GOLDEN, "exercise2_pq.json")))
    p = np.array(g["p"])
    q = np.array(g["q"], dtype=np.float32)
    logits = np.stack([np.log(p), np.log(p)]).astype(np.float32)
    cases = [(tok, u0) for tok in range(3) for u0 in (1e-3, 0.999)]
    B = len(cases)
    out = oracle_lib.verify_linear(
        tile(logits, B), tile(q[None, :], B), "f32",
        np.array([[c[0]] for c in cases], np.int32), np.ones(B, np.float32),
        np.array([[c[1], 0.5] for c in cases], np.float32))
    for i in range(B):
        if out["n_accepted"][i] == 0:
            assert abs(out["final_mass"][i] - g["derived"]["sum_residual"]) < 1e-6
        else:
            assert abs(out["final_mass"][i] - 1.0) < 1e-12
    assert (out["n_accepted"] == 0).any() and (out["n_accepted"] == 1).any()


def test_final_mass_is_the_conservation_complement(oracle_lib):
    """At a rejection at row k, Z = sum (p_k - q_k)+ = 1 - sum min(p_k, q_k)
    (Lemma 1's conservation), with p_k from scipy's softmax; a bonus draw
    has Z = sum p_gamma = 1.  Malformed requests report NaN."""
    rng = np.random.default_rng(31)
    B, gamma, V, T = 64, 4, 300, 0.8
    logits = rng.normal(0, 2, size=(B, gamma + 1, V)).astype(np.float32)
    q = special.softmax(rng.normal(0, 2, size=(B, gamma, V)), axis=-1).astype(np.float32)
    toks = np.array([[rng.choice(V, p=q[b, i] / q[b, i].sum()) for i in range(gamma)]
                     for b in range(B)], np.int32)
    temp = np.full(B, T, np.float32)
    temp[5] = -1.0                                      # malformed: bad temperature
    uni = rng.uniform(0.05, 0.95, size=(B, gamma + 1)).astype(np.float32)
    out = oracle_lib.verify_linear(logits, q, "f32", toks, temp, uni)
    p = special.softmax(logits.astype(np.float64) / float(np.float32(T)), axis=-1)  # T as stored
    for b in range(B):
        if out["row_status"][b]:
            assert np.isnan(out["final_mass"][b])
            continue
        k = int(out["n_accepted"][b])
        if k == gamma:
            want = p[b, gamma].sum()
        else:
            # sum (p - q)+ = sum p - sum min(p, q), whatever q (as stored) sums to
            want = 1.0 - np.minimum(p[b, k], q[b, k].astype(np.float64)).sum()
        assert abs(out["final_mass"][b] - want) < 1e-12, (b, k)
    assert 0 < out["n_accepted"].mean() < gamma


def test_final_mass_of_a_tree_after_rejected_siblings(oracle_lib):
    """A root with K children whose tests all fail: the final draw is from the
    root's residual after K renormalisations, whose mass relative to p is
    N_K = sum (p - c_K q)+ with c_0 = 0, N_0 = 1, c_{j+1} = c_j + N_j (the
    residual identity, here in numpy); with no rejection (a leaf) Z = 1."""
    rng = np.random.default_rng(8)
    B, K, V = 40, 3, 50
    N = K + 1
    logits = rng.normal(0, 1.5, size=(B, N, V)).astype(np.float32)
    q = special.softmax(rng.normal(0, 1.5, size=(B, N, V)), axis=-1)
    q = (q / q.sum(-1, keepdims=True)).astype(np.float32)
    parent = np.array([[-1] + [0] * K] * B, np.int32)
    toks = np.zeros((B, N), np.int32)
    for b in range(B):
        toks[b, 1:] = rng.choice(V, size=K, p=q[b, 0] / q[b, 0].sum())
    uni = np.full((B, N), 0.9999999, np.float32)      # every sibling test fails ...
    uni[::4, 1] = 1e-7                                  # ... except the first on every 4th tree
    uni[:, 0] = rng.uniform(0.01, 0.99, size=B)
    temp = np.ones(B, np.float32)
    out = oracle_lib.verify_tree(logits, q, "f32", toks, parent, temp, uni, max_depth=1)
    p = special.softmax(logits[:, 0].astype(np.float64), axis=-1)
    for b in range(B):
        assert out["row_status"][b] == 0
        if out["n_accepted"][b] == 1:                   # accepted child: a leaf, bonus draw
            assert abs(out["final_mass"][b] - 1.0) < 1e-12
            continue
        qq = q[b, 0].astype(np.float64)
        c, Nj = 0.0, 1.0
        for _ in range(K):                              # one renormalisation per rejected child
            r = np.maximum(p[b] - (c + Nj) * qq, 0).sum()
            if r <= 0:
                break
            c, Nj = c + Nj, r
        assert abs(out["final_mass"][b] - Nj) < 1e-12, (b, out["final_mass"][b], Nj)
    assert (out["n_accepted"] == 0).sum() > 20 and (out["n_accepted"] == 1).sum() > 5
