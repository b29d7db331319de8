"""GPU-vs-oracle comparison rules for the verify step.

Tolerances (written here, used by every parity test):
* target probabilities p_i(x~_i) / p_parent(t_n): absolute 2e-5 for float32
  inputs, 2e-3 for bfloat16 inputs;
* accepted counts, paths and every token: bit-exact, except in a request with
  a boundary draw: an accept test the oracle ran with |u - min(1, p/q)| < 1e-6,
  or a final draw whose U*Z lies within 1e-6*Z of a CDF boundary around the
  oracle's token.  A mismatch outside that band fails the test.  Mismatches
  inside the band ("excused") are counted.  The bound on them is a rate --
  at most 1e-4 of all draws -- which one case of a few hundred draws cannot
  estimate: a case fails when its count would be improbable (probability
  < 1e-3) if mismatches occurred at exactly that rate (``allowed_excused``:
  none in a case of a few draws, 1 in a case of tens to a few hundred, 2 in
  one of about a thousand), and
  ``test_gpu_boundary_rate.py`` checks the rate itself over tens of
  thousands of draws.  (With V ~ 1e5 a final draw can land in a cell only
  ~1e-8 of Z wide, and the float32 weights of the GPU path resolve CDF edges
  to about that precision; so in-band mismatches are rare but possible.)
* request status bitmasks: exact;
* the normaliser Z of each final draw (``specdec_final_mass``: the mass of
  max(0, p - q) at a rejection, of p for a bonus draw, of the final node's
  renormalised residual in the tree form), in target-probability units: the
  probability tolerance above, wherever the GPU and the oracle drew at the
  same row (greedy requests draw nothing and are skipped).
"""
import math

import numpy as np

BOUNDARY = 1e-6
P_TOL = {"f32": 2e-5, "bf16": 2e-3}
MISMATCH_RATE = 1e-4   # excused mismatches allowed per draw


def allowed_excused(draws: int, rate: float = MISMATCH_RATE, alpha: float = 1e-3) -> int:
    """Largest count m of excused mismatches a case of `draws` draws may show:
    the smallest m with P(X > m) < alpha for X ~ Binomial(draws, rate)."""
    if draws <= 0:
        return 0
    tail, m = 1.0, 0
    while True:
        # P(X = m), by the log-gamma form of the binomial coefficient
        lp = (math.lgamma(draws + 1) - math.lgamma(m + 1) - math.lgamma(draws - m + 1)
              + m * math.log(rate) + (draws - m) * math.log1p(-rate))
        tail -= math.exp(lp)
        if tail < alpha or m >= draws:
            return m
        m += 1


def linear_draws(o, gamma):
    k = o["n_accepted"].astype(np.int64)
    tests = np.minimum(k + 1, gamma)
    return int(tests.sum() + k.size)


def _mass_err(w, g, o, rows):
    """Largest |Z_gpu - Z_oracle| over the given requests (non-greedy, drawn at
    the same row by both sides); 0 when the GPU outputs carry no Z."""
    if g.get("final_mass") is None or o.get("final_mass") is None:
        return 0.0
    rows = [b for b in rows if w.temperature[b] != 0]
    if not rows:
        return 0.0
    gm = g["final_mass"][rows].astype(np.float64)
    om = o["final_mass"][rows]
    assert np.isfinite(gm).all(), ("no Z recorded for a drawn request", gm)
    return float(np.abs(gm - om).max())


def compare_linear(w, g, o, max_boundary_frac=1e-4):
    """g: GPU outputs as numpy dict; o: oracle outputs (with diagnostics)."""
    B, gamma = w.B, w.gamma
    rep = dict(B=B, draws=0, in_band=0, excused=0, max_p_err=0.0, max_mass_err=0.0)
    assert np.array_equal(g["row_status"], o["row_status"]), \
        (np.nonzero(g["row_status"] != o["row_status"]), g["row_status"], o["row_status"])
    ok = o["row_status"] == 0
    bad = ~ok
    if bad.any():
        assert (g["n_accepted"][bad] == 0).all() and (g["final_token"][bad] == -1).all()
        assert (g["out_tokens"][bad] == -1).all() and (g["is_bonus"][bad] == 0).all()
    if not ok.any():
        return rep
    if g.get("p_draft") is not None:
        err = np.abs(g["p_draft"][ok].astype(np.float64) - o["p_draft"][ok])
        rep["max_p_err"] = float(err.max())
        assert rep["max_p_err"] <= P_TOL[w.dtype], rep
    u = w.uniforms.astype(np.float64)
    same_rows = []
    for b in np.nonzero(ok)[0]:
        k = int(o["n_accepted"][b])
        ran = range(min(k + 1, gamma))
        greedy = w.temperature[b] == 0
        near = (not greedy) and any(abs(u[b, i] - o["ratio"][b, i]) < BOUNDARY for i in ran)
        near = near or ((not greedy) and o["final_margin"][b] < BOUNDARY)
        same = (g["n_accepted"][b] == k and g["final_token"][b] == o["final_token"][b]
                and g["is_bonus"][b] == o["is_bonus"][b]
                and np.array_equal(g["out_tokens"][b], o["out_tokens"][b]))
        if same:
            same_rows.append(int(b))
        if near:
            rep["in_band"] += 1
            rep["excused"] += int(not same)
            continue
        assert same, dict(b=int(b), gpu_k=int(g["n_accepted"][b]), ora_k=k,
                          gpu_tok=int(g["final_token"][b]), ora_tok=int(o["final_token"][b]),
                          ratio=o["ratio"][b], u=u[b], margin=o["final_margin"][b],
                          gpu_out=g["out_tokens"][b], ora_out=o["out_tokens"][b])
    rep["draws"] = linear_draws(o, gamma)
    assert rep["excused"] <= allowed_excused(rep["draws"], max_boundary_frac), rep
    rep["max_mass_err"] = _mass_err(w, g, o, same_rows)
    assert rep["max_mass_err"] <= P_TOL[w.dtype], rep
    return rep


def compare_tree(w, g, o, max_boundary_frac=1e-4):
    B = w.B
    rep = dict(B=B, draws=0, in_band=0, excused=0, max_p_err=0.0, max_mass_err=0.0)
    assert np.array_equal(g["row_status"], o["row_status"]), (g["row_status"], o["row_status"])
    ok = o["row_status"] == 0
    bad = ~ok
    if bad.any():
        assert (g["n_accepted"][bad] == 0).all() and (g["final_token"][bad] == -1).all()
        assert (g["out_tokens"][bad] == -1).all() and (g["path_nodes"][bad] == -1).all()
    if not ok.any():
        return rep
    if g.get("p_node") is not None:
        err = np.abs(g["p_node"][ok][:, 1:].astype(np.float64) - o["p_node"][ok][:, 1:])
        rep["max_p_err"] = float(err.max()) if err.size else 0.0
        assert rep["max_p_err"] <= P_TOL[w.dtype], rep
    same_rows = []
    for b in np.nonzero(ok)[0]:
        greedy = w.temperature[b] == 0
        near = (not greedy) and (o["test_margin"][b] < BOUNDARY or o["final_margin"][b] < BOUNDARY)
        same = all(np.array_equal(g[key][b], o[key][b]) for key in
                   ("n_accepted", "path_nodes", "out_tokens", "final_token", "is_bonus"))
        if same:
            same_rows.append(int(b))
        if near:
            rep["in_band"] += 1
            rep["excused"] += int(not same)
            continue
        assert same, dict(b=int(b), **{key: (g[key][b], o[key][b]) for key in
                                       ("n_accepted", "path_nodes", "out_tokens",
                                        "final_token", "is_bonus")},
                          tm=o["test_margin"][b], fm=o["final_margin"][b])
    rep["draws"] = int(o["n_accepted"].sum() + 2 * B)
    assert rep["excused"] <= allowed_excused(rep["draws"], max_boundary_frac), rep
    rep["max_mass_err"] = _mass_err(w, g, o, same_rows)
    assert rep["max_mass_err"] <= P_TOL[w.dtype], rep
    return rep


def gpu_linear(w, device="cuda", offset_elems=0):
    """Run the CUDA path on a LinearWorkload; returns numpy outputs.  With
    ``offset_elems`` the logits and q start that many elements past a
    16-byte boundary (exercises the unaligned edges of the bulk copies)."""
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    logits, q, toks, temp, uni = binding.linear_inputs_to_device(w, device)
    if offset_elems:
        logits = _offset_copy(logits, offset_elems)
        q = _offset_copy(q, offset_elems)
    dt = binding.dtype_code(logits)
    ws = binding.alloc_workspace(w.B, w.gamma + 1, w.V, dt, logits.device)
    out = binding.verify_linear(logits, q, toks, temp, uni, workspace=ws)
    mass = binding.final_mass(ws, w.B, w.gamma + 1, w.V, dt)
    torch.cuda.synchronize()
    g = {k: (None if v is None else v.cpu().numpy()) for k, v in vars(out).items()}
    g["final_mass"] = mass.cpu().numpy()
    return g


def gpu_tree(w, device="cuda", offset_elems=0):
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    logits, q, toks, par, temp, uni = binding.tree_inputs_to_device(w, device)
    if offset_elems:
        logits = _offset_copy(logits, offset_elems)
        q = _offset_copy(q, offset_elems)
    dt = binding.dtype_code(logits)
    ws = binding.alloc_workspace(w.B, w.N, w.V, dt, logits.device)
    out = binding.verify_tree(logits, q, toks, par, temp, uni, w.max_depth, workspace=ws)
    mass = binding.final_mass(ws, w.B, w.N, w.V, dt)
    torch.cuda.synchronize()
    g = {k: (None if v is None else v.cpu().numpy()) for k, v in vars(out).items()}
    g["final_mass"] = mass.cpu().numpy()
    return g


def _offset_copy(t, off):
    import torch
    flat = torch.empty(t.numel() + off, dtype=t.dtype, device=t.device)
    view = flat[off:].view(t.shape)
    view.copy_(t)
    return view
