"""A seeded random sweep of sizes and layouts: CUDA path against the oracle.

The parametrised tests elsewhere pin the edges one at a time.  This sweep
draws configurations at random -- from a fixed seed, so the cases are the
same on every run -- across the boundaries between the kernels' paths: the
one-launch small-batch kernel and its cluster sizes, the two-launch step with
the bulk-copy draw (16-byte aligned rows) and the chunked draw (odd rows or
an offset base pointer), float32 and bfloat16, sampled and greedy requests,
and for the tree form random shapes, depths and branching.  Every case is
compared element by element under the tolerances of ``parity.py``, and the
linear sweep checks that it reached every path.
"""
import numpy as np
import pytest

from parity import _offset_copy, compare_linear, compare_tree, gpu_linear, gpu_tree
from speculative_decoding_verification_64_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    from speculative_decoding_verification_64_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"

LAWS = ["normal2_q05", "normal2_tq08", "zipf_t07", "mixed_normal3"]
MAX_ELEMS = 12_000_000  # target and draft elements per case: the oracle's share in seconds


def _linear_cases(n=28, seed=20261202):
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        B = int(np.exp(rng.uniform(0.0, np.log(200.0))))
        gamma = int(rng.choice([1, 2, 3, 4, 5, 8, 12, 32]))
        V = int(np.exp(rng.uniform(np.log(2.0), np.log(60000.0))))
        if rng.random() < 0.5:
            V = -(-V // 8) * 8  # rows a multiple of 16 bytes: the small and bulk paths
        if B * (2 * gamma + 1) * V > MAX_ELEMS:
            continue
        cases.append(dict(law=LAWS[int(rng.integers(len(LAWS)))], B=B, gamma=gamma, V=V,
                          dtype=str(rng.choice(["f32", "bf16"])),
                          offset=int(rng.choice([0, 0, 0, 1, 3])), seed=len(cases) + 100))
    # one case certain to take each path, whatever the draws above gave
    cases += [dict(law="normal2_q05", B=2, gamma=4, V=4096, dtype="f32", offset=0, seed=90),
              dict(law="zipf_t07", B=160, gamma=3, V=8192, dtype="bf16", offset=0, seed=91),
              dict(law="mixed_normal3", B=160, gamma=3, V=8191, dtype="bf16", offset=0, seed=92),
              dict(law="normal2_tq08", B=40, gamma=2, V=1000, dtype="bf16", offset=1, seed=93)]
    return cases


LINEAR = _linear_cases()


def _path(c):
    """The path a case's call takes: "small", "bulk" or "chunked" (from the
    sizes and the base pointers' alignment alone)."""
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    dt = torch.float32 if c["dtype"] == "f32" else torch.bfloat16
    logits = torch.empty((c["B"], c["gamma"] + 1, c["V"]), dtype=dt, device="cuda")
    q = torch.empty((c["B"], c["gamma"], c["V"]), dtype=dt, device="cuda")
    if c["offset"]:
        logits, q = _offset_copy(logits, c["offset"]), _offset_copy(q, c["offset"])
    if binding.verify_linear_path(logits, q) == binding.PATH_SMALL_ONE_LAUNCH:
        return "small"
    es = logits.element_size()
    aligned = (c["V"] * es) % 16 == 0 and logits.data_ptr() % 16 == 0 and q.data_ptr() % 16 == 0
    return "bulk" if aligned else "chunked"


@pytest.mark.parametrize("i", range(len(LINEAR)),
                         ids=[f"{c['law']}-B{c['B']}-g{c['gamma']}-V{c['V']}-{c['dtype']}-o{c['offset']}"
                              for c in LINEAR])
def test_linear_sweep(oracle_lib, i):
    c = LINEAR[i]
    w = W.make_linear(c["law"], B=c["B"], gamma=c["gamma"], V=c["V"], dtype=c["dtype"],
                      seed=c["seed"], greedy_frac=0.2, temp_range=(0.3, 1.5))
    g = gpu_linear(w, offset_elems=c["offset"])
    rep = compare_linear(w, g, oracle_lib.verify_linear_workload(w))
    print(w.name, c, _path(c), rep)
    assert 0 <= g["n_accepted"].min() and g["n_accepted"].max() <= w.gamma


def test_linear_sweep_reaches_every_path():
    assert {_path(c) for c in LINEAR} == {"small", "bulk", "chunked"}


def _tree_cases(n=12, seed=20261203):
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        depth = int(rng.integers(1, 7))
        branching = int(rng.integers(1, 5))
        full = sum(branching ** d for d in range(depth + 1))
        N = int(rng.integers(1, min(full, 160) + 1))
        B = int(rng.integers(1, 13))
        V = int(np.exp(rng.uniform(np.log(2.0), np.log(30000.0))))
        if B * N * V * 2 > MAX_ELEMS:
            continue
        cases.append(dict(B=B, N=N, V=V, depth=depth, branching=branching,
                          dtype=str(rng.choice(["f32", "bf16"])),
                          T=float(rng.choice([0.7, 1.0, 1.3])),
                          offset=int(rng.choice([0, 0, 1])), seed=len(cases) + 200))
    return cases


TREE = _tree_cases()


@pytest.mark.parametrize("i", range(len(TREE)),
                         ids=[f"B{c['B']}-N{c['N']}-V{c['V']}-d{c['depth']}-k{c['branching']}-{c['dtype']}-o{c['offset']}"
                              for c in TREE])
def test_tree_sweep(oracle_lib, i):
    c = TREE[i]
    w = W.make_tree(B=c["B"], N=c["N"], V=c["V"], dtype=c["dtype"], seed=c["seed"],
                    max_depth=c["depth"], branching=c["branching"], temperature=c["T"])
    g = gpu_tree(w, offset_elems=c["offset"])
    rep = compare_tree(w, g, oracle_lib.verify_tree_workload(w))
    print(w.name, c, rep)
