"""The stage-ring handshake of the streaming kernels, checked on a model.

The stats pass and the bulk-copy draw stream rows through a ring of shared
memory slots: one producer thread issues a bulk copy per unit into slot
n % S, completing that slot's "full" mbarrier; consumer warp w takes stages
w, w + W, w + 2W, ... (U stages per unit) and arrives on the slot's "empty"
mbarrier once it holds its stage.  Waits test a phase parity, which tells
only two phases apart, and copies land in any order.  A warp that skips a
slot's previous use must therefore first wait for that use's release on the
empty barrier; with the full-barrier wait alone it can pass while the
previous copy is still landing.

The model plays producer, copies and warps in random orders with long,
random copy latencies, using each kernel's (W, U, S) read from its source,
and checks that no wait ever passes on the wrong phase and that every run
finishes.  It also checks that the single-barrier wait does fail the model,
so that the model is known to detect the hazard.
"""
import os
import random
import re

import pytest

CSRC = os.path.join(os.path.dirname(__file__), "..", "speculative_decoding_verification_64_gb300",
                    "csrc")


def _define(path, name):
    text = open(os.path.join(CSRC, path)).read()
    m = re.search(r"#define\s+%s\s+(\d+)" % name, text)
    assert m, name
    return int(m.group(1))


def _constexpr(path, name):
    text = open(os.path.join(CSRC, path)).read()
    m = re.search(r"constexpr int %s = (\d+);" % name, text)
    assert m, name
    return int(m.group(1))


def stats_ring():
    return (_define("stats_stage.cuh", "SPECDEC_K1_WARPS"), _define("stats_stage.cuh", "SPECDEC_K1_UNIT"),
            _define("stats_stage.cuh", "SPECDEC_K1_SLOTS"))


def draw_ring():
    return (_constexpr("finalize_linear.cu", "kWarps"), _constexpr("finalize_linear.cu", "kUnitStages"),
            _constexpr("finalize_linear.cu", "kSlots"))


def run(W, U, S, units, seed, two_barrier, max_delay=40):
    """One randomised run; returns (finished, wrong passes)."""
    rnd = random.Random(seed)
    full_done = [0] * S      # completed phases of each full barrier
    full_pending = [0] * S   # copies outstanding in its current phase
    empty_done = [0] * S
    empty_arrived = [0] * S
    landing = []             # (tick, slot)
    issued = 0
    stages = [list(range(w, units * U, W)) for w in range(W)]
    at = [0] * W
    wrong = 0
    tick = 0
    while True:
        tick += 1
        moved = False
        for item in [x for x in landing if x[0] <= tick]:
            landing.remove(item)
            full_pending[item[1]] -= 1
            if full_pending[item[1]] == 0:
                full_done[item[1]] += 1
            moved = True
        actors = ["producer"] + list(range(W))
        rnd.shuffle(actors)
        for a in actors:
            if a == "producer":
                if issued < units:
                    s, use = issued % S, issued // S
                    if use == 0 or (empty_done[s] & 1) != ((use - 1) & 1):
                        if use > 0 and empty_done[s] != use:
                            wrong += 1
                        if full_pending[s]:
                            wrong += 1  # a second expect-tx arrival in a pending phase
                        full_pending[s] += 1
                        landing.append((tick + rnd.randint(1, max_delay), s))
                        issued += 1
                        moved = True
                continue
            w = a
            if at[w] == len(stages[w]):
                continue
            unit = stages[w][at[w]] // U
            s, use = unit % S, unit // S
            if two_barrier and use > 0 and (empty_done[s] & 1) == ((use - 1) & 1):
                continue
            if (full_done[s] & 1) != (use & 1):
                if full_done[s] != use + 1:
                    wrong += 1
                empty_arrived[s] += 1
                if empty_arrived[s] == U:
                    empty_arrived[s] = 0
                    empty_done[s] += 1
                at[w] += 1
                moved = True
        if issued == units and all(at[w] == len(stages[w]) for w in range(W)) and not landing:
            return True, wrong
        if (not moved and not landing) or tick > 200000:
            return False, wrong


@pytest.mark.parametrize("ring", [stats_ring(), draw_ring()], ids=["stats pass", "bulk draw"])
def test_two_barrier_wait_is_safe(ring):
    W, U, S = ring
    assert W <= S * U  # the kernels assert the same
    for seed in range(40):
        finished, wrong = run(W, U, S, units=200, seed=seed, two_barrier=True)
        assert finished and wrong == 0, (ring, seed, wrong)


def test_single_barrier_wait_fails_the_model():
    """The full-barrier wait alone breaks once a warp's next stage shares its
    slot with a use that other warps consumed (15 warps, 2-stage units)."""
    bad = 0
    for seed in range(20):
        finished, wrong = run(15, 2, 12, units=200, seed=seed, two_barrier=False)
        bad += (not finished) or wrong > 0
    assert bad > 0
