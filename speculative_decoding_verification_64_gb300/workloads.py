"""Seeded synthetic inputs for the speculative-decoding verify step.

This module only *makes inputs*: target logits, the draft's stored
distributions q, draft tokens drawn from q, per-request temperatures, token
trees and the uniform buffer.  It holds none of the verify arithmetic (no
target softmax, no accept test, no residual, no draw from the target side);
both the CUDA path and the float64 oracle consume what it produces.

The draft distributions are a stand-in for a draft model: they are built here
in float64 numpy from perturbed logits (the draft side of the method is out of
scope, so q is an input), then stored in the same dtype as the logits.  Draft
tokens are drawn from the stored q, so every drafted token has q > 0.

Workload laws follow the five synthetic verify workloads of the method
description ("Speculative decoding" chapter 15.1 of the edge-inference
textbook for the algorithm; the workloads themselves are synthetic):

* ``linear_b1``   B=1,   gamma=4, V=32000,  fp32, l ~ N(0, 2^2), T=1,
                  q = softmax(l + N(0, 0.5^2))
* ``linear_b64``  B=64,  gamma=5, V=32000,  bf16, l ~ N(0, 2^2), T_p=1,
                  q = softmax((l + N(0, 1)) / 0.8)
* ``linear_b256`` B=256, gamma=8, V=128256, bf16, Zipf logits
                  l[perm[r]] = -1.1 ln(r+1) + N(0,1), T=0.7,
                  q = 0.7 p + 0.3 softmax(N(0,1)) with p = softmax(l/0.7)
* ``mixed_b512``  B=512, gamma=4, V=152064, bf16, l ~ N(0, 3^2),
                  T_b ~ U[0.3, 1.5], 10% of requests greedy (T=0),
                  q = softmax((l + N(0,1)) / T_b) (T_b=1 for greedy rows)
* ``tree_b32``    B=32, N=64 nodes, depth <= 5, branching <= 3, V=128256,
                  bf16, l ~ N(0, 2^2), T=1, q_n = softmax(l_n + N(0,1)),
                  node tokens i.i.d. from q_parent.

Random streams (all platform independent):
* uniforms: ``Generator(Philox(seed))`` raw 64-bit words, row-major over the
  whole [B, R] buffer, mapped to u = ((w >> 41) + 0.5) * 2^-23, i.e.
  u = (2k+1) 2^-24 with k < 2^23: exact in float32, never 0 or 1;
* per-request data: ``default_rng(SeedSequence([seed + 1000, b]))``;
* per-request draft tokens and tree shape:
  ``Generator(Philox(SeedSequence([seed + 1, b])))``.
Per-request streams make a smaller batch a prefix of a larger one.
"""
from __future__ import annotations

import concurrent.futures
import dataclasses
import os
from typing import Dict, Optional

import numpy as np

F32 = "f32"
BF16 = "bf16"


# ----------------------------------------------------------------------------
# encodings and random streams
# ----------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); returns uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    rounding = np.uint64(0x7FFF) + ((bits >> np.uint64(16)) & np.uint64(1))
    out = ((bits + rounding) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bits to float32."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def encode(x: np.ndarray, dtype: str) -> np.ndarray:
    """float array -> storage array (float32, or uint16 bf16 bits)."""
    if dtype == F32:
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == BF16:
        return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))
    raise ValueError(f"unknown dtype {dtype!r}")


def decode(a: np.ndarray, dtype: str) -> np.ndarray:
    """storage array -> float64 values (exact)."""
    if dtype == F32:
        return np.asarray(a, dtype=np.float32).astype(np.float64)
    if dtype == BF16:
        return bf16_bits_to_f32(a).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


def philox_uniforms(seed: int, shape, offset_words: int = 0) -> np.ndarray:
    """float32 uniforms in (0,1) from Philox(seed): u = ((w >> 41) + 0.5) * 2^-23.

    ``offset_words`` skips that many 64-bit words first (used to give each
    rank of a sharded run its own slice of one stream).
    """
    n = int(np.prod(shape)) if len(shape) else 1
    bg = np.random.Philox(seed)
    if offset_words:
        bg.advance(offset_words // 4)  # Philox counter step = 4 words
        skip = offset_words % 4
        if skip:
            bg.random_raw(skip)
    raw = bg.random_raw(n).astype(np.uint64)
    k = (raw >> np.uint64(41)).astype(np.float64)
    u = ((k + 0.5) * (2.0 ** -23)).astype(np.float32)
    return u.reshape(shape)


def _per_request(B: int, fill) -> None:
    """Run ``fill(b)`` for every request b on a pool of threads.  Each request
    draws from its own generators and writes only its own slices, so the
    result does not depend on the thread count or the order; numpy releases
    the interpreter lock inside the bulk draws and array arithmetic."""
    workers = max(1, min(B, os.cpu_count() or 1, 16))
    if workers == 1:
        for b in range(B):
            fill(b)
        return
    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
        for f in [ex.submit(fill, b) for b in range(B)]:
            f.result()


def _data_rng(seed: int, b: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([seed + 1000, b]))


def _token_rng(seed: int, b: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([seed + 1, b])))


def _draft_softmax(x: np.ndarray) -> np.ndarray:
    """Draft-model stand-in: exp-normalise along the last axis (float64)."""
    x = np.asarray(x, dtype=np.float64)
    e = np.exp(x - x.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def _draw_from_rows(rows: np.ndarray, rng: np.random.Generator) -> np.ndarray:
    """One categorical draw per row of non-negative weights (draft-side sampling)."""
    rows = np.asarray(rows, dtype=np.float64)
    cdf = np.cumsum(rows, axis=-1)
    total = cdf[..., -1]
    u = rng.random(rows.shape[:-1]) * total
    out = np.empty(rows.shape[:-1], dtype=np.int64)
    flat_cdf = cdf.reshape(-1, rows.shape[-1])
    flat_u = u.reshape(-1)
    flat_out = out.reshape(-1)
    for i in range(flat_cdf.shape[0]):
        flat_out[i] = np.searchsorted(flat_cdf[i], flat_u[i], side="right")
    np.minimum(out, rows.shape[-1] - 1, out=out)
    return out.astype(np.int32)


# ----------------------------------------------------------------------------
# workload containers
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class LinearWorkload:
    name: str
    dtype: str                 # "f32" | "bf16"
    B: int
    gamma: int
    V: int
    logits: np.ndarray         # [B, gamma+1, V] float32 or uint16 (bf16 bits)
    q: np.ndarray              # [B, gamma, V]   same storage dtype
    draft_tokens: np.ndarray   # int32 [B, gamma]
    temperature: np.ndarray    # float32 [B]; 0 = greedy
    uniforms: np.ndarray       # float32 [B, gamma+1]; slot gamma = final draw

    @property
    def rows(self) -> int:
        return self.gamma + 1

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == F32 else 2

    def subset(self, idx) -> "LinearWorkload":
        idx = np.asarray(idx)
        return dataclasses.replace(
            self, B=int(idx.size), logits=np.ascontiguousarray(self.logits[idx]),
            q=np.ascontiguousarray(self.q[idx]),
            draft_tokens=np.ascontiguousarray(self.draft_tokens[idx]),
            temperature=np.ascontiguousarray(self.temperature[idx]),
            uniforms=np.ascontiguousarray(self.uniforms[idx]))


@dataclasses.dataclass
class TreeWorkload:
    name: str
    dtype: str
    B: int
    N: int
    V: int
    max_depth: int
    logits: np.ndarray         # [B, N, V]: row n = target distribution after the path to node n
    q: np.ndarray              # [B, N, V]: row n = draft distribution of node n's children
    node_tokens: np.ndarray    # int32 [B, N]; entry 0 (root) unused
    parent: np.ndarray         # int32 [B, N]; parent[0] = -1, parent[n] < n
    temperature: np.ndarray    # float32 [B]
    uniforms: np.ndarray       # float32 [B, N]; slot 0 = final draw, slot n = node n's test

    @property
    def rows(self) -> int:
        return self.N

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == F32 else 2

    def subset(self, idx) -> "TreeWorkload":
        idx = np.asarray(idx)
        return dataclasses.replace(
            self, B=int(idx.size), logits=np.ascontiguousarray(self.logits[idx]),
            q=np.ascontiguousarray(self.q[idx]),
            node_tokens=np.ascontiguousarray(self.node_tokens[idx]),
            parent=np.ascontiguousarray(self.parent[idx]),
            temperature=np.ascontiguousarray(self.temperature[idx]),
            uniforms=np.ascontiguousarray(self.uniforms[idx]))


# ----------------------------------------------------------------------------
# per-request laws
# ----------------------------------------------------------------------------

def _linear_request(law: str, V: int, gamma: int, rng: np.random.Generator):
    """Returns (target logits [gamma+1, V] float64, draft q [gamma, V] float64, T)."""
    R = gamma + 1
    if law == "normal2_q05":          # B=1 fp32 workload
        l = rng.normal(0.0, 2.0, size=(R, V))
        q = _draft_softmax(l[:gamma] + rng.normal(0.0, 0.5, size=(gamma, V)))
        return l, q, 1.0
    if law == "normal2_tq08":         # B=64 workload
        l = rng.normal(0.0, 2.0, size=(R, V))
        q = _draft_softmax((l[:gamma] + rng.normal(0.0, 1.0, size=(gamma, V))) / 0.8)
        return l, q, 1.0
    if law == "zipf_t07":             # B=256 workload
        base = -1.1 * np.log(np.arange(V, dtype=np.float64) + 1.0)
        l = np.empty((R, V))
        for r in range(R):
            perm = rng.permutation(V)
            l[r, perm] = base + rng.normal(0.0, 1.0, size=V)
        T = 0.7
        p_draft_side = _draft_softmax(l[:gamma] / T)
        noise = _draft_softmax(rng.normal(0.0, 1.0, size=(gamma, V)))
        q = 0.7 * p_draft_side + 0.3 * noise
        return l, q, T
    raise ValueError(f"unknown linear law {law!r}")


def make_linear(law: str, B: int, gamma: int, V: int, dtype: str, seed: int,
                name: Optional[str] = None, greedy_frac: float = 0.0,
                temp_range=None) -> LinearWorkload:
    """Build a linear-verify workload.

    ``law`` in {"normal2_q05", "normal2_tq08", "zipf_t07", "mixed_normal3"}.
    For "mixed_normal3" the per-request temperature is U[temp_range] and a
    ``greedy_frac`` share of the requests (chosen by the seed) is greedy.
    """
    R = gamma + 1
    logits = np.empty((B, R, V), dtype=np.float32 if dtype == F32 else np.uint16)
    q = np.empty((B, gamma, V), dtype=np.float32 if dtype == F32 else np.uint16)
    toks = np.empty((B, gamma), dtype=np.int32)
    temp = np.empty((B,), dtype=np.float32)
    if law == "mixed_normal3":
        lo, hi = temp_range if temp_range is not None else (0.3, 1.5)
        sel = np.random.default_rng(np.random.SeedSequence([seed + 2000]))
        temps = sel.uniform(lo, hi, size=B)
        n_greedy = int(round(greedy_frac * B))
        greedy = np.zeros(B, dtype=bool)
        greedy[sel.permutation(B)[:n_greedy]] = True
        temps[greedy] = 0.0
    def fill(b):
        rng = _data_rng(seed, b)
        if law == "mixed_normal3":
            T = float(np.float32(temps[b]))
            l = rng.normal(0.0, 3.0, size=(R, V))
            Tq = T if T > 0 else 1.0
            qb = _draft_softmax((l[:gamma] + rng.normal(0.0, 1.0, size=(gamma, V))) / Tq)
        else:
            l, qb, T = _linear_request(law, V, gamma, rng)
        logits[b] = encode(l, dtype)
        q[b] = encode(qb, dtype)
        stored_q = decode(q[b], dtype)
        toks[b] = _draw_from_rows(stored_q, _token_rng(seed, b))
        temp[b] = T

    _per_request(B, fill)
    uni = philox_uniforms(seed, (B, R))
    return LinearWorkload(name or f"{law}_b{B}_g{gamma}_v{V}_{dtype}", dtype, B, gamma, V,
                          logits, q, toks, temp, uni)


def random_tree_shape(N: int, max_depth: int, branching: int,
                      rng: np.random.Generator) -> np.ndarray:
    """Parent array of a random N-node subtree of the full ``branching``-ary tree
    of depth ``max_depth``, grown one node at a time from a uniformly chosen free
    child slot, then renumbered breadth first (children in slot order), so
    parent[0] = -1 and parent[n] < n."""
    full = sum(branching ** d for d in range(max_depth + 1))
    if not 1 <= N <= full:
        raise ValueError("N does not fit the tree bounds")
    depth = [0]
    kids = [[]]                        # child slots used, in slot order
    par = [-1]
    slot_of = [0]
    free = [(0, s) for s in range(branching)] if max_depth > 0 else []
    while len(par) < N:
        i = int(rng.integers(len(free)))
        node, slot = free.pop(i)
        new = len(par)
        par.append(node)
        depth.append(depth[node] + 1)
        slot_of.append(slot)
        kids.append([])
        kids[node].append(new)
        if depth[new] < max_depth:
            free.extend((new, s) for s in range(branching))
    # breadth-first renumbering with children ordered by slot
    order = [0]
    head = 0
    while head < len(order):
        n = order[head]
        head += 1
        order.extend(sorted(kids[n], key=lambda c: slot_of[c]))
    new_id = {old: i for i, old in enumerate(order)}
    parent = np.full(N, -1, dtype=np.int32)
    for old in range(1, N):
        parent[new_id[old]] = new_id[par[old]]
    return parent


def make_tree(B: int, N: int, V: int, dtype: str, seed: int, max_depth: int = 5,
              branching: int = 3, temperature: float = 1.0, logit_sigma: float = 2.0,
              name: Optional[str] = None) -> TreeWorkload:
    """Build a token-tree verify workload (siblings i.i.d. from q_parent)."""
    logits = np.empty((B, N, V), dtype=np.float32 if dtype == F32 else np.uint16)
    q = np.empty((B, N, V), dtype=np.float32 if dtype == F32 else np.uint16)
    toks = np.zeros((B, N), dtype=np.int32)
    parent = np.empty((B, N), dtype=np.int32)
    def fill(b):
        rng = _data_rng(seed, b)
        trng = _token_rng(seed, b)
        parent[b] = random_tree_shape(N, max_depth, branching, trng)
        l = rng.normal(0.0, logit_sigma, size=(N, V))
        qb = _draft_softmax(l + rng.normal(0.0, 1.0, size=(N, V)))
        logits[b] = encode(l, dtype)
        q[b] = encode(qb, dtype)
        stored_q = decode(q[b], dtype)
        # node n's token is drawn from its parent's draft distribution
        draws = _draw_from_rows(stored_q[parent[b][1:]], trng)
        toks[b, 1:] = draws

    _per_request(B, fill)
    temp = np.full((B,), temperature, dtype=np.float32)
    uni = philox_uniforms(seed, (B, N))
    return TreeWorkload(name or f"tree_b{B}_n{N}_v{V}_{dtype}", dtype, B, N, V, max_depth,
                        logits, q, toks, parent, temp, uni)


# ----------------------------------------------------------------------------
# the five named workloads
# ----------------------------------------------------------------------------

WORKLOADS: Dict[str, dict] = {
    "linear_b1_g4_v32000_f32": dict(kind="linear", law="normal2_q05", B=1, gamma=4,
                                    V=32000, dtype=F32, seed=0),
    "linear_b64_g5_v32000_bf16": dict(kind="linear", law="normal2_tq08", B=64, gamma=5,
                                      V=32000, dtype=BF16, seed=1),
    "linear_b256_g8_v128256_bf16": dict(kind="linear", law="zipf_t07", B=256, gamma=8,
                                        V=128256, dtype=BF16, seed=2),
    "mixed_b512_g4_v152064_bf16": dict(kind="linear", law="mixed_normal3", B=512, gamma=4,
                                       V=152064, dtype=BF16, seed=3, greedy_frac=0.1,
                                       temp_range=(0.3, 1.5)),
    "tree_b32_n64_v128256_bf16": dict(kind="tree", B=32, N=64, V=128256, dtype=BF16,
                                      seed=4, max_depth=5, branching=3),
}


def make_workload(name: str, B: Optional[int] = None, V: Optional[int] = None,
                  seed_offset: int = 0):
    """Build a named workload; ``B``/``V`` override the batch or vocabulary size
    (smaller cases with the same law), ``seed_offset`` shifts every stream."""
    spec = dict(WORKLOADS[name])
    kind = spec.pop("kind")
    if B is not None:
        spec["B"] = B
    if V is not None:
        spec["V"] = V
    spec["seed"] += seed_offset
    if kind == "linear":
        law = spec.pop("law")
        return make_linear(law, name=name, **spec)
    return make_tree(name=name, **spec)
