"""Float64 CPU oracle for the speculative-decoding verify step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference legs of ``bench.py`` may import this package; the
product library never loads it and there is no CPU fallback through it.

The arithmetic lives in ``specdec_oracle.c`` (plain C, IEEE double, OpenMP over
independent requests); this module only builds it with gcc and marshals numpy
arrays through ctypes.  It shares no code with the CUDA library.

Parity pins: every function here is pinned in ``tests/test_oracle_pins.py``
against what the method description fixes (exact enumeration of the output
law, Lemma 1, the expected-accepted-count sums, a worked exercise, the
greedy limit, library softmax/argmax, boundary probes of the compare
conventions); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "specdec_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libspecdec_oracle.so")
_lib = None

DT_F32 = 0
DT_BF16 = 1
ROW_BAD_TOKEN = 1
ROW_BAD_Q = 2
ROW_NONFINITE = 4
ROW_BAD_TEMP = 8
ROW_BAD_TREE = 16


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (seconds).  Returns the library path."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-shared", "-fPIC", "-Wall",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        p = ctypes.c_void_p
        i = ctypes.c_int
        lib.specdec_oracle_verify_linear.argtypes = [p, p, i, p, p, p, i, i, i,
                                                     p, p, p, p, p, p, p, p, p, p]
        lib.specdec_oracle_verify_linear.restype = i
        lib.specdec_oracle_verify_tree.argtypes = [p, p, i, p, p, p, p, i, i, i, i,
                                                   p, p, p, p, p, p, p, p, p, p]
        lib.specdec_oracle_verify_tree.restype = i
        lib.specdec_oracle_num_threads.argtypes = []
        lib.specdec_oracle_num_threads.restype = i
        lib.specdec_oracle_set_threads.argtypes = [i]
        lib.specdec_oracle_set_threads.restype = None
        lib.specdec_oracle_verify_linear_topk.argtypes = [p, p, i, p, p, p, i, i, i, i,
                                                          p, p, p, p, p, p, p, p, p, p]
        lib.specdec_oracle_verify_linear_topk.restype = i
        lib.specdec_oracle_row_entropy.argtypes = [p, i, p, i, i, i, p]
        lib.specdec_oracle_row_entropy.restype = None
        lib.specdec_oracle_path_logprob.argtypes = [p, i, p, p, p, p, p, i, i, i, i, p]
        lib.specdec_oracle_path_logprob.restype = None
        lib.specdec_oracle_row_alpha.argtypes = [p, p, i, p, i, i, i, p]
        lib.specdec_oracle_row_alpha.restype = None
        u64 = ctypes.c_uint64
        lib.specdec_oracle_philox_words.argtypes = [p, p, u64, ctypes.c_int64, p]
        lib.specdec_oracle_philox_words.restype = None
        lib.specdec_oracle_philox_uniforms.argtypes = [p, p, u64, ctypes.c_int64, p]
        lib.specdec_oracle_philox_uniforms.restype = None
        _lib = lib
    return _lib


def _u64_array(x, n: int, name: str) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(x, dtype=np.uint64).reshape(-1))
    if a.size != n:
        raise ValueError(f"{name} must hold {n} 64-bit words")
    return a


def philox_words(key, counter, first: int, n: int) -> np.ndarray:
    """Raw Philox4x64-10 words [first, first + n) of the stream (key, counter)."""
    k = _u64_array(key, 2, "key")
    c = _u64_array(counter, 4, "counter")
    out = np.empty(n, dtype=np.uint64)
    _load().specdec_oracle_philox_words(k.ctypes.data, c.ctypes.data, int(first), int(n),
                                        out.ctypes.data)
    return out


def philox_uniforms(key, counter, first: int, n: int) -> np.ndarray:
    """float32 uniforms ((w >> 41) + 0.5) * 2^-23 of the words [first, first + n)."""
    k = _u64_array(key, 2, "key")
    c = _u64_array(counter, 4, "counter")
    out = np.empty(n, dtype=np.float32)
    _load().specdec_oracle_philox_uniforms(k.ctypes.data, c.ctypes.data, int(first), int(n),
                                           out.ctypes.data)
    return out


def row_entropy(logits: np.ndarray, dtype: str, temperature: np.ndarray) -> np.ndarray:
    """float64 [B, R] entropies (natural log) of the target rows of logits [B, R, V]
    (float32, or uint16 bf16 bits)."""
    B, R, V = logits.shape
    lg = np.ascontiguousarray(logits)
    tp = np.ascontiguousarray(temperature, dtype=np.float32)
    out = np.empty((B, R), dtype=np.float64)
    _load().specdec_oracle_row_entropy(lg.ctypes.data, _dtype_code(dtype), tp.ctypes.data,
                                       B, R, V, out.ctypes.data)
    return out


def row_alpha(logits: np.ndarray, q: np.ndarray, dtype: str, temperature: np.ndarray) -> np.ndarray:
    """float64 [B, gamma]: sum_v min(p_i(v), q_i(v)) of the drafted rows i < gamma, the
    acceptance probability of one draft from q_i (logits [B, gamma+1, V], q [B, gamma, V],
    float32 or uint16 bf16 bits)."""
    B, R, V = logits.shape
    gamma = R - 1
    assert q.shape == (B, gamma, V)
    lg = np.ascontiguousarray(logits)
    qq = np.ascontiguousarray(q)
    tp = np.ascontiguousarray(temperature, dtype=np.float32)
    out = np.empty((B, gamma), dtype=np.float64)
    _load().specdec_oracle_row_alpha(lg.ctypes.data, qq.ctypes.data, _dtype_code(dtype),
                                     tp.ctypes.data, B, gamma, V, out.ctypes.data)
    return out


def path_logprob(logits: np.ndarray, dtype: str, temperature: np.ndarray, out_tokens: np.ndarray,
                 n_accepted: np.ndarray, path_nodes: Optional[np.ndarray] = None,
                 row_status: Optional[np.ndarray] = None) -> np.ndarray:
    """float64 [B] log-probabilities of the emitted paths (see specdec_oracle.c)."""
    B, R, V = logits.shape
    lg = np.ascontiguousarray(logits)
    tp = np.ascontiguousarray(temperature, dtype=np.float32)
    ot = np.ascontiguousarray(out_tokens, dtype=np.int32)
    na = np.ascontiguousarray(n_accepted, dtype=np.int32)
    pn = None if path_nodes is None else np.ascontiguousarray(path_nodes, dtype=np.int32)
    rs = None if row_status is None else np.ascontiguousarray(row_status, dtype=np.int32)
    out = np.empty(B, dtype=np.float64)
    _load().specdec_oracle_path_logprob(lg.ctypes.data, _dtype_code(dtype), tp.ctypes.data,
                                        ot.ctypes.data, na.ctypes.data, _ptr(pn), _ptr(rs),
                                        B, R, V, ot.shape[1], out.ctypes.data)
    return out


def num_threads() -> int:
    """OpenMP threads the oracle's parallel loops use."""
    return int(_load().specdec_oracle_num_threads())


def set_threads(n: int) -> None:
    """Use n OpenMP threads in the oracle's parallel loops from now on."""
    _load().specdec_oracle_set_threads(int(n))


def _dtype_code(dtype: str) -> int:
    return {"f32": DT_F32, "bf16": DT_BF16}[dtype]


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _storage(a: np.ndarray, dtype: str) -> np.ndarray:
    want = np.float32 if dtype == "f32" else np.uint16
    return np.ascontiguousarray(a, dtype=want)


def verify_linear(logits, q, dtype, draft_tokens, temperature, uniforms,
                  diagnostics: bool = True) -> dict:
    """Run the oracle on host arrays shaped [B, gamma+1, V] / [B, gamma, V] / ...

    Returns numpy arrays: n_accepted, out_tokens, final_token, is_bonus,
    row_status and, with ``diagnostics``, p_draft, ratio, final_margin,
    row_diag ([B, gamma, 2]: sum min(p,q), sum max(0, p-q)) and final_mass
    (the total Z of the final draw's weights).
    """
    lib = _load()
    logits = _storage(logits, dtype)
    q = _storage(q, dtype)
    B, R, V = logits.shape
    gamma = R - 1
    if q.shape != (B, gamma, V):
        raise ValueError("q must be [B, gamma, V]")
    toks = np.ascontiguousarray(draft_tokens, dtype=np.int32).reshape(B, gamma)
    temp = np.ascontiguousarray(temperature, dtype=np.float32).reshape(B)
    uni = np.ascontiguousarray(uniforms, dtype=np.float32).reshape(B, R)
    out = dict(
        n_accepted=np.empty(B, np.int32), out_tokens=np.empty((B, R), np.int32),
        final_token=np.empty(B, np.int32), is_bonus=np.empty(B, np.uint8),
        row_status=np.empty(B, np.int32))
    if diagnostics:
        out.update(p_draft=np.empty((B, gamma)), ratio=np.empty((B, gamma)),
                   final_margin=np.empty(B), row_diag=np.empty((B, gamma, 2)),
                   final_mass=np.empty(B))
    rc = lib.specdec_oracle_verify_linear(
        _ptr(logits), _ptr(q), _dtype_code(dtype), _ptr(toks), _ptr(temp), _ptr(uni),
        B, gamma, V, _ptr(out["n_accepted"]), _ptr(out["out_tokens"]),
        _ptr(out["final_token"]), _ptr(out["is_bonus"]), _ptr(out["row_status"]),
        _ptr(out.get("p_draft")), _ptr(out.get("ratio")), _ptr(out.get("final_margin")),
        _ptr(out.get("row_diag")), _ptr(out.get("final_mass")))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return out


def verify_linear_topk(logits, q, dtype, draft_tokens, temperature, uniforms, topk: int) -> dict:
    """The linear step with the top-k residual (see specdec_oracle.c): the same
    outputs as ``verify_linear`` plus p_draft, ratio, final_margin, tv [B] (total
    variation between the exact residual law and the top-k one; NaN where no
    residual draw happened) and final_mass (the total of the drawn weights)."""
    lib = _load()
    logits = _storage(logits, dtype)
    q = _storage(q, dtype)
    B, R, V = logits.shape
    gamma = R - 1
    toks = np.ascontiguousarray(draft_tokens, dtype=np.int32).reshape(B, gamma)
    temp = np.ascontiguousarray(temperature, dtype=np.float32).reshape(B)
    uni = np.ascontiguousarray(uniforms, dtype=np.float32).reshape(B, R)
    out = dict(
        n_accepted=np.empty(B, np.int32), out_tokens=np.empty((B, R), np.int32),
        final_token=np.empty(B, np.int32), is_bonus=np.empty(B, np.uint8),
        row_status=np.empty(B, np.int32), p_draft=np.empty((B, gamma)),
        ratio=np.empty((B, gamma)), final_margin=np.empty(B), tv=np.empty(B),
        final_mass=np.empty(B))
    rc = lib.specdec_oracle_verify_linear_topk(
        _ptr(logits), _ptr(q), _dtype_code(dtype), _ptr(toks), _ptr(temp), _ptr(uni),
        B, gamma, V, int(topk), _ptr(out["n_accepted"]), _ptr(out["out_tokens"]),
        _ptr(out["final_token"]), _ptr(out["is_bonus"]), _ptr(out["row_status"]),
        _ptr(out["p_draft"]), _ptr(out["ratio"]), _ptr(out["final_margin"]), _ptr(out["tv"]),
        _ptr(out["final_mass"]))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return out


def verify_linear_topk_workload(w, topk: int) -> dict:
    """Top-k residual oracle on a ``workloads.LinearWorkload``."""
    return verify_linear_topk(w.logits, w.q, w.dtype, w.draft_tokens, w.temperature,
                              w.uniforms, topk)


def verify_tree(logits, q, dtype, node_tokens, parent, temperature, uniforms,
                max_depth: int, diagnostics: bool = True) -> dict:
    """Run the tree oracle on host arrays [B, N, V] / [B, N] / [B]."""
    lib = _load()
    logits = _storage(logits, dtype)
    q = _storage(q, dtype)
    B, N, V = logits.shape
    if q.shape != (B, N, V):
        raise ValueError("q must be [B, N, V]")
    toks = np.ascontiguousarray(node_tokens, dtype=np.int32).reshape(B, N)
    par = np.ascontiguousarray(parent, dtype=np.int32).reshape(B, N)
    temp = np.ascontiguousarray(temperature, dtype=np.float32).reshape(B)
    uni = np.ascontiguousarray(uniforms, dtype=np.float32).reshape(B, N)
    D1 = max_depth + 1
    out = dict(
        n_accepted=np.empty(B, np.int32), path_nodes=np.empty((B, D1), np.int32),
        out_tokens=np.empty((B, D1), np.int32), final_token=np.empty(B, np.int32),
        is_bonus=np.empty(B, np.uint8), row_status=np.empty(B, np.int32))
    if diagnostics:
        out.update(p_node=np.empty((B, N)), test_margin=np.empty(B),
                   final_margin=np.empty(B), final_mass=np.empty(B))
    rc = lib.specdec_oracle_verify_tree(
        _ptr(logits), _ptr(q), _dtype_code(dtype), _ptr(toks), _ptr(par), _ptr(temp),
        _ptr(uni), B, N, V, max_depth, _ptr(out["n_accepted"]), _ptr(out["path_nodes"]),
        _ptr(out["out_tokens"]), _ptr(out["final_token"]), _ptr(out["is_bonus"]),
        _ptr(out["row_status"]), _ptr(out.get("p_node")), _ptr(out.get("test_margin")),
        _ptr(out.get("final_margin")), _ptr(out.get("final_mass")))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return out


def verify_linear_workload(w, diagnostics: bool = True) -> dict:
    """Oracle on a ``workloads.LinearWorkload``."""
    return verify_linear(w.logits, w.q, w.dtype, w.draft_tokens, w.temperature,
                         w.uniforms, diagnostics=diagnostics)


def verify_tree_workload(w, diagnostics: bool = True) -> dict:
    """Oracle on a ``workloads.TreeWorkload``."""
    return verify_tree(w.logits, w.q, w.dtype, w.node_tokens, w.parent, w.temperature,
                       w.uniforms, w.max_depth, diagnostics=diagnostics)
