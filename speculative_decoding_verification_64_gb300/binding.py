"""ctypes binding of ``libspecdec.so`` (argument marshalling only).

Every step of the verify path runs in the library's CUDA kernels; this module
checks tensor shapes, dtypes and devices, allocates outputs and the workspace
with torch (device memory and streams are PyTorch's only role) and passes raw
device pointers to the C ABI declared in ``include/specdec.h``.  There is no
CPU fallback: if the library is missing or a call fails, an exception says so.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspecdec.so")

F32 = 0
BF16 = 1
OK = 0
ROW_BAD_TOKEN = 1
ROW_BAD_Q = 2
ROW_NONFINITE = 4
ROW_BAD_TEMP = 8
ROW_BAD_TREE = 16
ROW_INTERNAL = 32

_lib = None

_EXPORTS = {
    "specdec_abi_version": ([], ctypes.c_int),
    "specdec_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "specdec_workspace_size": ([ctypes.c_int] * 4, ctypes.c_size_t),
    "specdec_philox_uniforms": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_ulonglong,
                                 ctypes.c_longlong, ctypes.c_void_p, ctypes.c_void_p],
                                ctypes.c_int),
    "specdec_row_entropy": ([ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p,
                             ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                             ctypes.c_void_p], ctypes.c_int),
    "specdec_verify_linear_launches": ([ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "specdec_verify_linear_path": ([ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "specdec_final_mass": ([ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int,
                            ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p],
                           ctypes.c_int),
    "specdec_row_alpha": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                           ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                           ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "specdec_path_logprob": ([ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                              ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                              ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                              ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "specdec_verify_linear_topk": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                    ctypes.c_void_p], ctypes.c_int),
    "specdec_row_stats": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                           ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                           ctypes.c_uint, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p],
                          ctypes.c_int),
    "specdec_verify_linear": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int] +
                              [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 +
                              [ctypes.c_void_p] * 7 + [ctypes.c_size_t, ctypes.c_void_p],
                              ctypes.c_int),
    "specdec_linear_finalize": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int] +
                                [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 +
                                [ctypes.c_void_p] * 7 + [ctypes.c_size_t, ctypes.c_void_p],
                                ctypes.c_int),
    "specdec_verify_tree": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int] +
                            [ctypes.c_void_p] * 4 + [ctypes.c_int] * 4 +
                            [ctypes.c_void_p] * 8 + [ctypes.c_size_t, ctypes.c_void_p],
                            ctypes.c_int),
    "specdec_verify_linear_static": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int] +
                                     [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 +
                                     [ctypes.c_void_p] * 7, ctypes.c_int),
    "specdec_linear_staging_size": ([ctypes.c_int] * 4, ctypes.c_size_t),
    "specdec_tree_staging_size": ([ctypes.c_int] * 5, ctypes.c_size_t),
    "specdec_verify_linear_host": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int] +
                                   [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 +
                                   [ctypes.c_void_p] * 7 + [ctypes.c_size_t, ctypes.c_void_p],
                                   ctypes.c_int),
    "specdec_verify_tree_host": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int] +
                                 [ctypes.c_void_p] * 4 + [ctypes.c_int] * 4 +
                                 [ctypes.c_void_p] * 8 + [ctypes.c_size_t, ctypes.c_void_p],
                                 ctypes.c_int),
    "specdec_tree_finalize": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int] +
                              [ctypes.c_void_p] * 4 + [ctypes.c_int] * 4 +
                              [ctypes.c_void_p] * 8 + [ctypes.c_size_t, ctypes.c_void_p],
                              ctypes.c_int),
}


class SpecdecError(RuntimeError):
    pass


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load ``libspecdec.so``; raises if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise SpecdecError(
            f"{p} is missing: build it with __graft_entry__.build() or "
            "`python -m speculative_decoding_verification_64_gb300.build`")
    lib = ctypes.CDLL(p)
    for name, (args, res) in _EXPORTS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    if path is None:
        _lib = lib
    return lib


def status_string(code: int) -> str:
    return load_library().specdec_status_string(int(code)).decode()


def _check(rc: int, what: str):
    if rc != OK:
        raise SpecdecError(f"{what} failed: {status_string(rc)} (code {rc})")


def dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"logits/q must be float32 or bfloat16, got {t.dtype}")


def workspace_size(B: int, rows_per_request: int, V: int, dtype: int) -> int:
    return int(load_library().specdec_workspace_size(B, rows_per_request, V, dtype))


def alloc_workspace(B: int, rows_per_request: int, V: int, dtype: int,
                    device="cuda") -> torch.Tensor:
    n = max(workspace_size(B, rows_per_request, V, dtype), 256)
    return torch.empty(n, dtype=torch.uint8, device=device)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _cuda(**tensors):
    """Every given tensor (None skipped) must live on one CUDA device, the
    current one: the library reads and writes device memory only (it has no
    CPU path), launches on the current device, and the binding passes that
    device's current stream."""
    dev = None
    for name, t in tensors.items():
        if t is None:
            continue
        if t.device.type != "cuda":
            raise ValueError(f"{name} must be a CUDA tensor, got {t.device}")
        if dev is not None and t.device != dev:
            raise ValueError(f"{name} is on {t.device}, the other arrays on {dev}")
        dev = t.device
    if dev is not None:
        cur = torch.cuda.current_device()
        if (dev.index if dev.index is not None else cur) != cur:
            raise ValueError(f"the arrays are on {dev}, but the current device is cuda:{cur}: "
                             f"call under torch.cuda.device({dev.index})")


def _req(t: torch.Tensor, name: str, dtype, shape, device):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")


@dataclasses.dataclass
class LinearOut:
    n_accepted: torch.Tensor   # int32 [B]
    out_tokens: torch.Tensor   # int32 [B, gamma+1]
    final_token: torch.Tensor  # int32 [B]
    is_bonus: torch.Tensor     # uint8 [B]
    row_status: torch.Tensor   # int32 [B]
    p_draft: Optional[torch.Tensor]  # float32 [B, gamma]

    @staticmethod
    def empty(B, gamma, device, with_p=True):
        z = dict(dtype=torch.int32, device=device)
        return LinearOut(torch.empty(B, **z), torch.empty(B, gamma + 1, **z),
                         torch.empty(B, **z), torch.empty(B, dtype=torch.uint8, device=device),
                         torch.empty(B, **z),
                         torch.empty(B, gamma, dtype=torch.float32, device=device)
                         if with_p else None)


@dataclasses.dataclass
class TreeOut:
    n_accepted: torch.Tensor   # int32 [B]
    path_nodes: torch.Tensor   # int32 [B, max_depth+1]
    out_tokens: torch.Tensor   # int32 [B, max_depth+1]
    final_token: torch.Tensor  # int32 [B]
    is_bonus: torch.Tensor     # uint8 [B]
    row_status: torch.Tensor   # int32 [B]
    p_node: Optional[torch.Tensor]   # float32 [B, N]

    @staticmethod
    def empty(B, N, max_depth, device, with_p=True):
        z = dict(dtype=torch.int32, device=device)
        D1 = max_depth + 1
        return TreeOut(torch.empty(B, **z), torch.empty(B, D1, **z), torch.empty(B, D1, **z),
                       torch.empty(B, **z), torch.empty(B, dtype=torch.uint8, device=device),
                       torch.empty(B, **z),
                       torch.empty(B, N, dtype=torch.float32, device=device) if with_p else None)


def _linear_args(logits, q, draft_tokens, temperature, uniforms, out, workspace):
    _cuda(logits=logits, q=q, draft_tokens=draft_tokens, temperature=temperature,
          uniforms=uniforms, workspace=workspace,
          **({} if out is None else {k: v for k, v in vars(out).items()}))
    B, R, V = logits.shape
    gamma = R - 1
    dev = logits.device
    dt = dtype_code(logits)
    _req(q, "q", logits.dtype, (B, gamma, V), dev)
    _req(logits, "logits", logits.dtype, (B, R, V), dev)
    _req(draft_tokens, "draft_tokens", torch.int32, (B, gamma), dev)
    _req(temperature, "temperature", torch.float32, (B,), dev)
    _req(uniforms, "uniforms", torch.float32, (B, R), dev)
    if out is None:
        out = LinearOut.empty(B, gamma, dev)
    if workspace is None:
        workspace = alloc_workspace(B, R, V, dt, dev)
    return B, gamma, V, dt, out, workspace


def verify_linear(logits: torch.Tensor, q: torch.Tensor, draft_tokens: torch.Tensor,
                  temperature: torch.Tensor, uniforms: torch.Tensor,
                  out: Optional[LinearOut] = None, workspace: Optional[torch.Tensor] = None,
                  stream=None) -> LinearOut:
    """Linear verify step (``specdec_verify_linear``) on CUDA tensors."""
    B, gamma, V, dt, out, ws = _linear_args(logits, q, draft_tokens, temperature, uniforms,
                                            out, workspace)
    lib = load_library()
    rc = lib.specdec_verify_linear(
        _ptr(logits), _ptr(q), dt, _ptr(draft_tokens), _ptr(temperature), _ptr(uniforms),
        B, gamma, V, _ptr(out.n_accepted), _ptr(out.out_tokens), _ptr(out.final_token),
        _ptr(out.is_bonus), _ptr(out.row_status), _ptr(out.p_draft), _ptr(ws), ws.numel(),
        _stream_ptr(stream))
    _check(rc, "specdec_verify_linear")
    return out


STATS_ENTROPY = 1


def verify_linear_topk(logits: torch.Tensor, q: torch.Tensor, draft_tokens: torch.Tensor,
                       temperature: torch.Tensor, uniforms: torch.Tensor, topk: int,
                       out: Optional[LinearOut] = None, workspace: Optional[torch.Tensor] = None,
                       stream=None) -> LinearOut:
    """Linear verify with the top-k residual approximation (``specdec_verify_linear_topk``)."""
    B, gamma, V, dt, out, ws = _linear_args(logits, q, draft_tokens, temperature, uniforms,
                                            out, workspace)
    rc = load_library().specdec_verify_linear_topk(
        _ptr(logits), _ptr(q), dt, _ptr(draft_tokens), _ptr(temperature), _ptr(uniforms),
        B, gamma, V, int(topk), _ptr(out.n_accepted), _ptr(out.out_tokens),
        _ptr(out.final_token), _ptr(out.is_bonus), _ptr(out.row_status), _ptr(out.p_draft),
        _ptr(ws), ws.numel(), _stream_ptr(stream))
    _check(rc, "specdec_verify_linear_topk")
    return out


def row_stats(logits: torch.Tensor, temperature: torch.Tensor, workspace: torch.Tensor,
              q: Optional[torch.Tensor] = None, draft_tokens: Optional[torch.Tensor] = None,
              entropy: bool = False, stream=None) -> None:
    """Phase 1 only (``specdec_row_stats``): logits [B, R, V] -> stage partials in the
    workspace.  For the linear form pass q and draft_tokens too (phase 2 needs the
    drafted tokens' logits and q values, gathered here).  ``entropy`` keeps the sums
    ``row_entropy`` reads."""
    _cuda(logits=logits, temperature=temperature, workspace=workspace, q=q,
          draft_tokens=draft_tokens)
    B, R, V = logits.shape
    rc = load_library().specdec_row_stats(
        _ptr(logits), _ptr(q), dtype_code(logits), _ptr(draft_tokens), _ptr(temperature), B, R, V,
        STATS_ENTROPY if entropy else 0, _ptr(workspace), workspace.numel(), _stream_ptr(stream))
    _check(rc, "specdec_row_stats")


def linear_finalize(logits, q, draft_tokens, temperature, uniforms, out: LinearOut,
                    workspace: torch.Tensor, stream=None) -> LinearOut:
    """Phase 2 of the linear form (``specdec_linear_finalize``)."""
    B, gamma, V, dt, out, ws = _linear_args(logits, q, draft_tokens, temperature, uniforms,
                                            out, workspace)
    rc = load_library().specdec_linear_finalize(
        _ptr(logits), _ptr(q), dt, _ptr(draft_tokens), _ptr(temperature), _ptr(uniforms),
        B, gamma, V, _ptr(out.n_accepted), _ptr(out.out_tokens), _ptr(out.final_token),
        _ptr(out.is_bonus), _ptr(out.row_status), _ptr(out.p_draft), _ptr(ws), ws.numel(),
        _stream_ptr(stream))
    _check(rc, "specdec_linear_finalize")
    return out


def _tree_args(logits, q, node_tokens, parent, temperature, uniforms, max_depth, out,
               workspace):
    _cuda(logits=logits, q=q, node_tokens=node_tokens, parent=parent, temperature=temperature,
          uniforms=uniforms, workspace=workspace,
          **({} if out is None else {k: v for k, v in vars(out).items()}))
    B, N, V = logits.shape
    dev = logits.device
    dt = dtype_code(logits)
    _req(q, "q", logits.dtype, (B, N, V), dev)
    _req(logits, "logits", logits.dtype, (B, N, V), dev)
    _req(node_tokens, "node_tokens", torch.int32, (B, N), dev)
    _req(parent, "parent", torch.int32, (B, N), dev)
    _req(temperature, "temperature", torch.float32, (B,), dev)
    _req(uniforms, "uniforms", torch.float32, (B, N), dev)
    if out is None:
        out = TreeOut.empty(B, N, max_depth, dev)
    if workspace is None:
        workspace = alloc_workspace(B, N, V, dt, dev)
    return B, N, V, dt, out, workspace


def verify_tree(logits, q, node_tokens, parent, temperature, uniforms, max_depth: int,
                out: Optional[TreeOut] = None, workspace: Optional[torch.Tensor] = None,
                stream=None) -> TreeOut:
    """Token-tree verify step (``specdec_verify_tree``) on CUDA tensors."""
    B, N, V, dt, out, ws = _tree_args(logits, q, node_tokens, parent, temperature, uniforms,
                                      max_depth, out, workspace)
    rc = load_library().specdec_verify_tree(
        _ptr(logits), _ptr(q), dt, _ptr(node_tokens), _ptr(parent), _ptr(temperature),
        _ptr(uniforms), B, N, V, max_depth, _ptr(out.n_accepted), _ptr(out.path_nodes),
        _ptr(out.out_tokens), _ptr(out.final_token), _ptr(out.is_bonus), _ptr(out.row_status),
        _ptr(out.p_node), _ptr(ws), ws.numel(), _stream_ptr(stream))
    _check(rc, "specdec_verify_tree")
    return out


def tree_finalize(logits, q, node_tokens, parent, temperature, uniforms, max_depth: int,
                  out: TreeOut, workspace: torch.Tensor, stream=None) -> TreeOut:
    """Phase 2 of the tree form (``specdec_tree_finalize``)."""
    B, N, V, dt, out, ws = _tree_args(logits, q, node_tokens, parent, temperature, uniforms,
                                      max_depth, out, workspace)
    rc = load_library().specdec_tree_finalize(
        _ptr(logits), _ptr(q), dt, _ptr(node_tokens), _ptr(parent), _ptr(temperature),
        _ptr(uniforms), B, N, V, max_depth, _ptr(out.n_accepted), _ptr(out.path_nodes),
        _ptr(out.out_tokens), _ptr(out.final_token), _ptr(out.is_bonus), _ptr(out.row_status),
        _ptr(out.p_node), _ptr(ws), ws.numel(), _stream_ptr(stream))
    _check(rc, "specdec_tree_finalize")
    return out


# ---------------------------------------------------------------------------
# host-buffer calls: inputs and outputs in host memory, a device staging buffer
# ---------------------------------------------------------------------------

def linear_staging_size(B: int, gamma: int, V: int, dtype: int) -> int:
    return int(load_library().specdec_linear_staging_size(B, gamma, V, dtype))


def tree_staging_size(B: int, N: int, V: int, max_depth: int, dtype: int) -> int:
    return int(load_library().specdec_tree_staging_size(B, N, V, max_depth, dtype))


def _staging(nbytes: int, staging, device) -> torch.Tensor:
    if staging is None:
        return torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device)
    if staging.device.type != "cuda" or staging.dtype != torch.uint8:
        raise ValueError("staging must be a uint8 CUDA tensor")
    _cuda(staging=staging)
    return staging


def _host_out(out, make):
    """A result container in page-locked host memory (made when None)."""
    if out is None:
        out = make()
        for k, v in vars(out).items():
            if v is not None:
                setattr(out, k, v.pin_memory())
    return out


def verify_linear_host(logits: torch.Tensor, q: torch.Tensor, draft_tokens: torch.Tensor,
                       temperature: torch.Tensor, uniforms: torch.Tensor,
                       out: Optional[LinearOut] = None, staging: Optional[torch.Tensor] = None,
                       stream=None, sync: bool = True, device="cuda") -> LinearOut:
    """Linear verify of host tensors (``specdec_verify_linear_host``): inputs and the
    returned outputs live in host memory (page-locked keeps the copies
    asynchronous); ``staging`` is device memory of ``linear_staging_size`` bytes.
    With ``sync=False`` the outputs are valid only after ``stream`` has reached
    the call."""
    cpu = torch.device("cpu")
    B, R, V = logits.shape
    gamma = R - 1
    dt = dtype_code(logits)
    _req(logits, "logits", logits.dtype, (B, R, V), cpu)
    _req(q, "q", logits.dtype, (B, gamma, V), cpu)
    _req(draft_tokens, "draft_tokens", torch.int32, (B, gamma), cpu)
    _req(temperature, "temperature", torch.float32, (B,), cpu)
    _req(uniforms, "uniforms", torch.float32, (B, R), cpu)
    out = _host_out(out, lambda: LinearOut.empty(B, gamma, cpu))
    st = _staging(linear_staging_size(B, gamma, V, dt), staging, device)
    s = stream if stream is not None else torch.cuda.current_stream(st.device)
    rc = load_library().specdec_verify_linear_host(
        _ptr(logits), _ptr(q), dt, _ptr(draft_tokens), _ptr(temperature), _ptr(uniforms),
        B, gamma, V, _ptr(out.n_accepted), _ptr(out.out_tokens), _ptr(out.final_token),
        _ptr(out.is_bonus), _ptr(out.row_status), _ptr(out.p_draft), _ptr(st), st.numel(),
        ctypes.c_void_p(s.cuda_stream))
    _check(rc, "specdec_verify_linear_host")
    if sync:
        s.synchronize()
    return out


def verify_tree_host(logits, q, node_tokens, parent, temperature, uniforms, max_depth: int,
                     out: Optional[TreeOut] = None, staging: Optional[torch.Tensor] = None,
                     stream=None, sync: bool = True, device="cuda") -> TreeOut:
    """Token-tree verify of host tensors (``specdec_verify_tree_host``); as
    ``verify_linear_host``, with ``tree_staging_size`` bytes of staging."""
    cpu = torch.device("cpu")
    B, N, V = logits.shape
    dt = dtype_code(logits)
    _req(logits, "logits", logits.dtype, (B, N, V), cpu)
    _req(q, "q", logits.dtype, (B, N, V), cpu)
    _req(node_tokens, "node_tokens", torch.int32, (B, N), cpu)
    _req(parent, "parent", torch.int32, (B, N), cpu)
    _req(temperature, "temperature", torch.float32, (B,), cpu)
    _req(uniforms, "uniforms", torch.float32, (B, N), cpu)
    out = _host_out(out, lambda: TreeOut.empty(B, N, max_depth, cpu))
    st = _staging(tree_staging_size(B, N, V, max_depth, dt), staging, device)
    s = stream if stream is not None else torch.cuda.current_stream(st.device)
    rc = load_library().specdec_verify_tree_host(
        _ptr(logits), _ptr(q), dt, _ptr(node_tokens), _ptr(parent), _ptr(temperature),
        _ptr(uniforms), B, N, V, max_depth, _ptr(out.n_accepted), _ptr(out.path_nodes),
        _ptr(out.out_tokens), _ptr(out.final_token), _ptr(out.is_bonus), _ptr(out.row_status),
        _ptr(out.p_node), _ptr(st), st.numel(), ctypes.c_void_p(s.cuda_stream))
    _check(rc, "specdec_verify_tree_host")
    if sync:
        s.synchronize()
    return out


def to_host(a, bf16: bool = False, pin: bool = True) -> torch.Tensor:
    """numpy array -> CPU tensor (page-locked by default); uint16 arrays with
    ``bf16`` are bfloat16 bits."""
    import numpy as np
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a.view(np.int16) if bf16 else a)
    t = t.view(torch.bfloat16) if bf16 else t
    return t.pin_memory() if pin else t.clone()


def linear_inputs_to_host(w, pin: bool = True):
    bf = w.dtype == "bf16"
    return (to_host(w.logits, bf, pin), to_host(w.q, bf, pin), to_host(w.draft_tokens, pin=pin),
            to_host(w.temperature, pin=pin), to_host(w.uniforms, pin=pin))


def tree_inputs_to_host(w, pin: bool = True):
    bf = w.dtype == "bf16"
    return (to_host(w.logits, bf, pin), to_host(w.q, bf, pin), to_host(w.node_tokens, pin=pin),
            to_host(w.parent, pin=pin), to_host(w.temperature, pin=pin),
            to_host(w.uniforms, pin=pin))


# ---------------------------------------------------------------------------
# host <-> device marshalling for numpy workloads
# ---------------------------------------------------------------------------

def to_device(a, device="cuda", bf16: bool = False) -> torch.Tensor:
    """numpy array -> CUDA tensor; uint16 arrays with ``bf16`` are bfloat16 bits."""
    import numpy as np
    a = np.ascontiguousarray(a)
    if bf16:
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(a)
    return t.to(device)


def linear_inputs_to_device(w, device="cuda"):
    """A ``workloads.LinearWorkload`` as CUDA tensors (logits, q, tokens, T, u)."""
    bf = w.dtype == "bf16"
    return (to_device(w.logits, device, bf), to_device(w.q, device, bf),
            to_device(w.draft_tokens, device), to_device(w.temperature, device),
            to_device(w.uniforms, device))


def tree_inputs_to_device(w, device="cuda"):
    """A ``workloads.TreeWorkload`` as CUDA tensors (logits, q, tokens, parent, T, u)."""
    bf = w.dtype == "bf16"
    return (to_device(w.logits, device, bf), to_device(w.q, device, bf),
            to_device(w.node_tokens, device), to_device(w.parent, device),
            to_device(w.temperature, device), to_device(w.uniforms, device))


def philox_uniforms(key, counter, first_word: int, n: int, device="cuda", stream=None) -> torch.Tensor:
    """float32 uniforms of the Philox4x64-10 words [first_word, first_word + n) of the
    stream (key, counter), made on the device (``specdec_philox_uniforms``).  key: 2
    words, counter: 4 words (e.g. the state of ``numpy.random.Philox(seed)``)."""
    import numpy as np
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint64).reshape(-1))
    c = np.ascontiguousarray(np.asarray(counter, dtype=np.uint64).reshape(-1))
    if k.size != 2 or c.size != 4:
        raise ValueError("key must hold 2 and counter 4 64-bit words")
    out = torch.empty(int(n), dtype=torch.float32, device=device)
    rc = load_library().specdec_philox_uniforms(k.ctypes.data, c.ctypes.data, int(first_word),
                                                int(n), _ptr(out) if n > 0 else None,
                                                _stream_ptr(stream))
    _check(rc, "specdec_philox_uniforms")
    return out



def row_entropy(logits: torch.Tensor, temperature: torch.Tensor, workspace: torch.Tensor,
                stream=None) -> torch.Tensor:
    """Entropies [B, R] of the target rows of ``logits`` from the workspace of a
    ``row_stats(..., entropy=True)`` call on those logits (``specdec_row_entropy``)."""
    _cuda(logits=logits, temperature=temperature, workspace=workspace)
    B, R, V = logits.shape
    out = torch.empty((B, R), dtype=torch.float32, device=logits.device)
    rc = load_library().specdec_row_entropy(_ptr(workspace), workspace.numel(), dtype_code(logits),
                                            _ptr(temperature), B, R, V, _ptr(out),
                                            _stream_ptr(stream))
    _check(rc, "specdec_row_entropy")
    return out


def verify_linear_launches(logits: torch.Tensor, q: torch.Tensor) -> int:
    """Kernels ``verify_linear`` launches for these inputs: 1 (a small batch, one
    launch) or 2 (the stats pass, then the draw)."""
    B, R, V = logits.shape
    return int(load_library().specdec_verify_linear_launches(B, R - 1, V, dtype_code(logits),
                                                             _ptr(logits), _ptr(q)))


def final_mass(workspace: torch.Tensor, B: int, rows_per_request: int, V: int, dtype: int,
               stream=None) -> torch.Tensor:
    """Normaliser [B] of each request's final draw in the last verify call on
    ``workspace`` (``specdec_final_mass``; NaN where nothing was drawn)."""
    _cuda(workspace=workspace)
    out = torch.empty(B, dtype=torch.float32, device=workspace.device)
    rc = load_library().specdec_final_mass(_ptr(workspace), workspace.numel(), B,
                                           rows_per_request, V, dtype,
                                           _ptr(out) if B > 0 else None, _stream_ptr(stream))
    _check(rc, "specdec_final_mass")
    return out


PATH_NONE, PATH_SMALL_ONE_LAUNCH, PATH_TWO_LAUNCHES = 0, 1, 3
PATH_KERNELS = {PATH_SMALL_ONE_LAUNCH: "small_verify_kernel", PATH_TWO_LAUNCHES: "row_stats_kernel"}


def verify_linear_path(logits: torch.Tensor, q: torch.Tensor) -> int:
    """The path ``verify_linear`` takes for these inputs (``PATH_*``): a small
    batch in one launch, or two launches."""
    B, R, V = logits.shape
    return int(load_library().specdec_verify_linear_path(B, R - 1, V, dtype_code(logits),
                                                         _ptr(logits), _ptr(q)))


def row_alpha(logits: torch.Tensor, q: torch.Tensor, temperature: torch.Tensor,
              workspace: torch.Tensor, stream=None) -> torch.Tensor:
    """Acceptance rates [B, gamma], sum_v min(p_i, q_i) of every drafted row, from the
    logits [B, gamma+1, V], q [B, gamma, V] and the workspace of a ``row_stats`` call on
    those logits (``specdec_row_alpha``)."""
    _cuda(logits=logits, q=q, temperature=temperature, workspace=workspace)
    B, R, V = logits.shape
    gamma = R - 1
    out = torch.empty((B, gamma), dtype=torch.float32, device=logits.device)
    rc = load_library().specdec_row_alpha(_ptr(logits), _ptr(q), dtype_code(logits),
                                          _ptr(temperature), B, gamma, V, _ptr(workspace),
                                          workspace.numel(), _ptr(out), _stream_ptr(stream))
    _check(rc, "specdec_row_alpha")
    return out


def path_logprob(logits: torch.Tensor, temperature: torch.Tensor, out_tokens: torch.Tensor,
                 n_accepted: torch.Tensor, workspace: torch.Tensor,
                 path_nodes: Optional[torch.Tensor] = None,
                 row_status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Log-probabilities [B] of the emitted paths (``specdec_path_logprob``)."""
    _cuda(logits=logits, temperature=temperature, out_tokens=out_tokens, n_accepted=n_accepted,
          workspace=workspace, path_nodes=path_nodes, row_status=row_status)
    B, R, V = logits.shape
    out = torch.empty(B, dtype=torch.float32, device=logits.device)
    rc = load_library().specdec_path_logprob(
        _ptr(logits), dtype_code(logits), _ptr(temperature), _ptr(out_tokens), _ptr(n_accepted),
        _ptr(path_nodes), _ptr(row_status), B, R, V, out_tokens.shape[1], _ptr(workspace),
        workspace.numel(), _ptr(out), _stream_ptr(stream))
    _check(rc, "specdec_path_logprob")
    return out
