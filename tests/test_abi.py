"""The C-ABI library loads and exports every symbol include/specdec.h declares.

Runs without a GPU: only host-side entry points are called (version, status
strings, workspace sizing, and argument checks that return before any CUDA
call).
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specdec.h")


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_64_gb300 import build, binding
    build.build()
    return binding.load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(specdec_[a-z_]+)\s*\(", src)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("specdec_verify_linear", "specdec_verify_tree", "specdec_workspace_size",
                 "specdec_status_string", "specdec_row_stats", "specdec_linear_finalize",
                 "specdec_tree_finalize", "specdec_abi_version"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert lib.specdec_abi_version() == 1
    for code in range(5):
        s = lib.specdec_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.specdec_status_string(99).decode() == "unknown status"


def test_workspace_size_is_a_pure_function(lib):
    from speculative_decoding_verification_64_gb300.binding import BF16, F32
    a = lib.specdec_workspace_size(256, 9, 128256, BF16)
    assert a == lib.specdec_workspace_size(256, 9, 128256, BF16)
    assert a > 0 and a % 256 == 0
    assert a >= 256 * 9 * 16                      # at least one partial per row
    assert lib.specdec_workspace_size(0, 9, 128256, BF16) == 0
    assert lib.specdec_workspace_size(-1, 9, 128256, BF16) == 0
    assert lib.specdec_workspace_size(4, 9, 0, BF16) == 0
    assert lib.specdec_workspace_size(4, 9, 100, 7) == 0
    assert lib.specdec_workspace_size(4, 9, (1 << 21) + 1, F32) == 0
    assert lib.specdec_workspace_size(1, 5, 32000, F32) > 0


def test_argument_checks_before_any_device_work(lib):
    from speculative_decoding_verification_64_gb300.binding import BF16
    N = None
    vl = lib.specdec_verify_linear
    # B = 0 is a no-op
    assert vl(N, N, BF16, N, N, N, 0, 8, 1000, N, N, N, N, N, N, N, 0, N) == 0
    # null pointers
    assert vl(N, N, BF16, N, N, N, 4, 8, 1000, N, N, N, N, N, N, N, 0, N) == 1
    # gamma out of range
    assert vl(N, N, BF16, N, N, N, 4, 0, 1000, N, N, N, N, N, N, N, 0, N) == 1
    assert vl(N, N, BF16, N, N, N, 4, 33, 1000, N, N, N, N, N, N, N, 0, N) == 2
    # dtype
    assert vl(N, N, 5, N, N, N, 4, 4, 1000, N, N, N, N, N, N, N, 0, N) == 1
    # vocabulary limit
    assert vl(N, N, BF16, N, N, N, 4, 4, (1 << 21) + 1, N, N, N, N, N, N, N, 0, N) == 2
    # workspace too small (all other pointers are non-null dummies that are never touched)
    d = ctypes.c_void_p(16)
    assert vl(d, d, BF16, d, d, d, 4, 4, 1000, d, d, d, d, d, N, d, 8, N) == 3
    assert vl(d, d, BF16, d, d, d, 4, 4, 1000, d, d, d, d, d, N, N, 1 << 20, N) == 3
    vt = lib.specdec_verify_tree
    assert vt(N, N, BF16, N, N, N, N, 0, 64, 1000, 5, N, N, N, N, N, N, N, N, 0, N) == 0
    assert vt(N, N, BF16, N, N, N, N, 2, 0, 1000, 5, N, N, N, N, N, N, N, N, 0, N) == 1
    assert vt(N, N, BF16, N, N, N, N, 2, 2000, 1000, 5, N, N, N, N, N, N, N, N, 0, N) == 2
    assert vt(N, N, BF16, N, N, N, N, 2, 64, 1000, 65, N, N, N, N, N, N, N, N, 0, N) == 2
    rs = lib.specdec_row_stats
    assert rs(N, N, BF16, N, N, 0, 9, 1000, 0, N, 0, N) == 0
    assert rs(N, N, BF16, N, N, 2, 9, 1000, 0, N, 0, N) == 1
    # q without draft tokens (or the reverse) is rejected
    assert rs(d, d, BF16, N, d, 2, 9, 1000, 0, d, 1 << 30, N) == 1
    assert rs(d, N, BF16, d, d, 2, 9, 1000, 0, d, 1 << 30, N) == 1
    # unknown flag bits
    assert rs(d, N, BF16, N, d, 2, 9, 1000, 2, d, 1 << 30, N) == 1


def test_misaligned_arrays_are_refused_before_any_device_work(lib):
    """Each device array must start on a multiple of its element size (2 bytes
    for bf16 data, 4 for float32 data and the int32 / float32 arrays); the call
    returns INVALID_ARG (1) before launching anything.  With every array
    aligned and no workspace, the workspace check is the one that fails (3)."""
    from speculative_decoding_verification_64_gb300.binding import BF16, F32
    P = ctypes.c_void_p
    N = None
    a, two, odd = P(0x10000), P(0x10002), P(0x10001)   # never dereferenced

    def linear_args(**kw):
        names = ["logits", "q", "dtype", "tokens", "temperature", "uniforms", "B", "gamma",
                 "V", "n_accepted", "out_tokens", "final_token", "is_bonus", "row_status",
                 "p_draft", "workspace", "ws_bytes", "stream"]
        vals = dict(logits=a, q=a, dtype=BF16, tokens=a, temperature=a, uniforms=a, B=4,
                    gamma=4, V=1000, n_accepted=a, out_tokens=a, final_token=a, is_bonus=a,
                    row_status=a, p_draft=N, workspace=N, ws_bytes=0, stream=N)
        vals.update(kw)
        return [vals[n] for n in names]

    vl = lib.specdec_verify_linear
    assert vl(*linear_args()) == 3
    assert vl(*linear_args(logits=two, q=two)) == 3          # bf16: 2-byte alignment suffices
    assert vl(*linear_args(is_bonus=odd)) == 3               # uint8: any address
    assert vl(*linear_args(logits=odd)) == 1
    assert vl(*linear_args(q=odd)) == 1
    assert vl(*linear_args(dtype=F32, logits=two)) == 1
    assert vl(*linear_args(dtype=F32, q=two)) == 1
    for name in ("tokens", "temperature", "uniforms", "n_accepted", "out_tokens",
                 "final_token", "row_status", "p_draft"):
        assert vl(*linear_args(**{name: two})) == 1, name
    tk = lib.specdec_verify_linear_topk
    args = linear_args(logits=odd)
    assert tk(*(args[:9] + [32] + args[9:])) == 1
    args = linear_args()
    assert tk(*(args[:9] + [32] + args[9:])) == 3

    def tree_args(**kw):
        names = ["logits", "q", "dtype", "tokens", "parent", "temperature", "uniforms", "B", "N",
                 "V", "max_depth", "n_accepted", "path_nodes", "out_tokens", "final_token",
                 "is_bonus", "row_status", "p_node", "workspace", "ws_bytes", "stream"]
        vals = dict(logits=a, q=a, dtype=BF16, tokens=a, parent=a, temperature=a, uniforms=a,
                    B=2, N=64, V=1000, max_depth=5, n_accepted=a, path_nodes=a, out_tokens=a,
                    final_token=a, is_bonus=odd, row_status=a, p_node=N, workspace=N,
                    ws_bytes=0, stream=N)
        vals.update(kw)
        return [vals[n] for n in names]

    vt = lib.specdec_verify_tree
    assert vt(*tree_args()) == 3
    for name in ("logits", "q"):
        assert vt(*tree_args(**{name: odd})) == 1, name
    for name in ("tokens", "parent", "temperature", "uniforms", "n_accepted", "path_nodes",
                 "out_tokens", "final_token", "row_status", "p_node"):
        assert vt(*tree_args(**{name: two})) == 1, name

    rs = lib.specdec_row_stats
    assert rs(a, a, BF16, a, a, 2, 9, 1000, 0, N, 0, N) == 3
    assert rs(odd, a, BF16, a, a, 2, 9, 1000, 0, N, 0, N) == 1
    assert rs(a, a, BF16, two, a, 2, 9, 1000, 0, N, 0, N) == 1
    assert rs(a, N, F32, N, two, 2, 9, 1000, 0, N, 0, N) == 1
    ra = lib.specdec_row_alpha
    assert ra(a, a, BF16, a, 2, 8, 1000, N, 0, a, N) == 3
    assert ra(a, odd, BF16, a, 2, 8, 1000, N, 0, a, N) == 1
    assert ra(a, a, BF16, a, 2, 8, 1000, N, 0, two, N) == 1
    lp = lib.specdec_path_logprob
    assert lp(a, BF16, a, a, a, N, N, 2, 9, 1000, 9, N, 0, a, N) == 3
    assert lp(odd, BF16, a, a, a, N, N, 2, 9, 1000, 9, N, 0, a, N) == 1
    assert lp(a, BF16, a, a, a, two, N, 2, 9, 1000, 9, N, 0, a, N) == 1
    en = lib.specdec_row_entropy
    assert en(N, 0, BF16, a, 2, 9, 1000, a, N) == 3
    assert en(N, 0, BF16, a, 2, 9, 1000, two, N) == 1


def test_binding_refuses_to_run_without_the_library(tmp_path):
    from speculative_decoding_verification_64_gb300 import binding
    with pytest.raises(binding.SpecdecError):
        binding.load_library(str(tmp_path / "missing.so"))


def test_oracle_is_not_reachable_from_the_product_package():
    pkg = os.path.join(ROOT, "speculative_decoding_verification_64_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "specdec_oracle" not in text, f


def test_philox_argument_checks(lib):
    import numpy as np
    N = None
    key = np.zeros(2, dtype=np.uint64)
    ctr = np.zeros(4, dtype=np.uint64)
    k, c = key.ctypes.data, ctr.ctypes.data
    d = ctypes.c_void_p(16)
    ph = lib.specdec_philox_uniforms
    assert ph(k, c, 0, 0, N, N) == 0                    # n = 0 is a no-op
    assert ph(k, c, 0, -1, d, N) == 1                   # n < 0
    assert ph(N, c, 0, 4, d, N) == 1                    # null key
    assert ph(k, N, 0, 4, d, N) == 1                    # null counter
    assert ph(k, c, 0, 4, N, N) == 1                    # null output
    assert ph(k, c, 2**64 - 3, 4, d, N) == 1            # word range beyond 2^64
    assert ph(k, c, 0, (1 << 40) + 1, d, N) == 2        # beyond SPECDEC_MAX_UNIFORMS


def test_entropy_and_path_logprob_argument_checks(lib):
    from speculative_decoding_verification_64_gb300.binding import BF16
    N = None
    d = ctypes.c_void_p(16)
    en = lib.specdec_row_entropy
    assert en(N, 0, BF16, N, 0, 9, 1000, N, N) == 0               # B = 0
    assert en(d, 1 << 30, BF16, N, 2, 9, 1000, d, N) == 1         # no temperature
    assert en(d, 8, BF16, d, 2, 9, 1000, d, N) == 3               # workspace too small
    assert en(d, 1 << 30, 7, d, 2, 9, 1000, d, N) == 1            # dtype
    pl = lib.specdec_path_logprob
    assert pl(N, BF16, N, N, N, N, N, 0, 9, 1000, 9, N, 0, N, N) == 0
    assert pl(d, BF16, d, d, d, N, N, 2, 9, 1000, 0, d, 1 << 30, d, N) == 1   # path_len 0
    assert pl(d, BF16, d, N, d, N, N, 2, 9, 1000, 9, d, 1 << 30, d, N) == 1   # no tokens
    assert pl(d, BF16, d, d, d, N, N, 2, 9, 1000, 9, d, 8, d, N) == 3         # workspace


def test_topk_argument_checks(lib):
    from speculative_decoding_verification_64_gb300.binding import BF16
    N = None
    vt = lib.specdec_verify_linear_topk
    assert vt(N, N, BF16, N, N, N, 0, 8, 1000, 16, N, N, N, N, N, N, N, 0, N) == 0   # B = 0
    assert vt(N, N, BF16, N, N, N, 4, 8, 1000, 0, N, N, N, N, N, N, N, 0, N) == 1    # topk < 1
    assert vt(N, N, BF16, N, N, N, 4, 8, 1000, 1025, N, N, N, N, N, N, N, 0, N) == 2  # > max
    assert vt(N, N, BF16, N, N, N, 4, 8, 1000, 16, N, N, N, N, N, N, N, 0, N) == 1   # nulls


def test_row_alpha_argument_checks(lib):
    from speculative_decoding_verification_64_gb300.binding import BF16
    N = None
    d = ctypes.c_void_p(16)
    ra = lib.specdec_row_alpha
    assert ra(N, N, BF16, N, 0, 8, 1000, N, 0, N, N) == 0               # B = 0
    assert ra(d, d, BF16, d, 2, 0, 1000, d, 1 << 30, d, N) == 1         # gamma 0
    assert ra(d, d, BF16, d, 2, 33, 1000, d, 1 << 30, d, N) == 1        # gamma above the maximum
    assert ra(d, N, BF16, d, 2, 8, 1000, d, 1 << 30, d, N) == 1         # no q
    assert ra(d, d, BF16, d, 2, 8, 1000, d, 1 << 30, N, N) == 1         # no output
    assert ra(d, d, BF16, d, 2, 8, 1000, d, 8, d, N) == 3               # workspace too small
    assert ra(d, d, 7, d, 2, 8, 1000, d, 1 << 30, d, N) == 1            # dtype


def test_verify_linear_launches_query(lib):
    from speculative_decoding_verification_64_gb300.binding import BF16, F32
    N = None
    vl = lib.specdec_verify_linear_launches
    assert vl(0, 4, 1000, BF16, N, N) == 0                     # B = 0
    assert vl(1, 0, 1000, BF16, N, N) == -1                    # gamma 0
    assert vl(1, 4, 1000, 7, N, N) == -1                       # dtype
    # unaligned rows (7 bf16 elements = 14 bytes) take the two kernels
    assert vl(1, 4, 7, BF16, ctypes.c_void_p(256), ctypes.c_void_p(512)) == 2
    # a large batch takes the two kernels
    assert vl(4096, 8, 128256, BF16, ctypes.c_void_p(256), ctypes.c_void_p(512)) == 2


def test_verify_linear_path_query(lib):
    from speculative_decoding_verification_64_gb300 import binding
    BF16, N = binding.BF16, None
    vp = lib.specdec_verify_linear_path
    a, b = ctypes.c_void_p(256), ctypes.c_void_p(512)
    assert vp(0, 4, 1000, BF16, N, N) == binding.PATH_NONE
    assert vp(1, 0, 1000, BF16, N, N) == -1
    assert vp(1, 4, 32000, BF16, a, b) == binding.PATH_SMALL_ONE_LAUNCH
    assert vp(256, 8, 128256, BF16, a, b) == binding.PATH_TWO_LAUNCHES
    assert vp(1, 4, 32000, BF16, a, ctypes.c_void_p(514)) == binding.PATH_TWO_LAUNCHES  # unaligned q


def test_staging_sizes(lib):
    from speculative_decoding_verification_64_gb300.binding import BF16, F32
    ls, ts, ws = lib.specdec_linear_staging_size, lib.specdec_tree_staging_size, \
        lib.specdec_workspace_size
    B, g, V = 1, 4, 32000
    # the inputs, the outputs (each region 256-byte aligned) and the workspace
    inputs = B * (g + 1) * V * 4 + B * g * V * 4
    assert ls(B, g, V, F32) >= inputs + ws(B, g + 1, V, F32)
    assert ls(B, g, V, F32) <= inputs + ws(B, g + 1, V, F32) + 11 * 256 + 4096
    assert ls(B, g, V, F32) % 256 == 0
    assert ls(256, 8, 128256, BF16) > ls(128, 8, 128256, BF16) > 0
    for bad in ((0, 4, 1000, BF16), (-1, 4, 1000, BF16), (2, 0, 1000, BF16), (2, 33, 1000, BF16),
                (2, 4, 0, BF16), (2, 4, 1000, 7), (2, 4, (1 << 21) + 1, F32)):
        assert ls(*bad) == 0, bad
    n = 64
    assert ts(32, n, 128256, 8, BF16) >= 2 * 32 * n * 128256 * 2 + ws(32, n, 128256, BF16)
    for bad in ((0, n, 1000, 8, BF16), (2, 0, 1000, 8, BF16), (2, 2000, 1000, 8, BF16),
                (2, n, 1000, -1, BF16), (2, n, 1000, 65, BF16), (2, n, 1000, 8, 7)):
        assert ts(*bad) == 0, bad


def test_host_call_argument_checks(lib):
    from speculative_decoding_verification_64_gb300.binding import BF16
    N = None
    d = ctypes.c_void_p(16)
    vl = lib.specdec_verify_linear_host
    assert vl(N, N, BF16, N, N, N, 0, 8, 1000, N, N, N, N, N, N, N, 0, N) == 0     # B = 0
    assert vl(N, N, BF16, N, N, N, 0, 8, (1 << 21) + 1, N, N, N, N, N, N, N, 0, N) == 2
    assert vl(N, N, BF16, N, N, N, 4, 8, 1000, N, N, N, N, N, N, N, 0, N) == 1     # nulls
    assert vl(d, d, BF16, d, d, d, 4, 0, 1000, d, d, d, d, d, N, d, 1 << 30, N) == 1
    assert vl(d, d, BF16, d, d, d, 4, 33, 1000, d, d, d, d, d, N, d, 1 << 30, N) == 2
    assert vl(d, d, 5, d, d, d, 4, 4, 1000, d, d, d, d, d, N, d, 1 << 30, N) == 1
    # staging missing, too small or unaligned: nothing is copied
    need = lib.specdec_linear_staging_size(4, 4, 1000, BF16)
    assert vl(d, d, BF16, d, d, d, 4, 4, 1000, d, d, d, d, d, N, N, need, N) == 3
    assert vl(d, d, BF16, d, d, d, 4, 4, 1000, d, d, d, d, d, N, d, need - 1, N) == 3
    assert vl(d, d, BF16, d, d, d, 4, 4, 1000, d, d, d, d, d, N, ctypes.c_void_p(24), need,
              N) == 3
    vt = lib.specdec_verify_tree_host
    assert vt(N, N, BF16, N, N, N, N, 0, 64, 1000, 5, N, N, N, N, N, N, N, N, 0, N) == 0
    assert vt(N, N, BF16, N, N, N, N, 2, 64, 1000, 5, N, N, N, N, N, N, N, N, 0, N) == 1
    assert vt(N, N, BF16, N, N, N, N, 2, 0, 1000, 5, N, N, N, N, N, N, N, N, 0, N) == 1
    assert vt(N, N, BF16, N, N, N, N, 2, 2000, 1000, 5, N, N, N, N, N, N, N, N, 0, N) == 2
    assert vt(N, N, BF16, N, N, N, N, 2, 64, 1000, 65, N, N, N, N, N, N, N, N, 0, N) == 2
    need = lib.specdec_tree_staging_size(2, 64, 1000, 5, BF16)
    assert vt(d, d, BF16, d, d, d, d, 2, 64, 1000, 5, d, d, d, d, d, d, N, d, need - 1,
              N) == 3


def test_binding_refuses_host_tensors_for_device_calls():
    """The device calls take CUDA tensors only: host tensors are refused in the
    binding, before the library is called (the host-buffer calls are the ones
    for host memory)."""
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    B, g, V = 2, 3, 50
    logits = torch.zeros(B, g + 1, V)
    q = torch.full((B, g, V), 1.0 / V)
    toks = torch.zeros(B, g, dtype=torch.int32)
    temp = torch.ones(B)
    uni = torch.full((B, g + 1), 0.5)
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding.verify_linear(logits, q, toks, temp, uni)
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding.verify_linear_topk(logits, q, toks, temp, uni, 4)
    par = torch.tensor([[-1, 0, 0, 1]] * B, dtype=torch.int32)
    tl = torch.zeros(B, 4, V)
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding.verify_tree(tl, tl, torch.zeros(B, 4, dtype=torch.int32), par, temp,
                            torch.full((B, 4), 0.5), 3)
    ws = torch.empty(1 << 16, dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding.row_stats(logits, temp, ws)
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding.row_alpha(logits, q, temp, ws)
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding.row_entropy(logits, temp, ws)


def test_static_entry_point_checks_sizes_like_the_workspace_one(lib):
    """specdec_verify_linear_static runs the size checks of specdec_verify_linear
    first, so both entry points return the same code for the same sizes, B = 0
    included (no device work: every case returns before any CUDA call)."""
    from speculative_decoding_verification_64_gb300.binding import BF16
    N = None
    vl, vs = lib.specdec_verify_linear, lib.specdec_verify_linear_static
    cases = [
        (0, 8, 1000, BF16),          # B = 0: a no-op
        (0, 0, 1000, BF16),          # B = 0, gamma = 0: still a bad gamma
        (0, 33, 1000, BF16),         # gamma beyond the ABI's limit
        (0, 4, 1000, 7),             # unknown dtype
        (0, 4, (1 << 21) + 1, BF16),  # vocabulary beyond the limit
        (-1, 4, 1000, BF16),
        ((1 << 31) - 1, 8, 1000, BF16),  # B * (gamma + 1) past INT_MAX
    ]
    for B, g, V, dt in cases:
        want = vl(N, N, dt, N, N, N, B, g, V, N, N, N, N, N, N, N, 0, N)
        got = vs(N, N, dt, N, N, N, B, g, V, N, N, N, N, N, N, N)
        assert got == want, (B, g, V, dt, got, want)
    assert vs(N, N, BF16, N, N, N, 0, 0, 1000, N, N, N, N, N, N, N) == 1
    assert vs(N, N, BF16, N, N, N, (1 << 31) - 1, 8, 1000, N, N, N, N, N, N, N) == 2


def test_binding_refuses_tensors_off_the_current_device(monkeypatch):
    """The library launches on the current device and the binding passes that
    device's current stream: tensors on another device are refused before the
    library is called.  Checked with stand-in tensors (no GPU here)."""
    import torch
    from speculative_decoding_verification_64_gb300 import binding

    class Fake:
        def __init__(self, index):
            self.device = torch.device("cuda", index)

    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    binding._cuda(a=Fake(0), b=Fake(0), c=None)
    with pytest.raises(ValueError, match="current device"):
        binding._cuda(a=Fake(1), b=Fake(1))
    with pytest.raises(ValueError, match="the other arrays"):
        binding._cuda(a=Fake(0), b=Fake(1))
