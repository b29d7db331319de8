"""The host-buffer calls (specdec_verify_linear_host, specdec_verify_tree_host):
inputs in host memory, outputs copied back to host memory.  Their outputs
must equal the device calls' on the same inputs bit for bit, and the
oracle's."""
import numpy as np
import pytest

from parity import compare_linear, compare_tree
from speculative_decoding_verification_64_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    from speculative_decoding_verification_64_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def as_numpy(out):
    return {k: v.cpu().numpy() for k, v in vars(out).items() if v is not None}


def same(a, b):
    assert a.keys() == b.keys()
    for k in a:
        assert np.array_equal(a[k], b[k], equal_nan=True), k


@pytest.mark.parametrize("name,B,V,pin", [
    ("linear_b1_g4_v32000_f32", None, None, True),       # the one-launch path
    ("linear_b1_g4_v32000_f32", None, None, False),      # pageable host memory
    ("linear_b64_g5_v32000_bf16", None, None, True),     # the two-kernel path
    ("mixed_b512_g4_v152064_bf16", 24, 4099, True),      # greedy rows, unaligned rows
])
def test_linear_host_call(oracle_lib, name, B, V, pin):
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    w = W.make_workload(name, B=B, V=V)
    host = binding.linear_inputs_to_host(w, pin=pin)
    got = as_numpy(binding.verify_linear_host(*host))
    dev = as_numpy(binding.verify_linear(*binding.linear_inputs_to_device(w)))
    torch.cuda.synchronize()
    same(got, dev)
    compare_linear(w, got, oracle_lib.verify_linear_workload(w))


def test_linear_host_call_without_p_and_on_a_stream(oracle_lib):
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    w = W.make_workload("linear_b64_g5_v32000_bf16", B=9)
    host = binding.linear_inputs_to_host(w)
    out = binding.LinearOut.empty(w.B, w.gamma, "cpu", with_p=False)
    out = binding.LinearOut(**{k: (v.pin_memory() if v is not None else None)
                               for k, v in vars(out).items()})
    s = torch.cuda.Stream()
    st = torch.empty(binding.linear_staging_size(w.B, w.gamma, w.V, binding.BF16),
                     dtype=torch.uint8, device="cuda")
    binding.verify_linear_host(*host, out=out, staging=st, stream=s, sync=False)
    s.synchronize()
    got = as_numpy(out)
    assert "p_draft" not in got
    want = oracle_lib.verify_linear_workload(w)
    compare_linear(w, got, want)


@pytest.mark.parametrize("name,B,V", [
    ("tree_b32_n64_v128256_bf16", 4, None),
    ("tree_b32_n64_v128256_bf16", 3, 5001),
])
def test_tree_host_call(oracle_lib, name, B, V):
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    w = W.make_workload(name, B=B, V=V)
    host = binding.tree_inputs_to_host(w)
    got = as_numpy(binding.verify_tree_host(*host, w.max_depth))
    dev = as_numpy(binding.verify_tree(*binding.tree_inputs_to_device(w), w.max_depth))
    torch.cuda.synchronize()
    same(got, dev)
    compare_tree(w, got, oracle_lib.verify_tree_workload(w))
