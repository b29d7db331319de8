"""Device Philox4x64-10 uniforms (specdec_philox_uniforms) against the oracle's
statement of the generator, bit for bit, and as the source of a verify step."""
import numpy as np
import pytest

from speculative_decoding_verification_64_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    from speculative_decoding_verification_64_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


CASES = [
    ([0, 0], [0, 0, 0, 0], 0, 1),
    ([0, 0], [0, 0, 0, 0], 0, 4),
    ([0x0123456789ABCDEF, 0xFEDCBA9876543210], [2**64 - 3, 7, 0, 0], 5, 37),   # counter carry
    ([2**64 - 1, 1], [2**64 - 1, 2**64 - 1, 2**64 - 1, 2**64 - 5], 3, 1000),  # three carries
    ([12345, 678], [9, 0, 0, 0], 2**64 - 10, 10),                              # last words of the range
    ([1, 2], [3, 4, 5, 6], 1001, 300_001),                                     # many blocks, ragged ends
]


@pytest.mark.parametrize("key,counter,first,n", CASES)
def test_device_uniforms_match_the_oracle(oracle_lib, key, counter, first, n):
    from speculative_decoding_verification_64_gb300 import binding
    got = binding.philox_uniforms(key, counter, first, n).cpu().numpy()
    want = oracle_lib.philox_uniforms(key, counter, first, n)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_device_uniforms_drive_the_verify_step_like_the_host_ones():
    """The workloads draw their uniforms from numpy.random.Philox(seed); the device
    generator started from the same state gives the same buffer, hence the same
    verify outputs."""
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    w = W.make_workload("linear_b256_g8_v128256_bf16", B=12, V=20008)
    seed = W.WORKLOADS["linear_b256_g8_v128256_bf16"]["seed"]
    st = np.random.Philox(seed).state["state"]
    dev = binding.philox_uniforms(st["key"], st["counter"], 0, w.uniforms.size).reshape(w.uniforms.shape)
    assert np.array_equal(dev.cpu().numpy().view(np.uint32), w.uniforms.view(np.uint32))
    logits, q, toks, temp, uni = binding.linear_inputs_to_device(w)
    a = binding.verify_linear(logits, q, toks, temp, uni)
    b = binding.verify_linear(logits, q, toks, temp, dev)
    torch.cuda.synchronize()
    for k in ("n_accepted", "out_tokens", "final_token", "is_bonus", "row_status", "p_draft"):
        assert torch.equal(getattr(a, k), getattr(b, k)), k
