"""Helpers for the GPU parity tests (the tests call the CUDA path through the
C ABI via the binding, and the oracle on the host, on the same inputs)."""
import numpy as np
import pytest
import torch

from quantized_speculative_decoding_shared_gb300 import binding, synthetic as syn

W4A16_RTOL = 1e-2   # |gpu - ref| <= 1e-2 (1 + |ref|) against the fp64 value


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_speculative_decoding_shared_gb300 import build as qbuild
    qbuild.build()
    binding.load_library()
    return torch.device("cuda:0")


def status(dev):
    return torch.zeros(1, dtype=torch.int32, device=dev)


def read_status(st):
    torch.cuda.synchronize()
    return int(st.item())


bits = syn.bits16


def assert_w4a16_close(got_bf16, ref, what=""):
    got = got_bf16.float().cpu().numpy() if isinstance(got_bf16, torch.Tensor) else got_bf16
    err = np.abs(got - ref)
    bound = W4A16_RTOL * (1.0 + np.abs(ref))
    bad = err > bound
    assert not bad.any(), "%s: %d / %d outside tolerance, worst excess %g" % (
        what, int(bad.sum()), bad.size, float((err - bound).max()))


def sample_points(M, N, n, seed):
    rng = np.random.default_rng(seed)
    ms = rng.integers(0, M, n).astype(np.int32)
    ns = rng.integers(0, N, n).astype(np.int32)
    # always include the corners and the ragged edges
    ms[:4] = [0, M - 1, 0, M - 1]
    ns[:4] = [0, N - 1, N - 1, 0]
    return ms, ns
