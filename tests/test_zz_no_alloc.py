"""The allocation-free sampled verification (qspec_verify_sample_noalloc).

It exists for callers that cannot allocate device memory -- code running
while a CUDA graph is captured, or a plugin without an allocator -- and keeps
its scratch in a fixed array inside the library.  It must give exactly the
results of qspec_verify_sample with a caller-provided workspace.

This file is collected last on purpose, and must pass both on its own in a
fresh process and after every other test.
"""
import numpy as np
import pytest
import torch

from quantized_speculative_decoding_shared_gb300 import binding as q, synthetic as syn
from gpuhelp import need_gpu, read_status, status

pytestmark = pytest.mark.gpu


def run_both(P, Q, d, seed, rnd, dev):
    B, g1, V = P.shape
    gamma = g1 - 1
    n_ref = torch.full((B,), -7, dtype=torch.int32, device=dev)
    o_ref = torch.full((B, gamma + 1), -7, dtype=torch.int32, device=dev)
    ws = q.verify_workspace(B, gamma, V, dev)
    st_ref = status(dev)
    rc = q.qspec_verify_sample(P, Q, d, B, gamma, V, seed, rnd, n_ref, o_ref, ws, ws.numel(),
                               st_ref)
    assert rc == q.OK
    n_na = torch.full((B,), -9, dtype=torch.int32, device=dev)
    o_na = torch.full((B, gamma + 1), -9, dtype=torch.int32, device=dev)
    st_na = status(dev)
    rc = q.qspec_verify_sample_noalloc(P, Q, d, B, gamma, V, seed, rnd, n_na, o_na, st_na)
    assert rc == q.OK
    assert read_status(st_ref) == 0 and read_status(st_na) == 0
    assert np.array_equal(n_na.cpu().numpy(), n_ref.cpu().numpy())
    assert np.array_equal(o_na.cpu().numpy(), o_ref.cpu().numpy())
    return n_na.cpu().numpy()


def test_noalloc_matches_workspace_entry_point_two_calls_in_a_row():
    dev = need_gpu()
    # batch 16, gamma 4, vocab 128256 (target N(0, 3^2), draft = target + N(0, 0.5^2))
    P, Q, d = syn.logits_noisy_draft(16, 4, 128256, 2, device=dev)
    n1 = run_both(P, Q, d, seed=11, rnd=0, dev=dev)
    # second call in a row reuses the same scratch array: results must not depend on
    # what the first call left there
    P2, Q2, d2 = syn.logits_noisy_draft(3, 2, 1000, 5, device=dev)
    run_both(P2, Q2, d2, seed=12, rnd=1, dev=dev)
    n3 = run_both(P, Q, d, seed=11, rnd=0, dev=dev)
    assert np.array_equal(n1, n3)


def test_noalloc_one_block_per_row_path_on_dirty_scratch():
    dev = need_gpu()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    # B (2 gamma + 1) rows at or above two per SM take the one-block-per-row
    # statistics kernel (no clearing of the scratch); run it right after calls
    # of the chunked path, which leave their maxima and sums in the array
    B, gamma, V = 64, 4, 32000
    assert B * (2 * gamma + 1) >= 2 * sms
    assert q.qspec_verify_workspace_bytes(B, gamma, V) <= q.NOALLOC_SCRATCH_BYTES
    Ps, Qs, ds = syn.logits_noisy_draft(16, 4, 128256, 7, device=dev)
    run_both(Ps, Qs, ds, seed=3, rnd=2, dev=dev)
    P, Q, d = syn.logits_noisy_draft(B, gamma, V, 8, device=dev)
    n1 = run_both(P, Q, d, seed=21, rnd=5, dev=dev)
    run_both(Ps, Qs, ds, seed=4, rnd=3, dev=dev)
    n2 = run_both(P, Q, d, seed=21, rnd=5, dev=dev)
    assert np.array_equal(n1, n2)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    dev = need_gpu()
    B, gamma, V = 4096, 16, 600000
    assert q.qspec_verify_workspace_bytes(B, gamma, V) > q.NOALLOC_SCRATCH_BYTES
    one = torch.zeros(1, dtype=torch.int32, device=dev)
    rc = q.qspec_verify_sample_noalloc(one, one, one, B, gamma, V, 0, 0, one, one, None)
    assert rc == q.ERR_WORKSPACE
