"""The bounded waits of the tensor-core kernels, tested without any fault.

Through the diagnostic entry qspec_debug_linear_bounded a kernel's MMA
issuer is made to wait, with a short bound, on a barrier that nothing arrives
at.  The kernel must give up, leave its loops, drain what it has in flight,
free its tensor memory, report QSPEC_ERR_TIMEOUT in the status word and
return -- and the context must stay usable: the same kernel right after,
with the regular bound, is checked against the oracle (bit for bit for W4A4,
within the W4A16 tolerance) and, for W4A4, against the regular entry point.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_speculative_decoding_shared_gb300 import binding as q, synthetic as syn
from gpuhelp import assert_w4a16_close, bits, need_gpu, read_status, status

pytestmark = pytest.mark.gpu

REGULAR = 1 << 22           # the library's own bound
SHORT = 2000                # a bound the stalled wait runs through


def layer(N, K, seed, dev):
    codes, s, z = syn.weights(N, K, seed, device=dev)
    packed, sz = q.pack_weights(codes, s, z)
    rc, po, szo = oracle.pack_weights(codes.cpu().numpy(), bits(s), bits(z))
    assert rc == 0
    return packed, sz, po, szo


def run(kernel, x, xq, sx, qs, packed, sz, M, N, K, limit, stall, dev):
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
    st = status(dev)
    rc = q.qspec_debug_linear_bounded(kernel, x, xq, sx, qs, packed, sz, M, N, K, y, N, limit, stall, st)
    assert rc == q.OK, q.STATUS.get(rc, rc)
    torch.cuda.synchronize()                    # the kernel returned
    return y, read_status(st)


# (M, N, K): one CTA per tile, and (W4A16) tiles whose groups are split over
# a cluster of CTAs (few tiles: N = 300)
@pytest.mark.parametrize("M,N,K", [(24, 1000, 1024), (80, 300, 2048), (40, 2048, 4096)])
def test_w4a16_tc_timeout_exit_then_regular_call(M, N, K):
    dev = need_gpu()
    packed, sz, po, szo = layer(N, K, 90 + M, dev)
    x = syn.activations(M, K, 91).to(dev)
    _, st = run(q.KERNEL_W4A16_TC, x, None, None, None, packed, sz, M, N, K, SHORT, 1, dev)
    assert st == q.ERR_TIMEOUT
    y, st = run(q.KERNEL_W4A16_TC, x, None, None, None, packed, sz, M, N, K, REGULAR, 0, dev)
    assert st == 0
    assert_w4a16_close(y, oracle.linear_w4a16(bits(x.cpu()), po, szo), "after the timeout")


@pytest.mark.parametrize("kernel,M,N,K", [
    ("gemv", 5, 1000, 1024), ("gemv", 16, 20000, 4096),
    ("gemm", 16, 1000, 14336), ("gemm", 40, 1000, 1024), ("gemm", 130, 640, 2048),
    ("gemm", 300, 384, 1024)])
def test_w4a4_tc_timeout_exit_then_regular_call(kernel, M, N, K):
    dev = need_gpu()
    kid = q.KERNEL_W4A4_GEMV_TC if kernel == "gemv" else q.KERNEL_W4A4_TC
    packed, sz, po, szo = layer(N, K, 95 + M, dev)
    x = syn.activations(M, K, 96)
    xq, sx, qs = q.quant_act_int4(x.to(dev))
    _, st = run(kid, None, xq, sx, qs, packed, sz, M, N, K, SHORT, 1, dev)
    assert st == q.ERR_TIMEOUT
    y, st = run(kid, None, xq, sx, qs, packed, sz, M, N, K, REGULAR, 0, dev)
    assert st == 0
    rc, xqo, sxo, qso = oracle.quant_act_int4(bits(x))
    assert np.array_equal(bits(y), oracle.linear_w4a4(xqo, sxo, po, szo))
    # and the regular entry point on the same context
    assert np.array_equal(bits(q.linear_w4a4(xq, sx, qs, packed, sz)), bits(y))
