"""SpecQuant Q8 (next-3): FP8 E4M3 weights derived from the FP16 parent,
per-token E4M3 activations (both bit-exact against the oracle) and the FP8
linear on the tensor cores (within 1e-2 (1 + |ref|) of the oracle's fp64
value of the same sum)."""
import numpy as np
import pytest
import torch

import oracle
from quantized_speculative_decoding_shared_gb300 import binding as q, synthetic as syn
from gpuhelp import assert_w4a16_close, need_gpu, read_status, status

pytestmark = pytest.mark.gpu


def parent(N, K, seed, dev):
    """An FP16 parent weight matrix: N(0, 0.02^2), a few rows scaled up, one
    zero row (when there are several)."""
    g = torch.Generator().manual_seed(seed)
    w = torch.randn((N, K), generator=g) * 0.02
    w[:: max(1, N // 7)] *= 40.0
    if N > 3:
        w[N // 2] = 0.0
    return w.to(torch.float16)


def bits(t):
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("N,K", [(1, 128), (37, 640), (300, 4096), (129, 14336)])
def test_weight_derivation_bit_exact(N, K):
    dev = need_gpu()
    w16 = parent(N, K, N + K, dev)
    st = status(dev)
    w8, s8 = q.quant_weights_fp8(w16.to(dev), dev_status=st)
    assert read_status(st) == 0
    rc, w8o, s8o = oracle.quant_weights_fp8(bits(w16))
    assert rc == 0
    assert np.array_equal(w8.cpu().numpy(), w8o)
    assert np.array_equal(s8.cpu().numpy().view(np.uint32), s8o.view(np.uint32))


@pytest.mark.parametrize("M,K", [(1, 128), (5, 4096), (17, 1152), (64, 14336)])
def test_activation_quant_bit_exact(M, K):
    dev = need_gpu()
    x = syn.activations(M, K, M * 7 + K, outlier_frac=0.01)
    if M > 2:
        x[1] = 0.0
    st = status(dev)
    xq, sa = q.quant_act_fp8(x.to(dev), dev_status=st)
    assert read_status(st) == 0
    rc, xqo, sao = oracle.quant_act_fp8(bits(x))
    assert rc == 0
    assert np.array_equal(xq.cpu().numpy(), xqo)
    assert np.array_equal(sa.cpu().numpy().view(np.uint32), sao.view(np.uint32))


def test_quantisers_flag_nonfinite():
    dev = need_gpu()
    w16 = parent(8, 256, 3, dev)
    w16[2, 5] = float("inf")
    st = status(dev)
    q.quant_weights_fp8(w16.to(dev), dev_status=st)
    assert read_status(st) == q.ERR_NONFINITE
    x = syn.activations(3, 256, 4)
    x[1, 9] = float("nan")
    st = status(dev)
    q.quant_act_fp8(x.to(dev), dev_status=st)
    assert read_status(st) == q.ERR_NONFINITE


# decode (verify) shapes and larger M, ragged tiles, long K
@pytest.mark.parametrize("M,N,K", [(1, 64, 128), (5, 1000, 1024), (5, 6144, 4096), (16, 300, 14336),
                                   (17, 129, 640), (33, 700, 2048), (80, 1024, 4096), (130, 257, 1152)])
def test_fp8_linear_parity(M, N, K):
    dev = need_gpu()
    w16 = parent(N, K, 11 + N, dev)
    x = syn.activations(M, K, 12 + M, outlier_frac=0.01)
    st = status(dev)
    w8, s8 = q.quant_weights_fp8(w16.to(dev), dev_status=st)
    xq, sa = q.quant_act_fp8(x.to(dev), dev_status=st)
    y = q.linear_fp8(xq, sa, w8, s8, dev_status=st)
    assert read_status(st) == 0
    _, w8o, s8o = oracle.quant_weights_fp8(bits(w16))
    _, xqo, sao = oracle.quant_act_fp8(bits(x))
    ref = oracle.linear_fp8(xqo, sao, w8o, s8o)
    assert_w4a16_close(y, ref, "fp8 M=%d N=%d K=%d" % (M, N, K))


def test_fp8_linear_qwen_lm_head_m5():
    """The Qwen2.5-7B LM head (152064 x 3584) at the verify shape M = 5,
    checked on sampled outputs (the oracle computes the sampled columns)."""
    dev = need_gpu()
    N, K, M = 152064, 3584, 5
    g = torch.Generator(device=dev).manual_seed(5)
    w16 = (torch.randn((N, K), generator=g, device=dev) * 0.02).to(torch.float16)
    x = syn.activations(M, K, 13, outlier_frac=0.01)
    w8, s8 = q.quant_weights_fp8(w16)
    xq, sa = q.quant_act_fp8(x.to(dev))
    y = q.linear_fp8(xq, sa, w8, s8).float().cpu().numpy()
    cols = np.random.default_rng(6).integers(0, N, 512)
    cols[:2] = [0, N - 1]
    _, w8o, s8o = oracle.quant_weights_fp8(bits(w16[torch.from_numpy(cols).to(dev)]))
    _, xqo, sao = oracle.quant_act_fp8(bits(x))
    assert np.array_equal(w8o, w8[torch.from_numpy(cols).to(dev)].cpu().numpy())
    ref = oracle.linear_fp8(xqo, sao, w8o, s8o)
    assert_w4a16_close(y[:, cols], ref, "fp8 LM head")
