"""a1 pack and a2 activation quantiser: CUDA path vs oracle, bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from quantized_speculative_decoding_shared_gb300 import binding as q, synthetic as syn
from gpuhelp import bits, need_gpu, read_status, status

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,K,seed", [(512, 512, 0), (3, 128, 5), (1000, 384, 6),
                                      (14336, 4096, 1), (4096, 14336, 2), (17, 18944, 3)])
def test_pack_bit_exact(N, K, seed):
    dev = need_gpu()
    codes, s, z = syn.weights(N, K, seed)
    st = status(dev)
    packed, sz = q.pack_weights(codes.to(dev), s.to(dev), z.to(dev), dev_status=st)
    rc, po, szo = oracle.pack_weights(codes.numpy(), bits(s), bits(z))
    assert rc == 0 and read_status(st) == 0
    assert np.array_equal(packed.cpu().numpy(), po)
    assert np.array_equal(sz.cpu().numpy().view(np.uint32), szo)


@pytest.mark.parametrize("case,code", [("code16", q.ERR_RANGE), ("z_half", q.ERR_ZERO_POINT),
                                       ("z_16", q.ERR_ZERO_POINT), ("z_neg", q.ERR_ZERO_POINT),
                                       ("s_nan", q.ERR_NONFINITE)])
def test_pack_device_errors(case, code):
    dev = need_gpu()
    codes, s, z = syn.weights(64, 256, 9)
    if case == "code16":
        codes[7, 33] = 16
    elif case == "z_half":
        z[3, 1] = 2.5
    elif case == "z_16":
        z[0, 0] = 16.0
    elif case == "z_neg":
        z[5, 1] = -1.0
    else:
        s[2, 0] = float("nan")
    st = status(dev)
    q.pack_weights(codes.to(dev), s.to(dev), z.to(dev), dev_status=st)
    rc, _, _ = oracle.pack_weights(codes.numpy(), bits(s), bits(z))
    assert read_status(st) == code == rc


@pytest.mark.parametrize("M,K,outliers,seed", [(4, 512, 0.0, 0), (1, 4096, 0.01, 1),
                                               (5, 14336, 0.01, 2), (37, 384, 0.0, 3),
                                               (80, 4096, 0.0, 4), (4096, 4096, 0.01, 5),
                                               (3, 18944, 0.0, 6), (2, 128, 0.0, 7)])
def test_quant_act_bit_exact(M, K, outliers, seed):
    dev = need_gpu()
    x = syn.activations(M, K, seed, outlier_frac=outliers)
    st = status(dev)
    xq, sx, qs = q.quant_act_int4(x.to(dev), dev_status=st)
    rc, xqo, sxo, qso = oracle.quant_act_int4(bits(x))
    assert rc == 0 and read_status(st) == 0
    assert np.array_equal(xq.cpu().numpy(), xqo)
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), sxo.view(np.uint32))
    assert np.array_equal(qs.cpu().numpy(), qso)


def test_quant_act_edge_values():
    dev = need_gpu()
    rng = np.random.default_rng(11)
    M, K = 6, 512
    x = torch.from_numpy(rng.normal(0, 1, (M, K)).astype(np.float32))
    x[0] = 0.0                                   # all-zero groups
    x[1] *= 1e-38                                # bf16 subnormal range
    x[2] *= 1e37                                 # near the top of the range
    x[3, :128] = 3.0                             # constant group: every q = 7
    x[4, ::2] = 0.5                              # many exact ties after scaling
    x[4, 0] = 3.5
    x[4, 128] = 7.0                              # sx = 1: every other element an exact
    x[4, 129:256] = (torch.arange(1, 128) % 14) - 6.5   # half-integer tie (to even)
    x[5, :128] = torch.arange(128) - 64.0        # exact integers
    xb = x.to(torch.bfloat16)
    st = status(dev)
    xq, sx, qs = q.quant_act_int4(xb.to(dev), dev_status=st)
    rc, xqo, sxo, qso = oracle.quant_act_int4(bits(xb))
    assert rc == 0 and read_status(st) == 0
    assert np.array_equal(xq.cpu().numpy(), xqo)
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), sxo.view(np.uint32))
    assert np.array_equal(qs.cpu().numpy(), qso)


def test_quant_act_nonfinite_status():
    dev = need_gpu()
    x = syn.activations(2, 256, 3)
    x[1, 200] = float("inf")
    st = status(dev)
    q.quant_act_int4(x.to(dev), dev_status=st)
    assert read_status(st) == q.ERR_NONFINITE == oracle.quant_act_int4(bits(x))[0]


def test_quant_act_every_scale_near_ties():
    """One group per positive bf16 amax (every normal value, and a few
    subnormal ones, whose tiny scale takes the IEEE division): the group holds
    amax and the bf16 values at and up to two steps either side of every
    half-integer multiple (k + 1/2) sx, the quotients that decide rounding
    ties; the codes, scales and sums match the oracle bit for bit."""
    dev = need_gpu()
    rng = np.random.default_rng(12)
    ab = np.concatenate([np.arange(0x0080, 0x7F80, dtype=np.uint32), np.array([0x0001, 0x0040, 0x007F], np.uint32)])
    amax = (ab << 16).view(np.float32)
    sx = (amax / np.float32(7)).astype(np.float32)
    h = ((np.arange(-7, 7, dtype=np.float32) + np.float32(0.5))[None, :] * sx[:, None]).astype(np.float32)
    hb = torch.from_numpy(h).to(torch.bfloat16).view(torch.int16).numpy().astype(np.int32)
    mag, sign = hb & 0x7FFF, hb & 0x8000
    near = np.concatenate([((mag + d).clip(0, 0x7F7F) | sign) for d in (-2, -1, 0, 1, 2)], axis=1)   # [n][70]
    nearf = ((near.astype(np.uint32) & 0xFFFF) << 16).view(np.float32)
    nearf = np.where(np.abs(nearf) <= amax[:, None], nearf, 0.0).astype(np.float32)
    fill = (rng.uniform(-1, 1, (len(ab), 128 - 1 - nearf.shape[1])) * amax[:, None]).astype(np.float32)
    grp = np.concatenate([amax[:, None], nearf, fill], axis=1)                       # [n][128]
    G = 256
    n_rows = (len(ab) + G - 1) // G
    pad = np.zeros((n_rows * G - len(ab), 128), np.float32)
    x = torch.from_numpy(np.concatenate([grp, pad]).reshape(n_rows, G * 128)).to(torch.bfloat16)
    assert np.abs(x.float().numpy().reshape(-1, 128)[: len(ab), 0] - amax).max() == 0
    st = status(dev)
    xq, sx_g, qs = q.quant_act_int4(x.to(dev), dev_status=st)
    rc, xqo, sxo, qso = oracle.quant_act_int4(bits(x))
    assert rc == 0 and read_status(st) == 0
    assert np.array_equal(sx_g.cpu().numpy().view(np.uint32), sxo.view(np.uint32))
    assert np.array_equal(qs.cpu().numpy(), qso)
    assert np.array_equal(xq.cpu().numpy(), xqo)
