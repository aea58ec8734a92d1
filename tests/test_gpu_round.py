"""A whole QSPEC round (gamma draft steps, the verify pass, sampled
verification, the KV overwrite) captured into a CUDA graph and replayed,
against the oracle: the last outputs of every call site, the accepted
counts and tokens of the round id, and the KV cache after the overwrite."""
import numpy as np
import pytest
import torch

import oracle
from quantized_speculative_decoding_shared_gb300 import synthetic as syn
from quantized_speculative_decoding_shared_gb300.round import QspecRound
from gpuhelp import assert_w4a16_close, bits, need_gpu

pytestmark = pytest.mark.gpu

# a small model of the same structure: 2 layers, stacked q/k/v and gate/up
TINY = dict(hidden=256, q=256, kv=128, inter=384, vocab=1000, layers=2, kv_heads=2, head_dim=64)


def oracle_weights(rnd_obj, layer, j, N, K):
    # the same generator on the same device as the round's weights
    codes, s, z = syn.weights(N, K, rnd_obj.weight_seed(layer, j), device=rnd_obj.dev)
    rc, po, szo = oracle.pack_weights(codes.cpu().numpy(), bits(s), bits(z))
    assert rc == 0
    return po, szo


def oracle_w4a4(x, po, szo):
    rc, xq, sx, qs = oracle.quant_act_int4(bits(x))
    assert rc == 0
    y, _ = oracle.linear_w4a4(xq, sx, po, szo, want_I=True)
    return y


@pytest.mark.parametrize("B,gamma,rnd", [(2, 2, 5), (3, 4, 11)])
def test_captured_round_matches_oracle(B, gamma, rnd):
    dev = need_gpu()
    r = QspecRound(TINY, B, gamma, T=64, seed=3, device=dev, outliers=0.01)
    kc0, vc0 = bits(r.kc).copy(), bits(r.vc).copy()
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        r.run(rnd)                                  # eager round: kernel attributes, status
    assert r.device_status() == 0
    eager_out, eager_n = r.out.clone(), r.n_acc.clone()
    # reset the cache to its initial contents, then replay the captured round twice
    r.kc.copy_(torch.from_numpy(kc0.view(np.int16)).view(torch.bfloat16).to(dev))
    r.vc.copy_(torch.from_numpy(vc0.view(np.int16)).view(torch.bfloat16).to(dev))
    g = r.capture(rnd, stream)
    with torch.cuda.stream(stream):
        g.replay()
        g.replay()
    torch.cuda.synchronize()
    assert r.device_status() == 0
    assert torch.equal(r.out, eager_out) and torch.equal(r.n_acc, eager_n)

    L, g1 = r.L, gamma - 1
    # last draft step, last layer: each linear's output; the LM head of the last step
    for j, (name, N, K) in enumerate(r.linears):
        po, szo = oracle_weights(r, L - 1, j, N, K)
        want = oracle_w4a4(r.xd[name][g1, L - 1].cpu(), po, szo)
        assert np.array_equal(bits(r.yd[name]), want), "draft %s" % name
        want16 = oracle.linear_w4a16(bits(r.xv[name][L - 1].cpu()), po, szo)
        assert_w4a16_close(r.yv[name], want16, "verify %s" % name)
    po, szo = oracle_weights(r, -1, 0, r.V, r.hidden)
    assert np.array_equal(bits(r.yd_lm), oracle_w4a4(r.xd_lm[g1].cpu(), po, szo)), "draft LM head"
    assert_w4a16_close(r.yv_lm, oracle.linear_w4a16(bits(r.xv_lm.cpu()), po, szo), "verify LM head")
    # acceptance of round `rnd`
    st, n_acc, out = oracle.verify_sample(bits(r.P).reshape(B, gamma + 1, r.V),
                                          bits(r.Q).reshape(B, gamma, r.V), r.drafts.cpu().numpy(),
                                          r.verify_seed, rnd)
    assert st == 0
    assert np.array_equal(r.n_acc.cpu().numpy(), n_acc) and np.array_equal(r.out.cpu().numpy(), out)
    # the cache after the overwrite (applied twice by the two replays: the same rows)
    kc, vc = kc0.copy(), vc0.copy()
    assert oracle.kv_overwrite(kc, vc, bits(r.kn), bits(r.vn), r.base.cpu().numpy(), n_acc, gamma) == 0
    assert np.array_equal(bits(r.kc), kc) and np.array_equal(bits(r.vc), vc)
