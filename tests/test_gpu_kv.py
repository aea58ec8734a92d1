"""a7 KV overwrite: CUDA path vs oracle (bit copies) and range handling."""
import numpy as np
import pytest
import torch

import oracle
from quantized_speculative_decoding_shared_gb300 import binding as q, synthetic as syn
from gpuhelp import bits, need_gpu, read_status, status

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("L,B,H,T,D,gamma,seed", [(2, 3, 2, 64, 128, 3, 0), (1, 1, 1, 8, 8, 1, 1),
                                                   (4, 5, 8, 256, 64, 8, 2),
                                                   (3, 2, 4, 100, 136, 16, 3)])
def test_kv_overwrite_matches_oracle(L, B, H, T, D, gamma, seed):
    dev = need_gpu()
    kc, vc = syn.kv_cache(L, B, H, T, D, seed)
    kn, vn = syn.kv_new(L, B, gamma, H, D, seed + 1)
    base = syn.base_positions(B, T, gamma, seed)
    nacc = torch.from_numpy(np.random.default_rng(seed).integers(0, gamma + 1, B).astype(np.int32))
    kcd, vcd = kc.to(dev), vc.to(dev)
    st = status(dev)
    q.kv_overwrite(kcd, vcd, kn.to(dev), vn.to(dev), base.to(dev), nacc.to(dev), dev_status=st)
    ko, vo = bits(kc).copy(), bits(vc).copy()
    assert oracle.kv_overwrite(ko, vo, bits(kn), bits(vn), base.numpy(), nacc.numpy(), gamma) == 0
    assert read_status(st) == 0
    assert np.array_equal(bits(kcd), ko) and np.array_equal(bits(vcd), vo)


@pytest.mark.parametrize("base,nacc", [(-1, 0), (62, 2), (0, 4), (0, -1)])
def test_kv_overwrite_range(base, nacc):
    dev = need_gpu()
    L, B, H, T, D, gamma = 2, 2, 2, 64, 16, 3
    kc, vc = syn.kv_cache(L, B, H, T, D, 5)
    kn, vn = syn.kv_new(L, B, gamma, H, D, 6)
    bp = torch.tensor([base, 5], dtype=torch.int32)
    na = torch.tensor([nacc, 1], dtype=torch.int32)
    kcd, vcd = kc.to(dev), vc.to(dev)
    st = status(dev)
    q.kv_overwrite(kcd, vcd, kn.to(dev), vn.to(dev), bp.to(dev), na.to(dev), dev_status=st)
    ko, vo = bits(kc).copy(), bits(vc).copy()
    rc = oracle.kv_overwrite(ko, vo, bits(kn), bits(vn), bp.numpy(), na.numpy(), gamma)
    assert read_status(st) == rc == q.ERR_RANGE
    assert np.array_equal(bits(kcd), ko) and np.array_equal(bits(vcd), vo)


def test_kv_overwrite_llama_cache_full_size():
    """32 layers x 16 sequences x 8 heads x 4096 positions x 128 (bf16, K and V):
    the accepted rows equal the verify rows, every other byte is unchanged."""
    dev = need_gpu()
    L, B, H, T, D, gamma = 32, 16, 8, 4096, 128, 4
    g = torch.Generator(device=dev)
    g.manual_seed(2)
    kc = torch.randn((L, B, H, T, D), generator=g, device=dev).to(torch.bfloat16)
    vc = torch.randn((L, B, H, T, D), generator=g, device=dev).to(torch.bfloat16)
    kn = torch.randn((L, B, gamma + 1, H, D), generator=g, device=dev).to(torch.bfloat16)
    vn = torch.randn((L, B, gamma + 1, H, D), generator=g, device=dev).to(torch.bfloat16)
    base = syn.base_positions(B, T, gamma, 2).to(dev)
    nacc = torch.randint(0, gamma + 1, (B,), generator=g, device=dev, dtype=torch.int32)
    k0, v0 = kc.clone(), vc.clone()
    st = status(dev)
    q.kv_overwrite(kc, vc, kn, vn, base, nacc, dev_status=st)
    assert read_status(st) == 0
    touched = torch.zeros((B, T), dtype=torch.bool, device=dev)
    for b in range(B):
        p, a = int(base[b]), int(nacc[b])
        touched[b, p:p + a + 1] = True
        for r in range(a + 1):
            assert torch.equal(kc[:, b, :, p + r].view(torch.int16), kn[:, b, r].view(torch.int16))
            assert torch.equal(vc[:, b, :, p + r].view(torch.int16), vn[:, b, r].view(torch.int16))
    mask = ~touched[None, :, None, :, None].expand_as(kc)
    assert torch.equal(kc.view(torch.int16)[mask], k0.view(torch.int16)[mask])
    assert torch.equal(vc.view(torch.int16)[mask], v0.view(torch.int16)[mask])
