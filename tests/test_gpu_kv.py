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


# ----------------------------------------------------------------- a4 + a7: the k/v projection
# writing the cache from its epilogue (qspec_linear_w4a16_kv)
def _expected_caches(kc, vc, ref, B, gamma, H, D, c0, base, nacc):
    """The oracle's caches: the oracle's W4A16 values (fp64, rounded to bf16)
    of the K and V columns, placed by the oracle's KV overwrite."""
    M = B * (gamma + 1)
    rows = torch.from_numpy(ref).to(torch.bfloat16)                      # [M][N]
    kn = rows[:, c0:c0 + H * D].reshape(1, B, gamma + 1, H, D)
    vn = rows[:, c0 + H * D:c0 + 2 * H * D].reshape(1, B, gamma + 1, H, D)
    ko, vo = bits(kc).copy()[None], bits(vc).copy()[None]               # one layer
    assert oracle.kv_overwrite(ko, vo, bits(kn), bits(vn), base, nacc, gamma) == 0
    return ko[0], vo[0]


# (B, gamma, K): 15 verify rows (the small-M kernel) and 80 rows (the tensor-core kernel);
# n_acc given, or unknown (all gamma + 1 rows written)
@pytest.mark.parametrize("B,gamma,K,given", [(3, 4, 1024, True), (3, 4, 1024, False), (16, 4, 2048, True),
                                             (16, 4, 2048, False), (2, 7, 512, True)])
def test_w4a16_kv_epilogue_matches_oracle(B, gamma, K, given):
    from gpuhelp import W4A16_RTOL
    dev = need_gpu()
    H, D, T, c0 = 2, 128, 96, 384
    N = c0 + 2 * H * D
    M = B * (gamma + 1)
    codes, s, z = syn.weights(N, K, 21 + B)
    packed, sz = q.pack_weights(codes.to(dev), s.to(dev), z.to(dev))
    rc, po, szo = oracle.pack_weights(codes.numpy(), bits(s), bits(z))
    x = syn.activations(M, K, 22 + B, outlier_frac=0.01)
    kc, vc = syn.kv_cache(1, B, H, T, D, 23)
    kc, vc = kc[0].contiguous(), vc[0].contiguous()                    # [B][H][T][D]
    base = syn.base_positions(B, T, gamma, 24)
    nacc = torch.from_numpy(np.random.default_rng(B).integers(0, gamma + 1, B).astype(np.int32))
    kcd, vcd = kc.to(dev), vc.to(dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    st = status(dev)
    rc = q.qspec_linear_w4a16_kv(x.to(dev), K, packed, sz, M, N, K, y, N, c0, H, D, T, gamma, kcd, vcd,
                                 base.to(dev), nacc.to(dev) if given else None, st)
    assert rc == q.OK and read_status(st) == 0
    ref = oracle.linear_w4a16(bits(x), po, szo)
    # y as the plain W4A16 linear
    got = y.float().cpu().numpy()
    assert np.all(np.abs(got - ref) <= W4A16_RTOL * (1 + np.abs(ref)))
    written = nacc.numpy() if given else np.full(B, gamma, np.int32)
    ko, vo = _expected_caches(kc, vc, ref, B, gamma, H, D, c0, base.numpy(), written)
    for cache_gpu, cache_orc, col in ((kcd, ko, c0), (vcd, vo, c0 + H * D)):
        g = bits(cache_gpu)
        touched = np.zeros(g.shape, bool)
        for b in range(B):
            touched[b, :, base[b]:base[b] + written[b] + 1, :] = True
        # untouched positions: bit for bit the old cache (the oracle's copy of it)
        assert np.array_equal(g[~touched], cache_orc[~touched])
        # written positions: the W4A16 tolerance against the oracle's values,
        # and exactly the call's own outputs (placement)
        gv = torch.from_numpy(g.view(np.int16)).view(torch.bfloat16).float().numpy()
        for b in range(B):
            for r in range(written[b] + 1):
                m = b * (gamma + 1) + r
                refr = ref[m, col:col + H * D].reshape(H, D)
                sl = gv[b, :, base[b] + r, :]
                assert np.all(np.abs(sl - refr) <= W4A16_RTOL * (1 + np.abs(refr)))
                assert np.array_equal(g[b, :, base[b] + r, :],
                                      bits(y[m, col:col + H * D].reshape(H, D)))


def test_w4a16_kv_epilogue_range():
    dev = need_gpu()
    B, gamma, K, H, D, T, c0 = 2, 3, 256, 1, 64, 16, 0
    N = 2 * H * D
    M = B * (gamma + 1)
    codes, s, z = syn.weights(N, K, 31)
    packed, sz = q.pack_weights(codes.to(dev), s.to(dev), z.to(dev))
    x = syn.activations(M, K, 32).to(dev)
    kc, vc = syn.kv_cache(1, B, H, T, D, 33)
    kcd, vcd = kc[0].contiguous().to(dev), vc[0].contiguous().to(dev)
    before = bits(kcd).copy()
    base = torch.tensor([13, 2], dtype=torch.int32, device=dev)        # 13 + 3 >= 16: sequence 0 out of range
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    st = status(dev)
    rc = q.qspec_linear_w4a16_kv(x, K, packed, sz, M, N, K, y, N, c0, H, D, T, gamma, kcd, vcd, base, None, st)
    assert rc == q.OK and read_status(st) == q.ERR_RANGE
    after = bits(kcd)
    assert np.array_equal(after[0], before[0])                        # untouched
    assert not np.array_equal(after[1, :, 2:6], before[1, :, 2:6])    # written
    # host checks: M not a multiple of gamma + 1, columns past N
    one = torch.zeros(1, dtype=torch.int32, device=dev)
    assert q.qspec_linear_w4a16_kv(x, K, packed, sz, M - 1, N, K, y, N, c0, H, D, T, gamma, kcd, vcd, base, None,
                                   None) == q.ERR_SHAPE
    assert q.qspec_linear_w4a16_kv(x, K, packed, sz, M, N, K, y, N, 1, H, D, T, gamma, kcd, vcd, base, None,
                                   None) == q.ERR_SHAPE
