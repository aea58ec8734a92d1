"""a3 W4A4 (bit-exact: outputs and INT32 group accumulators) and a4 W4A16
(within 1e-2 (1 + |ref|) of fp64): CUDA path vs oracle on the same inputs."""
import numpy as np
import pytest
import torch

import oracle
from quantized_speculative_decoding_shared_gb300 import binding as q, synthetic as syn
from gpuhelp import assert_w4a16_close, bits, need_gpu, read_status, sample_points, status

pytestmark = pytest.mark.gpu


def make_layer(N, K, seed, dev):
    codes, s, z = syn.weights(N, K, seed, device=dev)
    packed, sz = q.pack_weights(codes, s, z)
    rc, po, szo = oracle.pack_weights(codes.cpu().numpy(), bits(s), bits(z))
    assert rc == 0
    assert np.array_equal(packed.cpu().numpy(), po)
    return packed, sz, po, szo


def run_w4a4(x, packed, sz, dev, want_I=True):
    st = status(dev)
    xq, sx, qs = q.quant_act_int4(x.to(dev), dev_status=st)
    out = q.linear_w4a4(xq, sx, qs, packed, sz, want_I=want_I, dev_status=st)
    assert read_status(st) == 0
    rc, xqo, sxo, qso = oracle.quant_act_int4(bits(x))
    assert np.array_equal(xq.cpu().numpy(), xqo)
    return out, xqo, sxo


# ----------------------------------------------------------------- small, full compare
@pytest.mark.parametrize("M,N,K,seed", [
    (4, 512, 512, 0),                     # the single-layer case: K = N = 512, M = gamma + 1 = 4
    (1, 16, 128, 1), (2, 100, 384, 2), (3, 1000, 1024, 3), (5, 48, 3072, 4),
    (8, 33, 256, 5), (9, 64, 512, 6), (13, 17, 128, 7), (16, 256, 640, 8), (17, 40, 384, 9),
    (33, 31, 1152, 10),
    # W4A16 with the groups of a tile split over a cluster of 4 or 8 CTAs
    # (uneven splits included), W4A4 on the tensor cores
    (80, 300, 1024, 11), (50, 1000, 2048, 12), (24, 130, 1152, 13), (128, 257, 4096, 14),
    # large K (one token per warp-MMA CTA): W4A4 at 13..32 tokens on the
    # tensor cores, fewer on the warp-MMA kernel with one CTA column per token
    (5, 150, 14336, 15), (16, 200, 14336, 16), (32, 130, 18944, 17), (4, 70, 14336, 18),
    (12, 90, 14336, 19), (13, 90, 18944, 20),
    # prefill-sized W4A4 (256 tokens and more) on its own kernel, ragged
    (300, 130, 1152, 21)])
def test_small_full_compare(M, N, K, seed):
    dev = need_gpu()
    packed, sz, po, szo = make_layer(N, K, seed, dev)
    x = syn.activations(M, K, seed + 100)
    (y4, I), xqo, sxo = run_w4a4(x, packed, sz, dev)
    y4o, Io = oracle.linear_w4a4(xqo, sxo, po, szo, want_I=True)
    assert np.array_equal(I.cpu().numpy(), Io)
    assert np.array_equal(bits(y4), y4o)
    y16 = q.linear_w4a16(x.to(dev), packed, sz)
    ref = oracle.linear_w4a16(bits(x), po, szo)
    assert_w4a16_close(y16, ref, "w4a16 M=%d N=%d K=%d" % (M, N, K))


@pytest.mark.parametrize("M", [3, 40, 300])
def test_extreme_codes_and_unit_scales(M):
    """codes and activations at the ends of their ranges: |I| reaches 128*7*15
    (warp-MMA, decode-batch tensor-core and prefill tensor-core W4A4 paths)."""
    dev = need_gpu()
    N, K = 160 if M > 3 else 64, 512
    G = K // 128
    rng = np.random.default_rng(0)
    codes = torch.from_numpy(rng.choice([0, 15], (N, K)).astype(np.uint8))
    z = torch.from_numpy(rng.choice([0.0, 15.0], (N, G))).to(torch.float16)
    s = torch.ones((N, G), dtype=torch.float16)
    x = torch.from_numpy(rng.choice([-7.0, 7.0], (M, K)).astype(np.float32))
    # worst case built in: row 0 all codes 15 with z = 0, token 0 all +7 -> I = 128 * 7 * 15;
    # row 1 all codes 0 with z = 15 -> I = -128 * 7 * 15
    codes[0], codes[1] = 15, 0
    z[0], z[1] = 0.0, 15.0
    x[0] = 7.0
    x = x.to(torch.bfloat16)
    packed, sz = q.pack_weights(codes.to(dev), s.to(dev), z.to(dev))
    rc, po, szo = oracle.pack_weights(codes.numpy(), bits(s), bits(z))
    (y4, I), xqo, sxo = run_w4a4(x, packed, sz, dev)
    y4o, Io = oracle.linear_w4a4(xqo, sxo, po, szo, want_I=True)
    assert Io[0, 0].max() == 128 * 7 * 15 and Io[0, 1].min() == -128 * 7 * 15
    assert np.array_equal(I.cpu().numpy(), Io) and np.array_equal(bits(y4), y4o)
    y16 = q.linear_w4a16(x.to(dev), packed, sz)
    assert_w4a16_close(y16, oracle.linear_w4a16(bits(x), po, szo), "extreme")


# ----------------------------------------------------------------- full-size layer shapes
LLAMA = syn.layer_linears(syn.LLAMA3_8B)
QWEN = syn.layer_linears(syn.QWEN25_7B)


def sampled_compare(M_list, shapes, seed, dev, outliers=0.0, w4a4=True, w4a16=True, points=384):
    for idx, (name, N, K) in enumerate(shapes):
        packed, sz, po, szo = make_layer(N, K, seed * 10 + idx, dev)
        for M in M_list:
            x = syn.activations(M, K, seed * 100 + idx, outlier_frac=outliers)
            ms, ns = sample_points(M, N, points, seed + idx + M)
            if w4a4:
                y4, xqo, sxo = run_w4a4(x, packed, sz, dev, want_I=False)
                y4o = oracle.linear_w4a4_points(xqo, sxo, po, szo, ms, ns)
                assert np.array_equal(bits(y4)[ms, ns], y4o), (name, M)
            if w4a16:
                y16 = q.linear_w4a16(x.to(dev), packed, sz)
                ref = oracle.linear_w4a16_points(bits(x), po, szo, ms, ns)
                assert_w4a16_close(y16.float().cpu().numpy()[ms, ns], ref, "%s M=%d" % (name, M))


def test_llama_decode_draft_m1_verify_m5():
    """Llama-3-8B-shaped decode linears, 1 % outlier channels x20: W4A4 draft
    at M = 1, W4A16 verify at M = gamma + 1 = 5."""
    dev = need_gpu()
    sampled_compare([1], LLAMA, 1, dev, outliers=0.01, w4a16=False)
    sampled_compare([5], LLAMA, 1, dev, outliers=0.01, w4a4=False)


def test_llama_batch16_verify_m80_with_lm_head():
    dev = need_gpu()
    sampled_compare([80], LLAMA + [("lm_head", 128256, 4096)], 2, dev, w4a4=False)


@pytest.mark.parametrize("gamma", [2, 4, 8])
def test_qwen_batch32(gamma):
    dev = need_gpu()
    shapes = QWEN if gamma == 4 else [QWEN[0], QWEN[6]]
    sampled_compare([32], shapes, 3, dev, w4a16=False)
    sampled_compare([32 * (gamma + 1)], shapes, 3, dev, w4a4=False)


def test_prefill_m4096():
    dev = need_gpu()
    shapes = [("gate_proj", 14336, 4096), ("down_proj", 4096, 14336)]
    sampled_compare([4096], shapes, 4, dev)


# ----------------------------------------------------------------- decode M, many row tiles
# Shapes with at least one 128-row tile per SM take the tensor-memory GEMV
# path at 3 <= M <= 16 (the one-token kernel and the warp-MMA kernel below
# that); a ragged last tile, an odd group count and every token count class
# (1, 2, 4, 8 and 16 token columns) are covered.
@pytest.mark.parametrize("M,K,seed", [(1, 1152, 20), (2, 2048, 21), (3, 1152, 22), (5, 2048, 23), (8, 1152, 24),
                                      (12, 1152, 25), (16, 2048, 26)])
def test_decode_many_tiles_full_compare(M, K, seed):
    dev = need_gpu()
    N = 19456 + 77
    packed, sz, po, szo = make_layer(N, K, seed, dev)
    x = syn.activations(M, K, seed + 100, outlier_frac=0.01)
    (y4, I), xqo, sxo = run_w4a4(x, packed, sz, dev)
    y4o, Io = oracle.linear_w4a4(xqo, sxo, po, szo, want_I=True)
    assert np.array_equal(I.cpu().numpy(), Io)
    assert np.array_equal(bits(y4), y4o)


def test_decode_many_tiles_extreme():
    """|I| = 128 * 7 * 15 in both signs on the decode path."""
    dev = need_gpu()
    M, N, K = 3, 19456 + 5, 256
    G = K // 128
    rng = np.random.default_rng(3)
    codes = torch.from_numpy(rng.choice([0, 15], (N, K)).astype(np.uint8))
    z = torch.from_numpy(rng.choice([0.0, 15.0], (N, G))).to(torch.float16)
    s = torch.ones((N, G), dtype=torch.float16)
    x = torch.from_numpy(rng.choice([-7.0, 7.0], (M, K)).astype(np.float32))
    codes[0], codes[1], codes[N - 1] = 15, 0, 15
    z[0], z[1], z[N - 1] = 0.0, 15.0, 0.0
    x[0] = 7.0
    x = x.to(torch.bfloat16)
    packed, sz = q.pack_weights(codes.to(dev), s.to(dev), z.to(dev))
    rc, po, szo = oracle.pack_weights(codes.numpy(), bits(s), bits(z))
    (y4, I), xqo, sxo = run_w4a4(x, packed, sz, dev)
    y4o, Io = oracle.linear_w4a4(xqo, sxo, po, szo, want_I=True)
    assert Io[0, 0].max() == 128 * 7 * 15 and Io[0, 1].min() == -128 * 7 * 15
    assert np.array_equal(I.cpu().numpy(), Io) and np.array_equal(bits(y4), y4o)


def test_lm_head_decode_m1_m4():
    """The LM head (128256 x 4096) at draft M = 1 and M = 4, sampled outputs."""
    dev = need_gpu()
    sampled_compare([1, 4], [("lm_head", 128256, 4096)], 6, dev, outliers=0.01, w4a16=False, points=1024)


# ----------------------------------------------------------------- quantiser fused into the linear
@pytest.mark.parametrize("M,N,K,seed", [(1, 300, 1152, 30), (2, 4096, 4096, 31), (5, 96, 640, 32),
                                        (8, 1000, 384, 33), (17, 64, 512, 34), (4, 19533, 1152, 35),
                                        (40, 200, 256, 36), (1, 4096, 14336, 37), (16, 19533, 2048, 38),
                                        (16, 300, 14336, 39), (32, 130, 18944, 40)])
def test_fused_quant_linear_equals_two_calls(M, N, K, seed):
    """qspec_linear_w4a4_bf16 gives bit for bit what qspec_quant_act_int4 then
    qspec_linear_w4a4 give (and the oracle), on every dispatch path."""
    dev = need_gpu()
    packed, sz, po, szo = make_layer(N, K, seed, dev)
    x = syn.activations(M, K, seed + 100, outlier_frac=0.01).to(dev)
    st = status(dev)
    y, xq, sx, qs, I = q.linear_w4a4_bf16(x, packed, sz, want_I=True, dev_status=st)
    assert read_status(st) == 0
    xq2, sx2, qs2 = q.quant_act_int4(x)
    y2, I2 = q.linear_w4a4(xq2, sx2, qs2, packed, sz, want_I=True)
    assert torch.equal(xq, xq2) and torch.equal(qs, qs2) and torch.equal(sx, sx2)
    assert torch.equal(I, I2) and np.array_equal(bits(y), bits(y2))
    rc, xqo, sxo, qso = oracle.quant_act_int4(bits(x.cpu()))
    y4o, Io = oracle.linear_w4a4(xqo, sxo, po, szo, want_I=True)
    assert np.array_equal(xq.cpu().numpy(), xqo) and np.array_equal(I.cpu().numpy(), Io)
    assert np.array_equal(bits(y), y4o)


@pytest.mark.gpu
@pytest.mark.parametrize("M,N,K,seed", [(16, 4096, 1024, 60), (16, 6144, 1024, 61), (9, 4096, 1152, 62),
                                        (24, 19533, 1152, 63), (32, 300, 14336, 64), (13, 600, 2048, 65)])
def test_fused_quant_tensor_core_plain(M, N, K, seed):
    """9..32 tokens through qspec_linear_w4a4_bf16 on the tensor-core kernel
    (16-token tiles, groups split over 4- and 2-CTA clusters, uneven splits;
    32-token tiles), without the debug output: y, xq, sx and qs bit for bit
    as the two calls and the oracle."""
    dev = need_gpu()
    packed, sz, po, szo = make_layer(N, K, seed, dev)
    x = syn.activations(M, K, seed + 100, outlier_frac=0.01).to(dev)
    st = status(dev)
    y, xq, sx, qs = q.linear_w4a4_bf16(x, packed, sz, dev_status=st)
    assert read_status(st) == 0
    xq2, sx2, qs2 = q.quant_act_int4(x)
    y2 = q.linear_w4a4(xq2, sx2, qs2, packed, sz)
    assert torch.equal(xq, xq2) and torch.equal(qs, qs2) and torch.equal(sx, sx2)
    assert np.array_equal(bits(y), bits(y2))
    rc, xqo, sxo, qso = oracle.quant_act_int4(bits(x.cpu()))
    y4o, _ = oracle.linear_w4a4(xqo, sxo, po, szo, want_I=True)
    assert np.array_equal(bits(y), y4o)


@pytest.mark.gpu
def test_fused_quant_tensor_core_flags_nonfinite():
    dev = need_gpu()
    packed, sz, _, _ = make_layer(4096, 1024, 66, dev)
    x = syn.activations(16, 1024, 67).to(dev)
    x[7, 300] = float("inf")
    st = status(dev)
    q.linear_w4a4_bf16(x, packed, sz, dev_status=st)
    assert q.STATUS[read_status(st)] == "QSPEC_ERR_NONFINITE"


def test_fused_quant_linear_flags_nonfinite():
    dev = need_gpu()
    packed, sz, _, _ = make_layer(64, 256, 37, dev)
    x = syn.activations(1, 256, 38).to(dev)
    x[0, 5] = float("nan")
    st = status(dev)
    q.linear_w4a4_bf16(x, packed, sz, dev_status=st)
    assert q.STATUS[read_status(st)] == "QSPEC_ERR_NONFINITE"


# ----------------------------------------------------------------- one token: byte dot products
# Rows split over every SM in balanced ranges, walked in chunks of up to
# 64 / S or 128 / S rows (S = units of 1024 codes per row); clusters of 8,
# 4 or 1 CTAs share the activations.  Covered: fewer rows than SMs, one and
# several chunks per CTA, a partial last unit (K % 1024 != 0), fewer groups
# than CTAs in a cluster, S = 64 and the largest S = 128.
@pytest.mark.parametrize("N,K,seed", [(5, 128, 40), (151, 1024, 41), (6083, 4096, 42), (300, 1152, 43),
                                      (40, 65536, 44), (24, 131072, 45), (152 * 33 + 7, 14336, 46),
                                      (16, 128, 49), (24, 768, 50),
                                      # warps per CTA a multiple of S: 6 (S = 3), 5 (S = 5),
                                      # 9 (S = 9); S = 19 (Qwen2.5-7B down projection) takes
                                      # the mixed-segment mapping
                                      (700, 2560, 51), (333, 5120, 52), (200, 9216, 54),
                                      (500, 18944, 53)])
def test_one_token_full_compare(N, K, seed):
    dev = need_gpu()
    packed, sz, po, szo = make_layer(N, K, seed, dev)
    x = syn.activations(1, K, seed + 100, outlier_frac=0.01)
    (y4, I), xqo, sxo = run_w4a4(x, packed, sz, dev)
    y4o, Io = oracle.linear_w4a4(xqo, sxo, po, szo, want_I=True)
    assert np.array_equal(I.cpu().numpy(), Io)
    assert np.array_equal(bits(y4), y4o)
    y, xq, sx, qs, I2 = q.linear_w4a4_bf16(x.to(dev), packed, sz, want_I=True)
    assert np.array_equal(xq.cpu().numpy(), xqo) and np.array_equal(I2.cpu().numpy(), Io)
    assert np.array_equal(bits(y), y4o)


@pytest.mark.parametrize("where", ["everywhere", "last_group_only", "none"])
def test_one_token_every_activation_code(where):
    """Quantised activations given directly with every nibble value, -8
    included (the quantiser never emits it; the definition covers it): -8 at
    random places, once in the last group only (the CTA that builds that
    group must tell the others of its cluster), or nowhere."""
    dev = need_gpu()
    N, K = 700, 2048
    G = K // 128
    packed, sz, po, szo = make_layer(N, K, 47, dev)
    rng = np.random.default_rng(47)
    if where == "everywhere":
        xq = rng.integers(0, 256, (1, K // 2), dtype=np.uint8)
        xq[0, :8] = 0x88                              # a run of -8 codes
    else:
        c = rng.integers(-7, 8, (1, K)).astype(np.int64) & 15
        xq = (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
        if where == "last_group_only":
            xq[0, K // 2 - 10] = (xq[0, K // 2 - 10] & 0xF0) | 0x08     # even code -8, group G - 1
    lo, hi = (xq & 15).astype(np.int32), (xq >> 4).astype(np.int32)
    codes = np.stack([lo, hi], axis=-1).reshape(1, K)
    codes = np.where(codes >= 8, codes - 16, codes)
    qs = codes.reshape(1, G, 128).sum(-1).astype(np.int32)
    sx = rng.uniform(0.01, 2.0, (1, G)).astype(np.float32)
    y, I = q.linear_w4a4(torch.from_numpy(xq).to(dev), torch.from_numpy(sx).to(dev),
                         torch.from_numpy(qs).to(dev), packed, sz, want_I=True)
    yo, Io = oracle.linear_w4a4(xq, sx, po, szo, want_I=True)
    assert np.array_equal(I.cpu().numpy(), Io) and np.array_equal(bits(y), yo)


def test_one_token_extreme():
    """|I| = 128 * 7 * 15 in both signs at one token."""
    dev = need_gpu()
    N, K = 333, 1152
    G = K // 128
    rng = np.random.default_rng(48)
    codes = torch.from_numpy(rng.choice([0, 15], (N, K)).astype(np.uint8))
    z = torch.from_numpy(rng.choice([0.0, 15.0], (N, G))).to(torch.float16)
    s = torch.ones((N, G), dtype=torch.float16)
    codes[0], codes[1], codes[N - 1] = 15, 0, 15
    z[0], z[1], z[N - 1] = 0.0, 15.0, 0.0
    x = torch.full((1, K), 7.0).to(torch.bfloat16)
    packed, sz = q.pack_weights(codes.to(dev), s.to(dev), z.to(dev))
    rc, po, szo = oracle.pack_weights(codes.numpy(), bits(s), bits(z))
    (y4, I), xqo, sxo = run_w4a4(x, packed, sz, dev)
    y4o, Io = oracle.linear_w4a4(xqo, sxo, po, szo, want_I=True)
    assert Io[0, 0].max() == 128 * 7 * 15 and Io[0, 1].min() == -128 * 7 * 15
    assert np.array_equal(I.cpu().numpy(), Io) and np.array_equal(bits(y4), y4o)


# ----------------------------------------------------------------- W4A16, one token tile
# Up to 8 tokens in one MMA column block: fewer rows than SMs, ragged tiles,
# K = 14336 with 5 and 8 tokens (the token fragments then halve the tokens
# per CTA), an odd group count.
@pytest.mark.parametrize("M,N,K,seed", [(1, 300, 1152, 60), (5, 6083, 4096, 61), (5, 1000, 14336, 62),
                                        (8, 777, 4096, 63), (3, 19533, 1152, 64), (7, 5, 640, 65),
                                        (8, 300, 14336, 66), (2, 151, 256, 67)])
def test_w4a16_one_token_tile(M, N, K, seed):
    dev = need_gpu()
    packed, sz, po, szo = make_layer(N, K, seed, dev)
    x = syn.activations(M, K, seed + 100, outlier_frac=0.01)
    y16 = q.linear_w4a16(x.to(dev), packed, sz)
    ref = oracle.linear_w4a16(bits(x), po, szo)
    assert_w4a16_close(y16, ref, "w4a16 M=%d N=%d K=%d" % (M, N, K))


# ----------------------------------------------------------------- W4A16, decode shapes (M <= 16)
# The Llama-3-8B decode linears at the verify shape M = 5 (and 8, 13, 16
# tokens), plus ragged tiles, few groups and many row tiles.
@pytest.mark.parametrize("M,N,K,seed", [
    (5, 6144, 4096, 70),     # Llama q/k/v stacked
    (8, 4096, 4096, 71),     # o
    (5, 4096, 14336, 72),    # down
    (13, 4096, 14336, 73),
    (5, 25600, 2048, 74),
    (16, 300, 1152, 75),
    (9, 130, 3072, 76),
    (1, 777, 384, 77),
    (7, 129, 128, 78),
    (2, 19533, 1152, 79),
    (11, 1000, 4096, 80),
])
def test_w4a16_decode_shapes(M, N, K, seed):
    dev = need_gpu()
    packed, sz, po, szo = make_layer(N, K, seed, dev)
    x = syn.activations(M, K, seed + 100, outlier_frac=0.01)
    st = status(dev)
    y16 = q.linear_w4a16(x.to(dev), packed, sz, dev_status=st)
    assert read_status(st) == 0
    ref = oracle.linear_w4a16(bits(x), po, szo)
    assert_w4a16_close(y16, ref, "w4a16 M=%d N=%d K=%d" % (M, N, K))


def test_w4a16_lm_head_m5():
    """The 128256 x 4096 LM head at M = gamma + 1 = 5."""
    dev = need_gpu()
    sampled_compare([5], [("lm_head", 128256, 4096)], 9, dev, outliers=0.01, w4a4=False, points=1024)


@pytest.mark.gpu
@pytest.mark.parametrize("M", [1, 5, 8, 16])
def test_w4a16_small_m_token_scales(M):
    """Tokens whose magnitudes span the bf16 range -- beyond the f16 range
    (2^40), far below it (2^-40), an all-zero token and ordinary ones -- in
    one call: each token's result, relative to its own scale, within the
    W4A16 tolerance of the oracle, and the zero token exactly zero."""
    dev = need_gpu()
    N, K = 272, 1024
    packed, sz, po, szo = make_layer(N, K, 31, dev)
    x = syn.activations(M, K, 77, outlier_frac=0.01).float()
    exps = [40, -40, 0, 12, -12, 0, 20, -20][:M] + [0] * max(0, M - 8)
    for t in range(M):
        x[t] *= 2.0 ** exps[t]
    if M > 2:
        x[2] = 0.0
    x = x.to(torch.bfloat16)
    st = status(dev)
    y16 = q.linear_w4a16(x.to(dev), packed, sz, dev_status=st)
    assert read_status(st) == 0
    got = y16.float().cpu().numpy()
    ref = oracle.linear_w4a16(bits(x), po, szo)
    for t in range(M):
        sc = 2.0 ** -exps[t]
        assert_w4a16_close(got[t] * sc, ref[t] * sc, "w4a16 M=%d token %d (scale 2^%d)" % (M, t, exps[t]))
    if M > 2:
        assert not got[2].any()


@pytest.mark.gpu
@pytest.mark.parametrize("M,N,K,seed", [(17, 384, 1024, 80), (40, 256, 2048, 81), (100, 640, 1152, 82),
                                        (129, 384, 1024, 83), (200, 272, 4096, 84), (64, 130, 14336, 85)])
def test_w4a16_tensor_core_token_tiles(M, N, K, seed):
    """W4A16 above 16 tokens: token tiles of 32, 48, 80, 112 and 64 tokens
    (one or two per call, a ragged channel tail, long K), against the oracle."""
    dev = need_gpu()
    packed, sz, po, szo = make_layer(N, K, seed, dev)
    x = syn.activations(M, K, seed + 100, outlier_frac=0.01)
    st = status(dev)
    y16 = q.linear_w4a16(x.to(dev), packed, sz, dev_status=st)
    assert read_status(st) == 0
    assert_w4a16_close(y16, oracle.linear_w4a16(bits(x), po, szo), "w4a16 M=%d N=%d K=%d" % (M, N, K))


@pytest.mark.gpu
@pytest.mark.parametrize("M,N,K,seed", [(3, 19533, 1152, 96), (8, 19533, 1152, 97), (9, 19533, 1152, 98),
                                        (16, 20000, 2048, 99)])
def test_w4a4_gemv_tc_forced_bit_exact(M, N, K, seed):
    """The tensor-memory GEMV (3..16 tokens; 9..16 in a second core-matrix
    row) forced through the bounded entry, on shapes the dispatcher may now
    send to the tensor-core kernel: outputs bit-exact with the oracle."""
    dev = need_gpu()
    packed, sz, po, szo = make_layer(N, K, seed, dev)
    x = syn.activations(M, K, seed + 100, outlier_frac=0.01)
    st = status(dev)
    xq, sx, qs = q.quant_act_int4(x.to(dev), dev_status=st)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    rc = q.qspec_debug_linear_bounded(q.KERNEL_W4A4_GEMV_TC, None, xq, sx, qs, packed, sz, M, N, K, y, N, 1 << 22, 0,
                                      st)
    assert rc == 0 and read_status(st) == 0
    rc, xqo, sxo, qso = oracle.quant_act_int4(bits(x))
    y4o, _ = oracle.linear_w4a4(xqo, sxo, po, szo, want_I=True)
    assert np.array_equal(bits(y), y4o)


@pytest.mark.gpu
@pytest.mark.parametrize("M,N,K,seed", [(16, 384, 1024, 90), (12, 600, 1152, 91), (16, 256, 2048, 92),
                                        (16, 130, 14336, 93), (16, 6144, 1024, 94), (11, 5000, 1152, 95)])
def test_w4a4_tc_split_groups_bit_exact(M, N, K, seed):
    """The W4A4 tensor-core kernel with a tile's groups split over a cluster
    (16-token tiles, few channel tiles: 4-CTA clusters, and 2-CTA clusters
    where 4 would not fit in one wave (39..76 channel tiles); uneven splits
    at 9 groups): the outputs bit-exact with the oracle's ordered fold."""
    dev = need_gpu()
    packed, sz, po, szo = make_layer(N, K, seed, dev)
    x = syn.activations(M, K, seed + 100, outlier_frac=0.01)
    st = status(dev)
    xq, sx, qs = q.quant_act_int4(x.to(dev), dev_status=st)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    rc = q.qspec_debug_linear_bounded(q.KERNEL_W4A4_TC, None, xq, sx, qs, packed, sz, M, N, K, y, N, 1 << 22, 0, st)
    assert rc == 0 and read_status(st) == 0
    rc, xqo, sxo, qso = oracle.quant_act_int4(bits(x))
    y4o, _ = oracle.linear_w4a4(xqo, sxo, po, szo, want_I=True)
    assert np.array_equal(bits(y), y4o)
