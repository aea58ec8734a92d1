"""Pins for the CPU oracle: each function is checked against something other
than itself -- published known answers, closed forms from the pages, brute
force on tiny inputs, exact rational arithmetic, special cases that reduce to
plain integer algebra, and statistical laws the method must obey.

Pages: "QSPEC: Speculative Decoding with Complementary Quantization Schemes"
summary (molayo1419.me) -- background terms (dequantisation, W4A4 INT32
accumulation, min(1, p/q) acceptance, greedy acceptance, first rejection,
E[A] and E[L]) and "QSPEC structure" (shared weights, KV overwrite);
"SpecKV: compression-aware gamma selection" blog, architecture section (the
draft statistics: confidence and entropy of the draft softmax).
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng_master = np.random.default_rng(12345)


# ---------------------------------------------------------------------------
# helpers written independently of the oracle
# ---------------------------------------------------------------------------
def f32_bits(x):
    return np.array([x], np.float32).view(np.uint32)[0]


def bf16_bits_of(values):
    """float values that are exact in bf16 -> uint16 bit patterns"""
    a = np.array(values, np.float32)
    bits = (a.view(np.uint32) >> 16).astype(np.uint16)
    back = (bits.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(back, a, equal_nan=True), "value not exact in bf16"
    return bits


def bf16_to_f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def fp16_bits(values):
    return np.asarray(values, np.float16).view(np.uint16)


def round_to_mantissa(x: Fraction, mant_bits: int) -> Fraction:
    """Round a rational to the nearest binary float with `mant_bits` fraction
    bits (normal range), ties to even.  Exact integer arithmetic."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    ulp = Fraction(2) ** (e - mant_bits)
    q, r = divmod(a, ulp)                 # a = q*ulp + r, 0 <= r < ulp
    if r * 2 > ulp or (r * 2 == ulp and q % 2 == 1):
        q += 1
    return sign * q * ulp


def f32(x: Fraction) -> Fraction:
    return round_to_mantissa(x, 23)


def unpack_weights_py(packed):
    lo = packed & 15
    hi = packed >> 4
    out = np.empty((packed.shape[0], packed.shape[1] * 2), np.int64)
    out[:, 0::2] = lo
    out[:, 1::2] = hi
    return out


def unpack_act_py(xq):
    w = unpack_weights_py(xq)
    return np.where(w >= 8, w - 16, w)


# ---------------------------------------------------------------------------
# Philox4x32-10 (random numbers of the sampled verification)
# ---------------------------------------------------------------------------
def test_philox_known_answers():
    n = 0
    for line in open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")):
        if line.startswith("#") or not line.strip():
            continue
        v = [int(t, 16) for t in line.split()]
        assert oracle.philox4x32_10(v[0:4], v[4:6]) == v[6:10]
        n += 1
    assert n == 3


def test_uniform24_counter_layout_and_uniformity():
    # counter = (slot, b, round lo, round hi), key = (seed lo, seed hi), U = word0 >> 8
    seed, rnd = 0x0123456789ABCDEF, 0xFEDCBA9876543210
    w = oracle.philox4x32_10([3, 7, rnd & 0xFFFFFFFF, rnd >> 32],
                             [seed & 0xFFFFFFFF, seed >> 32])
    assert oracle.uniform24(seed, rnd, 3, 7) == w[0] >> 8
    # chi-square over 64 bins of 20000 draws (fixed seed, deterministic)
    u = np.array([oracle.uniform24(11, 0, 0, b) for b in range(20000)])
    assert u.max() < 2 ** 24
    counts = np.bincount(u >> 18, minlength=64)
    exp = len(u) / 64
    chi2 = ((counts - exp) ** 2 / exp).sum()
    assert chi2 < 120.0   # 63 dof: P(chi2 > 120) ~ 2e-5


# ---------------------------------------------------------------------------
# own exp and fixed-point softmax
# ---------------------------------------------------------------------------
def test_qexp_error_bound():
    xs = np.concatenate([np.linspace(-32.0, 0.0, 20001), -np.logspace(-8, 1.5, 2000), [0.0]])
    worst = 0.0
    for x in xs.astype(np.float32):
        got = oracle.qexp(float(x))
        ref = math.exp(float(x))
        ulp = np.spacing(np.float32(ref))
        worst = max(worst, abs(got - ref) / float(ulp))
    assert worst <= 4.0, worst
    assert oracle.qexp(0.0) == 1.0
    assert oracle.qexp(-32.5) == 0.0 and oracle.qexp(-1e30) == 0.0


def test_fixed_softmax_matches_softmax():
    logits = rng_master.normal(0, 3, 5000).astype(np.float32)
    bits = (logits.view(np.uint32) >> 16).astype(np.uint16)          # truncate to bf16
    st, E, S, m = oracle.fixed_softmax_row(bits)
    assert st == 0
    l = bf16_to_f64(bits)
    assert m == l.max()
    assert S == int(E.sum(dtype=np.uint64))
    assert int(E[np.argmax(l)]) == 2 ** 32                           # exp(0) * 2^32
    p = np.exp(l - l.max())
    p /= p.sum()
    assert np.max(np.abs(E.astype(np.float64) / S - p)) < 1e-7
    # each weight is exp(l - m) * 2^32 to within a few ulp of fp32 plus rounding
    ref = np.exp(l - l.max()) * 2.0 ** 32
    assert np.all(np.abs(E.astype(np.float64) - ref) <= ref * 5e-7 + 0.5)


def test_fixed_softmax_status():
    assert oracle.fixed_softmax_row(bf16_bits_of([1.0, float("nan")]))[0] == oracle.ERR_NONFINITE
    assert oracle.fixed_softmax_row(bf16_bits_of([1.0, float("inf")]))[0] == oracle.ERR_NONFINITE
    assert oracle.fixed_softmax_row(bf16_bits_of([-np.inf, -np.inf]))[0] == oracle.ERR_NONFINITE
    st, E, S, _ = oracle.fixed_softmax_row(bf16_bits_of([0.0, -np.inf]))
    assert st == 0 and list(E) == [2 ** 32, 0]


# ---------------------------------------------------------------------------
# a1 pack
# ---------------------------------------------------------------------------
def test_pack_hand_example_and_round_trip():
    codes = np.zeros((2, 256), np.uint8)
    codes[0, :4] = [1, 2, 3, 15]          # bytes 0x21, 0xF3
    codes[1, 254:] = [10, 4]              # last byte 0x4A
    s = fp16_bits([[0.5, 0.25], [1.0, 2.0]])
    z = fp16_bits([[8, 0], [15, 3]])
    st, packed, sz = oracle.pack_weights(codes, s, z)
    assert st == 0
    assert packed[0, 0] == 0x21 and packed[0, 1] == 0xF3 and packed[1, 127] == 0x4A
    assert packed.sum() == 0x21 + 0xF3 + 0x4A
    # sz word: fp16(0.5) = 0x3800, fp16(8) = 0x4800
    assert sz[0, 0] == 0x3800 | (0x4800 << 16)
    assert sz[1, 1] == 0x4000 | (0x4200 << 16)      # fp16(2) = 0x4000, fp16(3) = 0x4200
    codes = rng_master.integers(0, 16, (3, 384)).astype(np.uint8)
    st, packed, _ = oracle.pack_weights(codes, np.zeros((3, 3), np.uint16),
                                        np.zeros((3, 3), np.uint16))
    assert st == 0 and np.array_equal(unpack_weights_py(packed), codes)


@pytest.mark.parametrize("case", ["code16", "z_half", "z_16", "z_neg", "s_inf"])
def test_pack_errors(case):
    codes = np.zeros((1, 128), np.uint8)
    s, z = fp16_bits([[1.0]]), fp16_bits([[3.0]])
    want = {"code16": oracle.ERR_RANGE, "z_half": oracle.ERR_ZERO_POINT,
            "z_16": oracle.ERR_ZERO_POINT, "z_neg": oracle.ERR_ZERO_POINT,
            "s_inf": oracle.ERR_NONFINITE}[case]
    if case == "code16":
        codes[0, 5] = 16
    elif case == "z_half":
        z = fp16_bits([[2.5]])
    elif case == "z_16":
        z = fp16_bits([[16.0]])
    elif case == "z_neg":
        z = fp16_bits([[-1.0]])
    else:
        s = fp16_bits([[np.inf]])
    assert oracle.pack_weights(codes, s, z)[0] == want


# ---------------------------------------------------------------------------
# a2 activation quantiser
# ---------------------------------------------------------------------------
def test_quant_act_crafted_group():
    x = np.zeros(128, np.float32)
    x[:8] = [7.0, -7.0, 2.5, 3.5, -2.5, 0.5, 1.5, -0.5]   # amax 7 -> sx = 1 exactly
    st, xq, sx, qs = oracle.quant_act_int4(bf16_bits_of(x)[None, :])
    assert st == 0 and sx[0, 0] == 1.0
    q = unpack_act_py(xq)[0]
    # ties to even: 2.5 -> 2, 3.5 -> 4, -2.5 -> -2, 0.5 -> 0, 1.5 -> 2, -0.5 -> 0
    assert list(q[:8]) == [7, -7, 2, 4, -2, 0, 2, 0]
    assert qs[0, 0] == 7 - 7 + 2 + 4 - 2 + 0 + 2 + 0
    assert xq[0, 0] == (7 | ((-7 & 15) << 4))             # two's-complement nibbles


def test_quant_act_zero_group_and_bounds():
    M, K = 3, 512
    x = rng_master.normal(0, 1, (M, K)).astype(np.float32)
    x[1, 128:256] = 0.0                                    # an all-zero group
    x[2, :] *= 1e-30                                       # tiny values stay exact
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    st, xq, sx, qs = oracle.quant_act_int4(bits)
    assert st == 0
    xv = bf16_to_f64(bits).reshape(M, K // 128, 128)
    q = unpack_act_py(xq).reshape(M, K // 128, 128)
    assert sx[1, 1] == 0.0 and np.all(q[1, 1] == 0)
    assert np.all(np.abs(q) <= 7)
    amax = np.abs(xv).max(axis=2)
    assert np.array_equal(sx, (amax.astype(np.float32) / np.float32(7.0)))
    # element at +-amax maps to +-7; reconstruction error at most sx / 2 (+ rounding of sx)
    err = np.abs(xv - q * sx[:, :, None].astype(np.float64))
    assert np.all(err <= sx[:, :, None] * (0.5 + 1e-6))
    idx = np.argmax(np.abs(xv), axis=2)
    top = np.take_along_axis(q, idx[:, :, None], 2)[:, :, 0]
    nz = amax > 0
    assert np.all(np.abs(top[nz]) == 7)
    assert np.array_equal(qs, q.sum(axis=2))


def test_quant_act_nonfinite():
    x = np.zeros((1, 128), np.float32)
    x[0, 3] = np.inf
    assert oracle.quant_act_int4(bf16_bits_of(x))[0] == oracle.ERR_NONFINITE


# ---------------------------------------------------------------------------
# a3 W4A4
# ---------------------------------------------------------------------------
def _random_w4a4_inputs(M, N, K, rng, extreme=False):
    G = K // 128
    if extreme:
        q = rng.choice([-7, 7], (M, K))
        W = rng.choice([0, 15], (N, K))
        z = rng.choice([0, 15], (N, G)).astype(np.float64)
    else:
        q = rng.integers(-7, 8, (M, K))
        W = rng.integers(0, 16, (N, K))
        z = rng.integers(0, 16, (N, G)).astype(np.float64)
    xq = ((q[:, 0::2] & 15) | ((q[:, 1::2] & 15) << 4)).astype(np.uint8)
    s = rng.uniform(0.005, 0.02, (N, G))
    st, packed, sz = oracle.pack_weights(W.astype(np.uint8), fp16_bits(s), fp16_bits(z))
    assert st == 0
    sx = rng.uniform(0.01, 1.0, (M, G)).astype(np.float32)
    return q, W, z, xq, sx, packed, sz


@pytest.mark.parametrize("K,extreme", [(128, False), (256, False), (256, True), (384, True)])
def test_w4a4_integer_accumulators_brute_force(K, extreme):
    rng = np.random.default_rng(K + extreme)
    M, N = 3, 5
    q, W, z, xq, sx, packed, sz = _random_w4a4_inputs(M, N, K, rng, extreme)
    _, I = oracle.linear_w4a4(xq, sx, packed, sz, want_I=True)
    G = K // 128
    ref = np.zeros((M, N, G), np.int64)
    for m in range(M):
        for n in range(N):
            for g in range(G):
                ks = slice(128 * g, 128 * g + 128)
                ref[m, n, g] = int(np.dot(q[m, ks], W[n, ks] - int(z[n, g])))
    assert np.array_equal(I, ref)
    if extreme:
        assert np.abs(ref).max() <= 128 * 7 * 15


def test_w4a4_fold_exact_rational():
    """y = bf16(fold_g fmaf(I_g, fl(sx*s), acc)), emulated with exact fractions."""
    rng = np.random.default_rng(7)
    M, N, K = 2, 4, 512
    q, W, z, xq, sx, packed, sz = _random_w4a4_inputs(M, N, K, rng)
    y, I, accs = oracle.linear_w4a4(xq, sx, packed, sz, want_I=True, want_acc=True)
    s32 = (sz & 0xFFFF).astype(np.uint16).view(np.float16).astype(np.float32)
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for g in range(K // 128):
                c = f32(Fraction(float(sx[m, g])) * Fraction(float(s32[n, g])))
                acc = f32(Fraction(int(I[m, n, g])) * c + acc)     # one rounding: fused
            assert Fraction(float(accs[m, n])) == acc, (m, n)
            want = round_to_mantissa(acc, 7)
            got = bf16_to_f64([y[m, n]])[0]
            assert Fraction(got) == want, (m, n)


def test_w4a4_unit_scales_is_integer_gemm():
    # all scales 1, one group: y = bf16(I) and I is the plain integer GEMM with zero points
    rng = np.random.default_rng(3)
    M, N, K = 4, 6, 128
    q = rng.integers(-7, 8, (M, K))
    W = rng.integers(0, 16, (N, K))
    z = rng.integers(0, 16, (N, 1))
    xq = ((q[:, 0::2] & 15) | ((q[:, 1::2] & 15) << 4)).astype(np.uint8)
    st, packed, sz = oracle.pack_weights(W.astype(np.uint8), fp16_bits(np.ones((N, 1))),
                                         fp16_bits(z))
    y = oracle.linear_w4a4(xq, np.ones((M, 1), np.float32), packed, sz)
    ref = q @ (W - z).T
    got = bf16_to_f64(y)
    want = np.array([[float(round_to_mantissa(Fraction(int(v)), 7)) for v in row] for row in ref])
    assert np.array_equal(got, want)


def test_w4a4_points_match_full():
    rng = np.random.default_rng(9)
    q, W, z, xq, sx, packed, sz = _random_w4a4_inputs(5, 9, 384, rng)
    y = oracle.linear_w4a4(xq, sx, packed, sz)
    ms, ns = np.array([0, 4, 2, 3]), np.array([8, 0, 5, 3])
    assert np.array_equal(oracle.linear_w4a4_points(xq, sx, packed, sz, ms, ns), y[ms, ns])


# ---------------------------------------------------------------------------
# a4 W4A16 (fp64 reference of Y = X W^, W^ = s (W - z))
# ---------------------------------------------------------------------------
def _pack(W, s, z):
    st, packed, sz = oracle.pack_weights(np.asarray(W, np.uint8), fp16_bits(s), fp16_bits(z))
    assert st == 0
    return packed, sz


def test_w4a16_unit_scale_zero_point_is_integer_gemm():
    rng = np.random.default_rng(4)
    M, N, K = 3, 7, 256
    X = rng.integers(-20, 21, (M, K)).astype(np.float32)     # exact in bf16
    W = rng.integers(0, 16, (N, K))
    packed, sz = _pack(W, np.ones((N, 2)), np.zeros((N, 2)))
    ref = oracle.linear_w4a16(bf16_bits_of(X), packed, sz)
    assert np.array_equal(ref, (X.astype(np.int64) @ W.T).astype(np.float64))


def test_w4a16_zero_point_sign_and_group_scale():
    M, N, K = 2, 3, 256
    X = np.ones((M, K), np.float32)
    X[1] = -2.0
    W = np.zeros((N, K), np.int64)
    W[1, :] = 15
    W[2, :128] = 4
    s = np.array([[0.5, 0.25], [1.0, 1.0], [2.0, 0.5]])
    z = np.array([[15, 15], [15, 0], [4, 0]])
    ref = oracle.linear_w4a16(bf16_bits_of(X), *_pack(W, s, z))
    # row 0: W - z = -15 everywhere: sum = 128*(0.5*-15) + 128*(0.25*-15)
    r0 = 128 * 0.5 * -15 + 128 * 0.25 * -15
    # row 1: group 0 -> 0, group 1 -> 15 * 1.0
    r1 = 128 * 15.0
    # row 2: group 0: W = z -> 0; group 1: W = 0, z = 0 -> 0
    assert ref[0].tolist() == [r0, r1, 0.0]
    assert ref[1].tolist() == [-2 * r0, -2 * r1, 0.0]


def test_w4a16_points_and_linearity():
    rng = np.random.default_rng(5)
    M, N, K = 4, 6, 384
    X = rng.normal(0, 1, (M, K)).astype(np.float32)
    Xb = (X.view(np.uint32) >> 16).astype(np.uint16)
    W = rng.integers(0, 16, (N, K))
    z = rng.integers(0, 16, (N, 3))
    s = rng.uniform(0.005, 0.02, (N, 3)).astype(np.float16).astype(np.float64)
    r1 = oracle.linear_w4a16(Xb, *_pack(W, s, z))
    r2 = oracle.linear_w4a16(Xb, *_pack(W, 2 * s, z))            # power-of-two scaling is exact
    assert np.array_equal(r2, 2 * r1)
    ms, ns = np.array([3, 0, 1]), np.array([5, 2, 0])
    assert np.array_equal(oracle.linear_w4a16_points(Xb, *_pack(W, s, z), ms, ns), r1[ms, ns])
    # and the definition via explicit dequantisation, in exact rationals, on one element
    xv = bf16_to_f64(Xb)
    exact = sum(Fraction(xv[1, k]) * Fraction(s[4, k // 128]) * (int(W[4, k]) - int(z[4, k // 128]))
                for k in range(K))
    assert abs(r1[1, 4] - float(exact)) <= 1e-12 * (1 + abs(float(exact)))


# ---------------------------------------------------------------------------
# a5 greedy verification
# ---------------------------------------------------------------------------
def _load_greedy_cases():
    rows, cases = [], []
    for line in open(os.path.join(GOLDEN, "greedy_worked_cases.txt")):
        t = line.split()
        if not t or t[0].startswith("#"):
            continue
        if t[0] == "row":
            rows.append([float(v) for v in t[2:]])
        elif t[0] == "case":
            a, b = line[len("case"):].split("->")
            n, out = b.split("|")
            cases.append(([int(v) for v in a.split()], int(n), [int(v) for v in out.split()]))
    return np.array(rows, np.float32), cases


def test_greedy_worked_cases():
    rows, cases = _load_greedy_cases()
    P = bf16_bits_of(rows)[None]
    assert len(cases) == 4
    for drafts, n_want, out_want in cases:
        st, n_acc, out = oracle.verify_greedy(P, np.array([drafts], np.int32))
        assert st == 0 and n_acc[0] == n_want and out[0].tolist() == out_want


def test_greedy_self_consistent_drafts_and_cutoff():
    rng = np.random.default_rng(1)
    B, gamma, V = 6, 5, 300
    l = rng.normal(0, 2, (B, gamma + 1, V)).astype(np.float32)
    P = (l.view(np.uint32) >> 16).astype(np.uint16)
    arg = np.argmax(bf16_to_f64(P), axis=2)          # numpy argmax: first maximum
    st, n_acc, out = oracle.verify_greedy(P, arg[:, :gamma].astype(np.int32))
    assert st == 0 and np.all(n_acc == gamma) and np.array_equal(out, arg)
    # break position j of sequence b; everything after j must not matter
    drafts = arg[:, :gamma].astype(np.int32).copy()
    for b in range(B):
        j = b % gamma
        drafts[b, j] = (drafts[b, j] + 1) % V
        drafts[b, j + 1:] = rng.integers(0, V, gamma - j - 1)
    st, n_acc, out = oracle.verify_greedy(P, drafts)
    for b in range(B):
        j = b % gamma
        assert n_acc[b] == j
        assert out[b, :j].tolist() == drafts[b, :j].tolist()
        assert out[b, j] == arg[b, j] and np.all(out[b, j + 1:] == -1)


def test_greedy_status():
    P = bf16_bits_of(np.zeros((1, 3, 4)))
    assert oracle.verify_greedy(P, np.array([[0, 4]], np.int32))[0] == oracle.ERR_RANGE
    P2 = P.copy()
    P2[0, 2, 1] = 0x7FC0                                    # NaN
    assert oracle.verify_greedy(P2, np.array([[0, 0]], np.int32))[0] == oracle.ERR_NONFINITE


# ---------------------------------------------------------------------------
# a6 sampled verification
# ---------------------------------------------------------------------------
def _fixed_probs(bits_row):
    st, E, S, _ = oracle.fixed_softmax_row(bits_row)
    assert st == 0
    return E.astype(np.float64) / S


def test_sampled_first_token_follows_target_chi_square():
    """Speculative sampling keeps the output distributed as the target p: over
    many rounds the first emitted token is p'-distributed (p' the fixed-point
    target distribution), whatever the draft distribution."""
    V, gamma = 8, 1
    lp = np.array([1.0, 0.5, 0.0, -1.0, 2.0, -0.5, 0.25, 1.5], np.float32)
    lq = np.array([0.0, 1.5, 1.0, 0.5, 0.0, 1.0, -1.0, 0.5], np.float32)
    lb = np.array([0.0, -1.0, 1.0, -2.0, 0.5, 0.0, 2.0, -0.5], np.float32)
    pb, qb, bb = bf16_bits_of(lp), bf16_bits_of(lq), bf16_bits_of(lb)
    p, q, pbonus = _fixed_probs(pb), _fixed_probs(qb), _fixed_probs(bb)
    B, R = 250000, 4
    rng = np.random.default_rng(2024)
    P = np.broadcast_to(np.stack([pb, bb])[None], (B, 2, V)).copy()
    Q = np.broadcast_to(qb[None, None], (B, 1, V)).copy()
    first, bonus, rejected_tok = [], [], []
    for r in range(R):
        drafts = rng.choice(V, size=(B, 1), p=q).astype(np.int32)
        st, n_acc, out = oracle.verify_sample(P, Q, drafts, seed=77, rnd=r)
        assert st == 0
        first.append(out[:, 0])
        bonus.append(out[n_acc == 1, 1])
        rejected_tok.append(out[n_acc == 0, 0])
    first = np.concatenate(first)

    def chi2(samples, probs):
        counts = np.bincount(samples, minlength=V)
        exp = probs * len(samples)
        keep = exp > 0
        assert counts[~keep].sum() == 0
        return ((counts[keep] - exp[keep]) ** 2 / exp[keep]).sum(), keep.sum() - 1

    from scipy.stats import chi2 as chi2dist
    c, dof = chi2(first, p)
    assert chi2dist.sf(c, dof) > 1e-3, c
    # bonus tokens (all drafts accepted) follow the last target row
    c, dof = chi2(np.concatenate(bonus), pbonus)
    assert chi2dist.sf(c, dof) > 1e-3, c
    # the token after a rejection follows the normalised residual max(0, p - q)
    res = np.maximum(p - q, 0)
    res /= res.sum()
    c, dof = chi2(np.concatenate(rejected_tok), res)
    assert chi2dist.sf(c, dof) > 1e-3, c
    # acceptance rate = sum_v min(p, q)
    acc_rate = 1 - sum(len(x) for x in rejected_tok) / (B * R)
    assert abs(acc_rate - np.minimum(p, q).sum()) < 4 * math.sqrt(0.25 / (B * R))


@pytest.mark.parametrize("alpha", [0.3, 0.6, 0.9])
@pytest.mark.parametrize("gamma", [2, 4, 8])
def test_sampled_expected_length_closed_form(alpha, gamma):
    """E[L] = (1 - a^(K+1)) / (1 - a), E[A] = a (1 - a^K) / (1 - a) for i.i.d.
    acceptance a: draft q' = (1, 0), target p' = (a, 1 - a)."""
    V, B = 2, 100000
    lp = np.array([math.log(alpha), math.log(1 - alpha)], np.float32)
    pbits = (lp.view(np.uint32) >> 16).astype(np.uint16)
    qbits = bf16_bits_of([0.0, -100.0])
    st, E, S, _ = oracle.fixed_softmax_row(pbits)
    # a 24-bit uniform U accepts iff U < 2^24 * Ep0 / Sp
    a = math.ceil(2 ** 24 * int(E[0]) / S) / 2 ** 24
    P = np.broadcast_to(pbits[None, None], (B, gamma + 1, V)).copy()
    Q = np.broadcast_to(qbits[None, None], (B, gamma, V)).copy()
    st, n_acc, out = oracle.verify_sample(P, Q, np.zeros((B, gamma), np.int32), seed=5,
                                          rnd=gamma)
    assert st == 0
    L = n_acc + 1
    EL = (1 - a ** (gamma + 1)) / (1 - a)
    EA = a * (1 - a ** gamma) / (1 - a)
    sigma = L.std() / math.sqrt(B)
    assert abs(L.mean() - EL) < 4 * sigma
    assert abs(n_acc.mean() - EA) < 4 * sigma
    # after a rejection the correction is token 1 (the only residual mass)
    rej = n_acc < gamma
    assert np.all(out[rej, n_acc[rej]] == 1)


def test_sampled_identities():
    rng = np.random.default_rng(8)
    B, gamma, V = 64, 4, 50
    l = rng.normal(0, 2, (B, gamma + 1, V)).astype(np.float32)
    P = (l.view(np.uint32) >> 16).astype(np.uint16)
    drafts = rng.integers(0, V, (B, gamma)).astype(np.int32)
    # p == q: every draft accepted (the bonus comes from row gamma)
    st, n_acc, out = oracle.verify_sample(P, P[:, :gamma].copy(), drafts, 1, 2)
    assert st == 0 and np.all(n_acc == gamma)
    assert np.array_equal(out[:, :gamma], drafts)
    # q(t) > 0 = p(t) at position 3: never accepted beyond position 2
    P2 = P.copy()
    for b in range(B):
        P2[b, 2, drafts[b, 2]] = 0xFF80                          # -inf: p(t) = 0
    st, n_acc, out = oracle.verify_sample(P2, P[:, :gamma].copy(), drafts, 1, 3)
    assert st == 0 and np.all(n_acc == 2)
    assert np.all(out[np.arange(B), 2] != drafts[:, 2])          # p(t) = 0: never emitted
    # p(t) = q(t) = 0 at position 2: 0 < 0 is false, so rejected as well
    Q3 = P[:, :gamma].copy()
    for b in range(B):
        Q3[b, 1, drafts[b, 1]] = 0xFF80
    P3 = Q3.copy()
    P3 = np.concatenate([P3, P[:, gamma:]], axis=1)
    st, n_acc, out = oracle.verify_sample(P3, Q3, drafts, 1, 4)
    assert st == 0 and np.all(n_acc == 1)


def test_sampled_first_rejection_cutoff():
    rng = np.random.default_rng(9)
    B, gamma, V = 200, 6, 40
    P = (rng.normal(0, 2, (B, gamma + 1, V)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    Q = (rng.normal(0, 2, (B, gamma, V)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    drafts = rng.integers(0, V, (B, gamma)).astype(np.int32)
    st, n_acc, out = oracle.verify_sample(P, Q, drafts, 3, 4)
    assert st == 0 and n_acc.min() < gamma
    # mutate every draft and every draft row after the first rejection
    d2, Q2 = drafts.copy(), Q.copy()
    for b in range(B):
        A = n_acc[b]
        if A + 1 < gamma:
            d2[b, A + 1:] = rng.integers(0, V, gamma - A - 1)
            Q2[b, A + 1:] = rng.integers(0, 0x3F00, (gamma - A - 1, V))
    st, n2, o2 = oracle.verify_sample(P, Q2, d2, 3, 4)
    assert np.array_equal(n2, n_acc) and np.array_equal(o2, out)
    assert np.all(out[np.arange(gamma + 1)[None, :] > n_acc[:, None]] == -1)


def test_sampled_status():
    P = bf16_bits_of(np.zeros((1, 2, 4)))
    Q = bf16_bits_of(np.zeros((1, 1, 4)))
    assert oracle.verify_sample(P, Q, np.array([[4]], np.int32), 0, 0)[0] == oracle.ERR_RANGE
    Q2 = Q.copy()
    Q2[0, 0, :] = 0xFF80
    assert oracle.verify_sample(P, Q2, np.array([[0]], np.int32), 0, 0)[0] == oracle.ERR_NONFINITE
    P2 = P.copy()
    P2[0, 1, 2] = 0x7F80
    assert oracle.verify_sample(P2, Q, np.array([[0]], np.int32), 0, 0)[0] == oracle.ERR_NONFINITE


# ---------------------------------------------------------------------------
# draft-side sampling and the draft statistics (SpecKV blog, architecture:
# confidence = largest probability, entropy = -sum p log(p + 1e-9))
# ---------------------------------------------------------------------------
NEG_INF_BF16 = 0xFF80


def test_draft_statistics_closed_forms():
    """Uniform rows have p = 1/V exactly: confidence 1/V and entropy
    -log(1/V + 1e-9) (the 1e-9 moves it by ~V * 1e-9, far above the
    tolerance); k equal logits and the rest -inf give 1/k; a single finite
    logit gives confidence 1, entropy -log(1 + 1e-9) < 0 and that token."""
    half = bf16_bits_of([0.5])[0]
    for V in (1, 2, 7, 1000, 128256):
        st, tok, conf, ent = oracle.draft_sample(np.full((1, V), half, np.uint16), 3, 4, 1)
        assert st == 0 and 0 <= tok[0] < V
        assert conf[0] == np.float32(1.0 / V)
        assert abs(ent[0] + math.log(1.0 / V + 1e-9)) <= 1e-9
    for V, k in ((10, 3), (5000, 17), (128256, 1000)):
        row = np.full(V, NEG_INF_BF16, np.uint16)
        hot = np.random.default_rng(V).choice(V, k, replace=False)
        row[hot] = bf16_bits_of([-1.25])[0]
        st, tok, conf, ent = oracle.draft_sample(row[None], 5, 6, 2)
        assert st == 0 and tok[0] in hot
        assert conf[0] == np.float32(1.0 / k)
        assert abs(ent[0] + math.log(1.0 / k + 1e-9)) <= 1e-9
    row = np.full(300, bf16_bits_of([-40.0])[0], np.uint16)     # e^-40 is below the fixed-point grid
    row[123] = bf16_bits_of([2.0])[0]
    st, tok, conf, ent = oracle.draft_sample(row[None], 7, 8, 16)
    assert st == 0 and tok[0] == 123 and conf[0] == 1.0
    assert abs(ent[0] + math.log(1.0 + 1e-9)) <= 1e-15 and ent[0] < 0


def test_draft_statistics_match_float64_softmax():
    """Random rows (N(0, 2^2), some -inf): confidence and entropy against the
    float64 softmax computed with numpy, within the fixed-point weights'
    error (own exp within 4 ulp of fp32, E rounded to 2^-32)."""
    rng = np.random.default_rng(31)
    B, V = 6, 5000
    l = (rng.standard_normal((B, V)) * 2).astype(np.float32)
    bits = (l.view(np.uint32) >> 16).astype(np.uint16)        # truncate to bf16
    bits[:, rng.choice(V, 50, replace=False)] = NEG_INF_BF16
    st, tok, conf, ent = oracle.draft_sample(bits, 11, 12, 3)
    assert st == 0
    lf = bf16_to_f64(bits)
    p = np.exp(lf - lf.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    H = -(p * np.log(p + 1e-9)).sum(1)
    np.testing.assert_allclose(conf, p.max(1), rtol=1e-6)
    assert np.all(np.abs(ent - H) <= 1e-5 * (1 + H))
    assert np.all(p[np.arange(B), tok] > 0)                   # never a -inf token


def test_draft_draw_rule_and_slot():
    """Two equal logits: E = (2^32, 2^32), so T = floor(U 2^33 / 2^24) and
    token 1 is drawn exactly when U >= 2^23, U the Philox uniform of slot
    16 + step for row b (Philox pinned by its known answers)."""
    B = 64
    q = np.tile(bf16_bits_of([0.75, 0.75]), (B, 1))
    for step in (1, 7, 16):
        st, tok, _, _ = oracle.draft_sample(q, 2024, 99, step)
        assert st == 0
        want = [int(oracle.uniform24(2024, 99, 16 + step, b) >= (1 << 23)) for b in range(B)]
        assert tok.tolist() == want


def test_draft_draw_rule_exact_on_uniform_rows():
    """Uniform rows: E_v = 2^32, W = V 2^32, T = floor(U V 2^8) and the first
    prefix (v + 1) 2^32 above T gives token floor(U V / 2^24) exactly.  With
    V = 4096 the threshold equals a prefix sum (U V a multiple of 2^24) about
    once in 4096 rows; the sample below holds such rows, where a >= in place
    of > would pick the token before."""
    V, B, seed, rnd, step = 4096, 16384, 606, 17, 5
    q = np.full((B, V), bf16_bits_of([1.0])[0], np.uint16)
    st, tok, conf, _ = oracle.draft_sample(q, seed, rnd, step)
    assert st == 0 and np.all(conf == np.float32(1.0 / V))
    U = np.array([oracle.uniform24(seed, rnd, 16 + step, b) for b in range(B)], np.int64)
    assert np.array_equal(tok, (U * V) >> 24)
    assert ((U * V) % (1 << 24) == 0).sum() >= 1                # ties present in the sample


def test_draft_confidence_is_rounded_exact_quotient():
    """confidence = max E / S (max E = 2^32, the weight of the row maximum)
    as the fp64 quotient rounded to fp32: checked bit for bit against exact
    rational arithmetic on random rows (S from the fixed-point row sums)."""
    rng = np.random.default_rng(47)
    B, V = 40, 3000
    l = (rng.standard_normal((B, V)) * 1.5).astype(np.float32)
    bits = (l.view(np.uint32) >> 16).astype(np.uint16)
    st, _, conf, _ = oracle.draft_sample(bits, 1, 2, 3)
    assert st == 0
    for b in range(B):
        st_r, E, S, _ = oracle.fixed_softmax_row(bits[b])
        assert st_r == 0 and int(E.max()) == 1 << 32
        want = round_to_mantissa(round_to_mantissa(Fraction(1 << 32, int(S)), 52), 23)
        assert Fraction(float(conf[b])) == want


def test_draft_tokens_follow_softmax_chi_square():
    """Over many rows of the same logits (independent uniforms per row) the
    drawn token follows the softmax of the row, and the draws of two draft
    positions differ."""
    from scipy.stats import chi2 as chi2dist
    V, B = 8, 200000
    lv = np.array([1.0, 0.5, 0.0, -1.0, 2.0, -0.5, 0.25, 1.5], np.float32)
    row = bf16_bits_of(lv)
    p = np.exp(lv.astype(np.float64) - lv.max())
    p /= p.sum()
    draws = []
    for step in (1, 2):
        st, tok, _, _ = oracle.draft_sample(np.tile(row, (B, 1)), 5, 0, step)
        assert st == 0
        counts = np.bincount(tok, minlength=V)
        exp = p * B
        assert chi2dist.sf(((counts - exp) ** 2 / exp).sum(), V - 1) > 1e-3
        draws.append(tok)
    assert (draws[0] != draws[1]).mean() > 0.5


def test_draft_status():
    q = np.tile(bf16_bits_of([0.0, 1.0, 2.0]), (3, 1))
    assert oracle.draft_sample(q, 0, 0, 1)[0] == 0
    for bad in (0x7FC0, 0x7F80):                               # NaN, +inf
        q2 = q.copy()
        q2[1, 2] = bad
        assert oracle.draft_sample(q2, 0, 0, 1)[0] == oracle.ERR_NONFINITE
    q3 = q.copy()
    q3[2, :] = NEG_INF_BF16                                    # a row without mass
    assert oracle.draft_sample(q3, 0, 0, 1)[0] == oracle.ERR_NONFINITE


# ---------------------------------------------------------------------------
# a7 KV overwrite
# ---------------------------------------------------------------------------
def test_kv_overwrite_canary():
    rng = np.random.default_rng(10)
    L, B, H, T, D, gamma = 2, 3, 2, 16, 8, 3
    kc = rng.integers(0, 2 ** 16, (L, B, H, T, D)).astype(np.uint16)
    vc = rng.integers(0, 2 ** 16, (L, B, H, T, D)).astype(np.uint16)
    kn = rng.integers(0, 2 ** 16, (L, B, gamma + 1, H, D)).astype(np.uint16)
    vn = rng.integers(0, 2 ** 16, (L, B, gamma + 1, H, D)).astype(np.uint16)
    base = np.array([0, 5, 12], np.int32)
    nacc = np.array([3, 0, 2], np.int32)
    k2, v2 = kc.copy(), vc.copy()
    assert oracle.kv_overwrite(k2, v2, kn, vn, base, nacc, gamma) == 0
    ek, ev = kc.copy(), vc.copy()
    for b in range(B):
        for r in range(nacc[b] + 1):
            ek[:, b, :, base[b] + r, :] = kn[:, b, r, :, :]
            ev[:, b, :, base[b] + r, :] = vn[:, b, r, :, :]
    assert np.array_equal(k2, ek) and np.array_equal(v2, ev)
    # rows outside [base, base + n_acc] untouched (canary)
    assert np.array_equal(k2[:, 1, :, 6:], kc[:, 1, :, 6:])


@pytest.mark.parametrize("base,nacc", [(-1, 0), (14, 2), (0, 4), (0, -1)])
def test_kv_overwrite_range(base, nacc):
    L, B, H, T, D, gamma = 1, 1, 1, 16, 8, 3
    kc = np.zeros((L, B, H, T, D), np.uint16)
    vc = kc.copy()
    kn = np.ones((L, B, gamma + 1, H, D), np.uint16)
    st = oracle.kv_overwrite(kc, vc, kn, kn.copy(), np.array([base], np.int32),
                             np.array([nacc], np.int32), gamma)
    assert st == oracle.ERR_RANGE and not kc.any()


# ----------------------------------------------------------------- SpecQuant Q8 (FP8, next-3)
# SpecQuant summary page, contributions and approach: FP8 (Q8) variant
# derived from the FP16 parent.  The E4M3 codec against torch's float8_e4m3fn
# (an independent implementation of the same format), the derivation against
# invariants of its definition, the linear against an integer matmul.
def test_e4m3_decode_every_code_matches_library():
    import torch
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    got = np.array([oracle.e4m3_value(b) for b in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin].astype(np.float64))
    # the extremes of the format: 448 and the smallest subnormal 2^-9
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(0x01) == 2.0 ** -9


def test_e4m3_encode_matches_library_and_saturates():
    import torch
    rng = np.random.default_rng(41)
    x = np.concatenate([rng.standard_normal(40000) * 0.01, rng.standard_normal(40000) * 30,
                        rng.uniform(-447.9, 447.9, 20000), rng.uniform(-2.0 ** -7, 2.0 ** -7, 20000)])
    # exact midpoints between neighbouring codes: ties go to the even code
    pos = np.array([oracle.e4m3_value(b) for b in range(0x7E)])
    mids = (pos + np.array([oracle.e4m3_value(b + 1) for b in range(0x7E)])) / 2
    x = np.concatenate([x, mids, -mids]).astype(np.float32)
    got = oracle.e4m3_from_float(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)
    assert all(int(oracle.e4m3_from_float(np.float32(m))[0]) % 2 == 0 for m in mids)
    # saturation at 448, NaN, signed zero
    big = np.array([448.0, 464.0, 1e6, 3e38, -500.0], np.float32)
    assert oracle.e4m3_from_float(big).tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE]
    assert int(oracle.e4m3_from_float(np.float32("nan"))[0]) == 0x7F
    assert int(oracle.e4m3_from_float(np.float32(-0.0))[0]) == 0x80


def test_fp8_weight_derivation_invariants():
    rng = np.random.default_rng(42)
    W = (rng.standard_normal((40, 512)) * 0.02).astype(np.float16)
    W[3, :] = 0.0                                        # an all-zero row
    W[5, 7] = np.float16(-3.5)                           # a negative row maximum
    st, w8, s8 = oracle.quant_weights_fp8(W.view(np.uint16))
    assert st == 0
    Wf = W.astype(np.float64)
    amax = np.abs(Wf).max(axis=1)
    dec = np.vectorize(oracle.e4m3_value)(w8)
    for n in range(W.shape[0]):
        if amax[n] == 0:
            assert s8[n] == 0 and not w8[n].any()
            continue
        j = int(np.argmax(np.abs(Wf[n])))
        assert w8[n, j] == (0xFE if Wf[n, j] < 0 else 0x7E)            # the row maximum maps to 448
        rec = dec[n] * float(s8[n])
        # E4M3 keeps 3 mantissa bits: a half-ulp error of at most 2^-4 of the
        # value (normal range), at most 2^-10 s8 in the subnormal range
        bound = np.maximum(np.abs(Wf[n]) * 2.0 ** -4, 2.0 ** -10 * float(s8[n])) * (1 + 1e-6)
        assert np.all(np.abs(rec - Wf[n]) <= bound)
        assert abs(float(s8[n]) * 448 - amax[n]) <= amax[n] * 2.0 ** -23
    bad = W.copy()
    bad[0, 0] = np.float16("inf")
    assert oracle.quant_weights_fp8(bad.view(np.uint16))[0] == 8


def test_fp8_activation_quant_invariants():
    import torch
    rng = np.random.default_rng(43)
    x = torch.from_numpy(rng.standard_normal((6, 384)).astype(np.float32)).to(torch.bfloat16)
    x[2] = 0.0
    st, xq, sa = oracle.quant_act_fp8(x.view(torch.int16).numpy().view(np.uint16))
    assert st == 0
    xf = x.float().numpy().astype(np.float64)
    for m in range(6):
        if sa[m] == 0:
            assert not xq[m].any()
            continue
        j = int(np.argmax(np.abs(xf[m])))
        assert xq[m, j] == (0xFE if xf[m, j] < 0 else 0x7E)


def test_fp8_linear_reduces_to_integer_matmul():
    # codes holding the integers -8..8 exactly, unit scales: an integer matmul
    rng = np.random.default_rng(44)
    ints = np.arange(-8, 9)
    code_of = {int(v): int(oracle.e4m3_from_float(np.float32(v))[0]) for v in ints}
    assert all(oracle.e4m3_value(c) == v for v, c in code_of.items())
    A = rng.integers(-8, 9, (5, 256))
    B = rng.integers(-8, 9, (7, 256))
    xq = np.vectorize(code_of.get)(A).astype(np.uint8)
    w8 = np.vectorize(code_of.get)(B).astype(np.uint8)
    ref = oracle.linear_fp8(xq, np.ones(5, np.float32), w8, np.ones(7, np.float32))
    assert np.array_equal(ref, (A @ B.T).astype(np.float64))
    # power-of-two scales scale the result exactly; the operands are not swapped
    ref2 = oracle.linear_fp8(xq, np.full(5, 0.25, np.float32), w8, np.arange(1, 8, dtype=np.float32))
    assert np.array_equal(ref2, (A @ B.T) * 0.25 * np.arange(1, 8)[None, :])
