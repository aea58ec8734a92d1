"""a5 greedy / a6 sampled verification: every acceptance count, emitted token
and row statistic bit-exact against the oracle; statistical laws on the GPU."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from quantized_speculative_decoding_shared_gb300 import binding as q, synthetic as syn
from gpuhelp import bits, need_gpu, read_status, status

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def gpu_greedy(P, drafts, dev):
    st = status(dev)
    n, out = q.verify_greedy(P.to(dev), drafts.to(dev), dev_status=st)
    return read_status(st), n.cpu().numpy(), out.cpu().numpy()


def gpu_sample(P, Q, drafts, seed, rnd, dev, ws=None):
    st = status(dev)
    n, out = q.verify_sample(P.to(dev), Q.to(dev), drafts.to(dev), seed, rnd, workspace=ws,
                             dev_status=st)
    return read_status(st), n.cpu().numpy(), out.cpu().numpy()


def check_both(P, Q, drafts, dev, seed=7, rnd=3):
    rc, n, out = gpu_greedy(P, drafts, dev)
    rco, no, outo = oracle.verify_greedy(bits(P), drafts.numpy())
    assert rc == rco == 0
    assert np.array_equal(n, no) and np.array_equal(out, outo)
    rc, n, out = gpu_sample(P, Q, drafts, seed, rnd, dev)
    rco, no, outo = oracle.verify_sample(bits(P), bits(Q), drafts.numpy(), seed, rnd)
    assert rc == rco == 0
    assert np.array_equal(n, no) and np.array_equal(out, outo)
    return n


def test_greedy_worked_cases():
    dev = need_gpu()
    rows, cases = [], []
    for line in open(os.path.join(GOLDEN, "greedy_worked_cases.txt")):
        t = line.split()
        if not t or t[0].startswith("#"):
            continue
        if t[0] == "row":
            rows.append([float(v) for v in t[2:]])
        elif t[0] == "case":
            a, b = line[4:].split("->")
            n, o = b.split("|")
            cases.append(([int(v) for v in a.split()], int(n), [int(v) for v in o.split()]))
    P = torch.tensor(rows, dtype=torch.float32).to(torch.bfloat16)[None]
    for d, n_want, out_want in cases:
        rc, n, out = gpu_greedy(P, torch.tensor([d], dtype=torch.int32), dev)
        assert rc == 0 and n[0] == n_want and out[0].tolist() == out_want


def test_single_layer_case_vocab_1024():
    """batch 1, gamma 3, vocab 1024, N(0,2) logits plus a shared N(0,1) offset."""
    dev = need_gpu()
    P, Q, d = syn.logits_shared_offset(1, 3, 1024, seed=0)
    for rnd in range(20):
        rc, n, out = gpu_sample(P, Q, d, 0, rnd, dev)
        rco, no, outo = oracle.verify_sample(bits(P), bits(Q), d.numpy(), 0, rnd)
        assert rc == rco == 0 and np.array_equal(n, no) and np.array_equal(out, outo)
    check_both(P, Q, d, dev)


@pytest.mark.parametrize("B,gamma,V,seed", [
    (1, 1, 2, 0), (3, 2, 7, 1), (2, 4, 8, 2), (4, 16, 1000, 3), (16, 3, 4099, 4),
    (5, 8, 30000, 5), (2, 1, 1, 6), (7, 5, 2048, 7), (1, 16, 70001, 8), (2, 2, 600000, 9),
    # at least two rows per SM: one CTA per row (V % 8 != 0 takes the scalar loads)
    (64, 4, 3001, 10), (40, 7, 1000, 11), (70, 4, 8192, 12)])
def test_random_shapes(B, gamma, V, seed):
    dev = need_gpu()
    P, Q, d = syn.logits_noisy_draft(B, gamma, V, seed, p_std=3.0, q_noise=0.5)
    for rnd in range(3):
        check_both(P, Q, d, dev, seed=seed, rnd=rnd)


@pytest.mark.parametrize("B", [3, 64])
def test_row_statistics_in_workspace(B):
    """The sampled call leaves each row's max and exact fixed-point sum in the
    workspace (rows: P[b][i] then Q[b][i]); they match the oracle's, both for
    chunked rows (B = 3) and one CTA per row (B = 64: 320 rows)."""
    dev = need_gpu()
    gamma, V = 2, 5000
    P, Q, d = syn.logits_noisy_draft(B, gamma, V, 3)
    ws = q.verify_workspace(B, gamma, V, dev)
    gpu_sample(P, Q, d, 1, 1, dev, ws=ws)
    wsb = ws.cpu().numpy()
    rows = B * (2 * gamma + 1)
    rows_g = B * (gamma + 1)
    off_max = (((rows_g + 1024) * 8 + 15) // 16) * 16      # after the (row, chunk) argmax keys
    off_sum = off_max + ((rows * 4 + 15) // 16) * 16
    enc = wsb[off_max:off_max + rows * 4].view(np.uint32)
    S = wsb[off_sum:off_sum + rows * 8].view(np.uint64)
    allrows = np.concatenate([bits(P).reshape(-1, V), bits(Q).reshape(-1, V)])
    for r in range(rows):
        st, E, So, m = oracle.fixed_softmax_row(allrows[r])
        assert int(S[r]) == So, r
        u = np.array([m], np.float32).view(np.uint32)[0]
        want = (~u & 0xFFFFFFFF) if (u & 0x80000000) else (u | 0x80000000)
        assert int(enc[r]) == int(want)


@pytest.mark.parametrize("B,gamma,V,seed", [(16, 4, 128256, 2)])
def test_llama_batch16_full_vocab(B, gamma, V, seed):
    dev = need_gpu()
    P, Q, d = syn.logits_noisy_draft(B, gamma, V, seed, p_std=3.0, q_noise=0.5)
    n = check_both(P, Q, d, dev, seed=seed, rnd=0)
    assert 0 < n.mean() < gamma


@pytest.mark.parametrize("gamma", [2, 4, 8])
def test_qwen_batch32_full_vocab(gamma):
    dev = need_gpu()
    P, Q, d = syn.logits_noisy_draft(32, gamma, 152064, 3 + gamma, p_std=3.0, q_noise=0.5)
    check_both(P, Q, d, dev, seed=gamma, rnd=1)


def test_batch256_vocab128256():
    dev = need_gpu()
    P, Q, d = syn.logits_noisy_draft(256, 4, 128256, 4, p_std=3.0, q_noise=0.5)
    rc, n, out = gpu_sample(P, Q, d, 4, 0, dev)
    rco, no, outo = oracle.verify_sample(bits(P), bits(Q), d.numpy(), 4, 0)
    assert rc == rco == 0 and np.array_equal(n, no) and np.array_equal(out, outo)


def test_degenerate_rows():
    dev = need_gpu()
    B, gamma, V = 6, 3, 64
    P = torch.zeros((B, gamma + 1, V))
    Q = torch.zeros((B, gamma, V))
    d = torch.zeros((B, gamma), dtype=torch.int32)
    P[1] = torch.randn(gamma + 1, V)                       # b=1: Q uniform, P random
    P[2, :, 5:] = float("-inf")                            # b=2: P mass only on 0..4
    d[2] = torch.tensor([7, 1, 2])                         # draft 7 has p = 0: rejected
    Q[3, :, 0] = float("-inf")                             # b=3: q(0) = 0 < p(0)
    P[4], Q[4] = 1.0, 1.0                                  # b=4: p = q uniform
    d[4] = torch.tensor([3, 9, 63])
    P[5, 0, 10] = float("-inf")                            # b=5: p(t) = q(t) = 0 at t = 10
    Q[5, 0, 10] = float("-inf")
    d[5, 0] = 10
    check_both(P.to(torch.bfloat16), Q.to(torch.bfloat16), d, dev)


@pytest.mark.parametrize("B", [2, 64])
@pytest.mark.parametrize("what", ["p_nan", "q_inf", "q_all_neg_inf", "draft_range"])
def test_device_status(what, B):
    dev = need_gpu()
    P, Q, d = syn.logits_noisy_draft(B, 4 if B > 2 else 2, 300, 1)
    if what == "p_nan":
        P[1, 2, 17] = float("nan")
    elif what == "q_inf":
        Q[0, 1, 3] = float("inf")
    elif what == "q_all_neg_inf":
        Q[1, 0, :] = float("-inf")
    else:
        d[1, 1] = 300
    rc, _, _ = gpu_sample(P, Q, d, 0, 0, dev)
    rco, _, _ = oracle.verify_sample(bits(P), bits(Q), d.numpy(), 0, 0)
    assert rc == rco != 0
    if what in ("p_nan", "draft_range"):
        rc, _, _ = gpu_greedy(P, d, dev)
        rco, _, _ = oracle.verify_greedy(bits(P), d.numpy())
        assert rc == rco != 0


def test_first_token_follows_target_on_gpu():
    """chi-square on V = 8: the first emitted token is distributed as p'."""
    from scipy.stats import chi2 as chi2dist
    dev = need_gpu()
    V, B = 8, 1 << 20
    lp = torch.tensor([1.0, 0.5, 0.0, -1.0, 2.0, -0.5, 0.25, 1.5])
    lq = torch.tensor([0.0, 1.5, 1.0, 0.5, 0.0, 1.0, -1.0, 0.5])
    P = torch.stack([lp, lp]).to(torch.bfloat16)[None].expand(B, 2, V).contiguous()
    Q = lq.to(torch.bfloat16)[None, None].expand(B, 1, V).contiguous()
    pq = oracle.fixed_softmax_row(bits(Q[0, 0]))
    q_probs = pq[1].astype(np.float64) / pq[2]
    p_st = oracle.fixed_softmax_row(bits(P[0, 0]))
    p_probs = p_st[1].astype(np.float64) / p_st[2]
    g = np.random.default_rng(5)
    d = torch.from_numpy(g.choice(V, size=(B, 1), p=q_probs).astype(np.int32))
    rc, n, out = gpu_sample(P, Q, d, 99, 0, dev)
    assert rc == 0
    counts = np.bincount(out[:, 0], minlength=V)
    exp = p_probs * B
    c = ((counts - exp) ** 2 / exp).sum()
    assert chi2dist.sf(c, V - 1) > 1e-3, c


def test_expected_accept_length_on_gpu():
    """E[L] = (1 - a^(gamma+1)) / (1 - a) for i.i.d. acceptance a."""
    dev = need_gpu()
    alpha, gamma, B = 0.6, 4, 1 << 18
    lp = torch.tensor([math.log(alpha), math.log(1 - alpha)]).to(torch.bfloat16)
    lq = torch.tensor([0.0, -100.0]).to(torch.bfloat16)
    st, E, S, _ = oracle.fixed_softmax_row(bits(lp))
    a = math.ceil(2 ** 24 * int(E[0]) / S) / 2 ** 24
    P = lp[None, None].expand(B, gamma + 1, 2).contiguous()
    Q = lq[None, None].expand(B, gamma, 2).contiguous()
    rc, n, out = gpu_sample(P, Q, torch.zeros((B, gamma), dtype=torch.int32), 17, 2, dev)
    assert rc == 0
    L = n + 1
    EL = (1 - a ** (gamma + 1)) / (1 - a)
    assert abs(L.mean() - EL) < 4 * L.std() / math.sqrt(B)


@pytest.mark.parametrize("B", [1, 64])
def test_greedy_signed_zero_tie(B):
    """A row whose largest logit is zero with -0 before +0: float comparison
    ties them, so the lower index wins (the oracle's reading), whether the two
    fall in different chunks of the row (B = 1) or one CTA scans the row
    (B = 64)."""
    dev = need_gpu()
    gamma, V = 4, 50000
    P = torch.full((B, gamma + 1, V), -5.0)
    P[:, :, 100] = -0.0
    P[:, :, 40000] = 0.0
    P[:, 1, 7] = 0.0                                       # row 1: +0 first, then -0 at 100
    P = P.to(torch.bfloat16)
    d = torch.full((B, gamma), 100, dtype=torch.int32)
    rc, n, out = gpu_greedy(P, d, dev)
    rco, no, outo = oracle.verify_greedy(bits(P), d.numpy())
    assert rc == rco == 0
    assert np.array_equal(n, no) and np.array_equal(out, outo)
    assert n[0] == 1 and out[0, 1] == 7                    # row 0 argmax 100 (accepted), row 1 argmax 7
