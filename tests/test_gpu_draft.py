"""Draft-side sampling with the draft statistics: tokens and confidence
bit-exact against the oracle, entropy within 1e-4 (1 + H) of the oracle's
fp64 value, on the one-launch cluster path (V >= 2048, fewer than two rows
per SM), the chunked path (shorter rows) and the row-per-CTA path (many
rows), with V a multiple of 8 or not; special rows, status codes on each
path, and a full round (drafts drawn here, then sampled verification)
against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from quantized_speculative_decoding_shared_gb300 import binding as q, synthetic as syn
from gpuhelp import bits, need_gpu, read_status, status

pytestmark = pytest.mark.gpu
NEG_INF = float("-inf")


def run(Q, seed, rnd, step, dev, ws=None):
    st = status(dev)
    tok, conf, ent = q.draft_sample(Q.to(dev), seed, rnd, step, workspace=ws, dev_status=st)
    return read_status(st), tok.cpu().numpy(), conf.cpu().numpy(), ent.cpu().numpy()


def compare(Q, seed, rnd, step, dev):
    rc, tok, conf, ent = run(Q, seed, rnd, step, dev)
    rco, toko, confo, ento = oracle.draft_sample(bits(Q), seed, rnd, step)
    assert rc == rco == 0
    assert np.array_equal(tok, toko)
    assert np.array_equal(conf.view(np.uint32), confo.view(np.uint32))
    assert np.all(np.abs(ent.astype(np.float64) - ento) <= 1e-4 * (1 + np.abs(ento))), \
        np.abs(ent - ento).max()
    return tok


# (320, 4096) and (310, 999): at least two rows per SM, one CTA per row;
# V >= 2048 below that: a cluster of CTAs per row (2048 the smallest, 20001
# with element-wise loads, 303 rows the most, 196608 the longest row a
# cluster of 16 holds in registers); shorter rows: rows split into chunks
# (2047 the longest), as are longer ones (196616).  V = 1001, 999, 7:
# element-wise loads.
@pytest.mark.parametrize("B,V,seed", [(1, 1024, 0), (3, 1001, 1), (1, 128256, 2), (16, 128256, 3),
                                      (5, 7, 4), (320, 4096, 5), (310, 999, 6), (32, 152064, 7),
                                      (2, 2048, 8), (2, 2047, 9), (7, 20001, 10), (303, 2048, 11),
                                      (2, 196608, 12), (2, 196616, 13)])
def test_draft_sample_matches_oracle(B, V, seed):
    dev = need_gpu()
    g = torch.Generator().manual_seed(seed)
    Q = (torch.randn((B, V), generator=g) * 3.0).to(torch.bfloat16)
    compare(Q, 11 + seed, 5, 1 + seed % 16, dev)


def test_draft_special_rows():
    """uniform, one finite logit, k equal logits with the rest -inf, a row
    whose maximum repeats, and -inf scattered through a random row"""
    dev = need_gpu()
    V = 20000
    rows = [torch.full((V,), 0.5), torch.full((V,), NEG_INF), torch.full((V,), NEG_INF),
            torch.zeros(V), torch.randn(V, generator=torch.Generator().manual_seed(9)) * 2]
    rows[1][12345] = 3.0
    rows[2][torch.randperm(V, generator=torch.Generator().manual_seed(8))[:37]] = -1.25
    rows[3][[5, 600, 19999]] = 4.0
    rows[4][torch.randperm(V, generator=torch.Generator().manual_seed(7))[:500]] = NEG_INF
    Q = torch.stack(rows).to(torch.bfloat16)
    tok = compare(Q, 3, 1, 2, dev)
    assert tok[1] == 12345 and tok[2] in set(np.flatnonzero(Q[2].float().numpy() > NEG_INF).tolist())


def test_draft_deterministic_and_slots():
    """the same call twice gives the same bits; another draft position or
    round draws other tokens"""
    dev = need_gpu()
    Q = (torch.randn((64, 4096), generator=torch.Generator().manual_seed(1)) * 0.5).to(torch.bfloat16)
    ws = q.draft_workspace(64, 4096, dev)
    a = run(Q, 1, 2, 3, dev, ws)
    b = run(Q, 1, 2, 3, dev, ws)
    assert all(np.array_equal(x, y) for x, y in zip(a[1:], b[1:]))
    c = run(Q, 1, 2, 4, dev, ws)
    d = run(Q, 1, 3, 3, dev, ws)
    assert (a[1] != c[1]).any() and (a[1] != d[1]).any()
    assert np.array_equal(a[2], c[2]) and np.array_equal(a[3], c[3])   # statistics do not depend on the uniform


@pytest.mark.parametrize("V", [3000, 1500])            # the cluster path, the chunked path
def test_draft_status(V):
    dev = need_gpu()
    Q = torch.randn((4, V), generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    for bad in (float("nan"), float("inf")):
        Q2 = Q.clone()
        Q2[2, V - 1234] = bad
        assert run(Q2, 0, 0, 1, dev)[0] == q.ERR_NONFINITE
        assert oracle.draft_sample(bits(Q2), 0, 0, 1)[0] == oracle.ERR_NONFINITE
    Q3 = Q.clone()
    Q3[1] = NEG_INF
    assert run(Q3, 0, 0, 1, dev)[0] == q.ERR_NONFINITE


def test_round_drafts_then_sampled_verification():
    """gamma draft positions drawn here (step i + 1 for position i), then the
    sampled verification of those drafts: every token and acceptance count
    equal to the same round run through the oracle"""
    dev = need_gpu()
    B, g, V = 8, 4, 128256
    P, Q, _ = syn.logits_noisy_draft(B, g, V, 21, p_std=3.0, q_noise=0.5)
    Qd = Q.to(dev)
    drafts = torch.stack([q.draft_sample(Qd[:, i, :].contiguous(), 77, 9, i + 1)[0] for i in range(g)], 1)
    n_acc, out = q.verify_sample(P.to(dev), Qd, drafts, 77, 9)
    do = np.stack([oracle.draft_sample(bits(Q[:, i, :].contiguous()), 77, 9, i + 1)[1] for i in range(g)], 1)
    st, no, oo = oracle.verify_sample(bits(P), bits(Q), do, 77, 9)
    assert st == 0
    assert np.array_equal(drafts.cpu().numpy(), do)
    assert np.array_equal(n_acc.cpu().numpy(), no) and np.array_equal(out.cpu().numpy(), oo)
