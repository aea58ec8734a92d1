"""Draft-logit noise for the Qwen2.5-7B batch-32 workload, found by bisection
on the oracle.

The workload draws target logits P ~ N(0, 3^2) over V = 152064 and draft
logits Q = P + N(0, sigma_q^2); sigma_q is chosen so that the mean
acceptance probability per draft position, sum_v min(p'_v, q'_v) with p', q'
the oracle's fixed-point softmax weights E / S (SpecQuant summary page,
results: acceptance rates of 57.9-66.1 %), is 0.60.  Writes
qwen_q_noise.json beside this file.  Uses only the oracle and the seeded
input generator.

    python tests/golden/calibrate_q_noise.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from quantized_speculative_decoding_shared_gb300 import synthetic as syn  # noqa: E402

V, ROWS, SEED, TARGET = 152064, 64, 3, 0.60


def acceptance(sigma: float) -> float:
    P, Q, _ = syn.logits_noisy_draft(ROWS, 1, V, SEED, p_std=3.0, q_noise=sigma)
    Pb, Qb = syn.bits16(P), syn.bits16(Q)
    total = 0.0
    for b in range(ROWS):
        st_p, Ep, Sp, _ = oracle.fixed_softmax_row(Pb[b, 0])
        st_q, Eq, Sq, _ = oracle.fixed_softmax_row(Qb[b, 0])
        assert st_p == 0 and st_q == 0
        # sum_v min(Ep / Sp, Eq / Sq), in exact integers, then one division
        m = np.minimum(Ep.astype(object) * Sq, Eq.astype(object) * Sp)
        total += float(sum(m)) / (Sp * Sq)
    return total / ROWS


def main():
    lo, hi = 0.05, 4.0          # acceptance falls as the noise grows
    a_lo, a_hi = acceptance(lo), acceptance(hi)
    assert a_lo > TARGET > a_hi, (a_lo, a_hi)
    for _ in range(22):
        mid = 0.5 * (lo + hi)
        if acceptance(mid) > TARGET:
            lo = mid
        else:
            hi = mid
    sigma = 0.5 * (lo + hi)
    out = {"workload": "qwen2.5-7b-b32 (V 152064, target logits N(0, 3^2))", "rows": ROWS, "seed": SEED,
           "target_acceptance": TARGET, "q_noise": round(sigma, 4), "acceptance": round(acceptance(sigma), 4)}
    with open(os.path.join(HERE, "qwen_q_noise.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")
    print(out)


if __name__ == "__main__":
    main()
