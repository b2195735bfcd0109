"""Recompute the draft-noise scale of the B=256, V=128256, K=5, T=0.7 workload.

The workload asks for a mean acceptance of about 0.75, where the acceptance of
one position is sum_v min(p_v, q_v) (the probability that the accept test
passes, "Speculative Decoding: from idea to SOTA", section 3: beta =
sum_x q(x) * min(1, p(x)/q(x))).  This script bisects sigma with the oracle's
softmax on a sample of generated rows and prints the result; the generator
module stores the value it printed (0.445).

    python tests/golden/calibrate_sigma.py [--rows 64]
"""
import argparse
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from speculative_decoding_verification_52_gb300 import inputs as gen  # noqa: E402


def mean_acceptance(sigma, seqs, T=0.7):
    b = gen.gaussian_chain(256, 128256, 5, sigma=sigma, T=T, dtype=gen.BF16, seed=52_300, seqs=seqs)
    tot, n = 0.0, 0
    for i in range(b.B):
        zt = gen.as_f64(b.target[i], b.dtype)
        zd = gen.as_f64(b.draft[i], b.dtype)
        for t in range(b.K):
            p = oracle.softmax(zt[t], T)
            q = oracle.softmax(zd[t], T)
            tot += float(np.minimum(p, q).sum())
            n += 1
    return tot / n


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--seqs", type=int, default=8)
    ap.add_argument("--target", type=float, default=0.75)
    a = ap.parse_args()
    seqs = list(range(a.seqs))
    lo, hi = 0.3, 0.6
    for _ in range(12):
        mid = 0.5 * (lo + hi)
        if mean_acceptance(mid, seqs) > a.target:
            lo = mid
        else:
            hi = mid
    print(f"sigma = {0.5 * (lo + hi):.4f}  (acceptance {mean_acceptance(0.5 * (lo + hi), seqs):.4f})")


if __name__ == "__main__":
    main()
