"""The pages' acceptance measurements, run on the GPU.

* "Speculative decoding: draft, verify, repeat", step 4 measures the acceptance
  rate against the divergence of the draft from the verifier.  Position 0 of
  every sequence is accepted with probability sum_v min(p, q) ("Speculative
  Decoding: from idea to SOTA", section 3), so the empirical accept rate of
  spec_verify_sample over many sequences must match the mean of spec_row_stats'
  alpha within its standard error, at every noise level of the draft.
* "Speculative decoding and EAGLE", section "Expected speedup" and its
  exercises: with i.i.d. per-position acceptance alpha, a target pass yields
  (1 - alpha^(K+1)) / (1 - alpha) tokens on average.  The controlled-copy
  generator makes acceptance i.i.d. across positions, so the mean of
  num_accepted + 1 must match the closed form at the realised alpha.
"""
import numpy as np
import pytest
import torch

import gpu_util as gu
import speculative_decoding_verification_52_gb300 as sv
from speculative_decoding_verification_52_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

SIGMAS = (0.1, 0.6, 2.0)


def _gpu(b):
    t, d = gu.dev_tensor(b.target, "f32"), gu.dev_tensor(b.draft, "f32")
    alpha, kl, tv = sv.spec_row_stats(t, d, b.T)
    _, n = sv.spec_verify_sample(t, d, gu.i32(b.draft_tokens), gu.f32(b.uniforms), b.T)
    return (alpha.cpu().numpy().astype(np.float64), kl.cpu().numpy().astype(np.float64),
            tv.cpu().numpy().astype(np.float64), n.cpu().numpy())


def test_accept_rate_follows_sum_min_across_noise_levels(orc):
    """10,000 one-draft sequences in all (V=2048, f32, T=1) at three noise
    levels: the accept rate of position 0 equals the mean sum min(p, q) within
    four standard errors; alpha falls and KL(q||p) rises with the noise; each
    row obeys Pinsker's bound 1 - alpha = TV <= sqrt(KL / 2)."""
    rates, alphas, kls = [], [], []
    for i, s in enumerate(SIGMAS):
        B = 4000 if i < 2 else 2000
        b = gen.gaussian_chain_batch(B, 2048, 1, sigma=s, T=1.0, seed=52_610 + i)
        a, kl, tv, n = _gpu(b)
        m = a[:, 0].mean()
        acc = (n >= 1).mean()
        se = np.sqrt(m * (1.0 - m) / B)
        assert abs(acc - m) < 4 * se + 1e-3, (s, acc, m, se)
        assert (1.0 - a[:, 0] <= np.sqrt(kl[:, 0] / 2.0) + 1e-5).all()
        np.testing.assert_allclose(tv, 1.0 - a, atol=2e-6)
        # the statistics themselves against the oracle on a few sequences
        r = orc.row_stats(b.target[:8], "f32", b.draft[:8], "f32", False, 1.0)
        np.testing.assert_allclose(a[:8], r[0], rtol=0, atol=2e-6)
        np.testing.assert_allclose(kl[:8], r[1], rtol=1e-5, atol=1e-5)
        rates.append(acc)
        alphas.append(m)
        kls.append(kl[:, 0].mean())
    assert alphas[0] > alphas[1] > alphas[2]
    assert kls[0] < kls[1] < kls[2]
    assert rates[0] > rates[1] > rates[2]


@pytest.mark.parametrize("copy_prob", [0.04, 0.42, 0.81])
def test_tokens_per_pass_match_closed_form(copy_prob):
    """Tokens per target pass against K at alpha ~ 0.5 / 0.7 / 0.9."""
    for K in (2, 5, 8):
        b = gen.controlled_chain_batch(3000, K, 1024, copy_prob, 1.0, seed=52_660 + K)
        a, _, _, n = _gpu(b)
        alpha = a.mean()
        tok = n.astype(np.float64) + 1.0
        closed = (1.0 - alpha ** (K + 1)) / (1.0 - alpha)
        se = tok.std() / np.sqrt(len(tok))
        assert abs(tok.mean() - closed) < 4 * se + 0.01, (copy_prob, K, tok.mean(), closed, se)
        assert (n >= 0).all() and (n <= K).all()
