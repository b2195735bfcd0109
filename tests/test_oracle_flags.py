"""Pins of two oracle parts that the GPU parity tests lean on: the residual row
(the reference for the device's replacement distribution, "within 1e-6" rule)
and the tolerance flags that take near-tie decisions out of the bit-exact
comparison.

The residual row is checked against scipy's softmax with the whole draft row
subtracted ("Speculative Decoding: from idea to SOTA", section 3, resampling
rule p' = max(0, p - q) / sum; "Speculative decoding: draft, verify, repeat",
step 2), at every (sequence, position) of a small batch, so a wrong row offset
or a wrong bonus-row branch fails.  The flags are checked on hand-built
decisions placed 5e-7 and 2e-6 from their boundary, so a flag that fires too
often (or never) fails."""
import numpy as np
import pytest
from scipy.special import softmax as sp_softmax

from speculative_decoding_verification_52_gb300 import inputs as gen

TOL = 1e-6


def _batch(seed, B, K, V, dtype):
    rng = np.random.default_rng(seed)
    tgt = rng.standard_normal((B, K + 1, V)) * 1.5
    dr = tgt[:, :K] + rng.standard_normal((B, K, V)) * 0.8
    if dtype == "bf16":
        tb, db = gen.f32_to_bf16_bits(tgt.astype(np.float32)), gen.f32_to_bf16_bits(dr.astype(np.float32))
        return tb, db, gen.bf16_bits_to_f64(tb), gen.bf16_bits_to_f64(db)
    tf, df = tgt.astype(np.float32), dr.astype(np.float32)
    return tf, df, tf.astype(np.float64), df.astype(np.float64)


def _expected_residual(p, q):
    w = np.clip(p - q, 0.0, None)
    return w / w.sum(), w.sum()


# --- orc_residual_row ---------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_residual_row_every_position(orc, dtype):
    """Each (b, t < K) against scipy softmax(target/T) - softmax(draft/T),
    clipped at 0 and renormalised; t == K against softmax(target/T) alone."""
    B, K, V, T = 3, 3, 37, 0.8
    tgt, dr, tgt64, dr64 = _batch(11, B, K, V, dtype)
    for b in range(B):
        for t in range(K + 1):
            row, mass = orc.residual_row(tgt, dtype, dr, dtype, False, T, b, t)
            p = sp_softmax(tgt64[b, t] / T)
            if t < K:
                exp_row, exp_mass = _expected_residual(p, sp_softmax(dr64[b, t] / T))
            else:
                exp_row, exp_mass = p, 1.0
            np.testing.assert_allclose(row, exp_row, rtol=0, atol=1e-14)
            assert mass == pytest.approx(exp_mass, abs=1e-14)
            assert row.sum() == pytest.approx(1.0, abs=1e-14)


def test_residual_row_rows_are_distinct(orc):
    """Neighbouring (b, t) give different rows, so the comparison above would
    see an offset slip (e.g. a stride of K instead of K+1 over target rows)."""
    B, K, V, T = 2, 3, 37, 1.0
    tgt, dr, _, _ = _batch(12, B, K, V, "f32")
    rows = [orc.residual_row(tgt, "f32", dr, "f32", False, T, b, t)[0] for b in range(B) for t in range(K + 1)]
    for i in range(len(rows)):
        for j in range(i + 1, len(rows)):
            assert np.abs(rows[i] - rows[j]).max() > 1e-3


def test_residual_row_zero_mass_falls_back_to_p(orc):
    """A draft row equal to the target row (same bits) gives p == q, so
    sum (p - q)+ == 0 and the row falls back to p_t with mass sum p_t."""
    B, K, V, T = 2, 2, 29, 0.6
    tgt, dr, tgt64, _ = _batch(13, B, K, V, "f32")
    dr[1, 1] = tgt[1, 1]
    row, mass = orc.residual_row(tgt, "f32", dr, "f32", False, T, 1, 1)
    p = sp_softmax(tgt64[1, 1] / T)
    np.testing.assert_allclose(row, p, rtol=0, atol=1e-14)
    assert mass == pytest.approx(1.0, abs=1e-14)
    # its neighbour (b=1, t=0) still subtracts its own draft row
    row0, _ = orc.residual_row(tgt, "f32", dr, "f32", False, T, 1, 0)
    assert np.abs(row0 - sp_softmax(tgt64[1, 0] / T)).max() > 1e-3


def test_residual_row_with_draft_probabilities(orc):
    """Draft probabilities are subtracted exactly as given (not renormalised,
    not tempered)."""
    B, K, V, T = 2, 2, 23, 0.9
    rng = np.random.default_rng(14)
    tgt = (rng.standard_normal((B, K + 1, V)) * 1.2).astype(np.float32)
    q = rng.random((B, K, V)).astype(np.float32)
    q /= q.sum(axis=-1, keepdims=True) * np.float32(1.05)   # sums to ~0.95: used as given
    for b in range(B):
        for t in range(K + 1):
            row, mass = orc.residual_row(tgt, "f32", q, "f32", True, T, b, t)
            p = sp_softmax(tgt[b, t].astype(np.float64) / T)
            if t < K:
                exp_row, exp_mass = _expected_residual(p, q[b, t].astype(np.float64))
            else:
                exp_row, exp_mass = p, 1.0
            np.testing.assert_allclose(row, exp_row, rtol=0, atol=1e-14)
            assert mass == pytest.approx(exp_mass, abs=1e-14)


# --- tolerance flags ------------------------------------------------------------

def _f32_near(x):
    """The float32 nearest x, and its distance from x."""
    f = np.float32(x)
    return f, abs(float(f) - x)


def _flag_case(offset, t_near):
    """One sequence, K = 3, V = 4, target given as logits log p (T = 1), draft
    as probabilities.  Positions before t_near accept with a wide margin, those
    after it reject with one (u = 0.9 against ratios 0.5 and 0.67); the accept
    test at t_near has u = p(x)/q(x) + offset (to float32 rounding)."""
    p = np.array([[0.30, 0.20, 0.40, 0.10],
                  [0.25, 0.25, 0.25, 0.25],
                  [0.10, 0.50, 0.20, 0.20],
                  [0.40, 0.30, 0.20, 0.10]])
    q = np.array([[0.60, 0.10, 0.20, 0.10],
                  [0.10, 0.50, 0.20, 0.20],
                  [0.20, 0.40, 0.30, 0.10]], np.float32)
    x = np.array([0, 1, 2], np.int32)
    target = np.log(p).astype(np.float32)
    # the ratio the oracle sees: softmax of the float32 logits, over float32 q
    ratio = sp_softmax(target.astype(np.float64), axis=-1)[np.arange(3), x] / q.astype(np.float64)[np.arange(3), x]
    u = np.full((4, 2), 0.9, np.float32)   # later positions reject, far from their boundary
    u[:, 1] = 0.123
    for t in range(t_near):
        u[t, 0] = np.float32(ratio[t] * 0.25)   # accepts, far from its boundary
    u[t_near, 0], _ = _f32_near(ratio[t_near] + offset)
    dist = abs(float(u[t_near, 0]) - ratio[t_near])
    return target[None], q[None], x[None], u[None], ratio, dist


@pytest.mark.parametrize("t_near", [0, 1, 2])
@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_near_accept_flag_set_within_tolerance(orc, t_near, sign):
    target, q, x, u, ratio, dist = _flag_case(sign * 5e-7, t_near)
    assert 4e-7 < dist < 6e-7
    r = orc.verify_sample(target, "f32", q, "f32", True, x, u, 1.0)
    assert int(r["near_accept"][0]) == t_near
    # the decision itself follows the strict rule u < p/q
    accepted = float(u[0, t_near, 0]) < ratio[t_near]
    n = int(r["num_accepted"][0])
    assert (n > t_near) == accepted


@pytest.mark.parametrize("t_near", [0, 1, 2])
@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_near_accept_flag_clear_outside_tolerance(orc, t_near, sign):
    target, q, x, u, ratio, dist = _flag_case(sign * 2e-6, t_near)
    assert 1.9e-6 < dist < 2.1e-6
    r = orc.verify_sample(target, "f32", q, "f32", True, x, u, 1.0)
    assert int(r["near_accept"][0]) == -1


def test_near_accept_flags_first_near_position_only(orc):
    """Two near tests in a row (both accepting): the flag names the first."""
    target, q, x, u, ratio, _ = _flag_case(-5e-7, 0)
    u[0, 1, 0], _ = _f32_near(ratio[1] - 5e-7)
    r = orc.verify_sample(target, "f32", q, "f32", True, x, u, 1.0)
    assert int(r["near_accept"][0]) == 0


def _cdf_case(offset):
    """One sequence, K = 1, V = 5, rejected at t = 0 (u0 close to 1).  The
    replacement draw's uniform sits `offset` (relative to R) past the CDF
    boundary after token 1 of w = (p - q)+."""
    p = np.array([[0.30, 0.25, 0.05, 0.30, 0.10], [0.2, 0.2, 0.2, 0.2, 0.2]])
    q = np.array([[0.10, 0.05, 0.45, 0.20, 0.20]], np.float32)
    target = np.log(p).astype(np.float32)
    p64 = sp_softmax(target.astype(np.float64), axis=-1)
    w = np.clip(p64[0] - q[0].astype(np.float64), 0.0, None)
    C = np.cumsum(w) / w.sum()
    u = np.array([[0.999, 0.0], [0.5, 0.5]], np.float32)
    u[0, 1], _ = _f32_near(C[1] + offset)
    dist = abs(float(u[0, 1]) - C[1])
    return target[None], q[None], np.array([[2]], np.int32), u[None], C, dist


@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_near_cdf_flag(orc, sign):
    target, q, x, u, C, dist = _cdf_case(sign * 5e-7)
    assert 4e-7 < dist < 6e-7
    r = orc.verify_sample(target, "f32", q, "f32", True, x, u, 1.0)
    assert int(r["num_accepted"][0]) == 0
    # w = (0.2, 0.2, 0, 0.1, 0): just past the boundary after token 1 the draw
    # skips the zero-weight token 2 and lands on 3; just before it, on 1
    assert int(r["out_tokens"][0, 0]) == (3 if sign > 0 else 1)
    assert int(r["near_cdf"][0]) == 1
    assert int(r["near_accept"][0]) == -1

    target, q, x, u, C, dist = _cdf_case(sign * 2e-6)
    assert 1.9e-6 < dist < 2.1e-6
    r = orc.verify_sample(target, "f32", q, "f32", True, x, u, 1.0)
    assert int(r["near_cdf"][0]) == 0


def test_near_flags_off_for_bonus_far_from_boundary(orc):
    """All accepted, bonus draw far from every boundary of p_K: no flag."""
    target, q, x, u, ratio, _ = _flag_case(0.0, 0)
    for t in range(3):
        u[0, t, 0] = np.float32(ratio[t] * 0.25)
    u[0, 3, 1] = np.float32(0.2)          # p_K CDF: 0.4, 0.7, 0.9, 1.0
    r = orc.verify_sample(target, "f32", q, "f32", True, x, u, 1.0)
    assert int(r["num_accepted"][0]) == 3
    assert int(r["out_tokens"][0, 3]) == 0
    assert int(r["near_accept"][0]) == -1 and int(r["near_cdf"][0]) == 0
    pK = sp_softmax(target[0, 3].astype(np.float64))
    u[0, 3, 1], _ = _f32_near(pK[0] + 5e-7)   # just past the boundary after token 0
    r = orc.verify_sample(target, "f32", q, "f32", True, x, u, 1.0)
    assert int(r["out_tokens"][0, 3]) == 1
    assert int(r["near_cdf"][0]) == 1
