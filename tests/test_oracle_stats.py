"""Statistical pins of the oracle (no GPU): chi-square goodness of fit of the
emitted tokens against the target distributions over 10^6 seeded trials
(V <= 64), and the closed form E = (1 - a^(k+1)) / (1 - a) at k = 15
("Speculative decoding and multi-token prediction", "Acceptance rate is the
whole economics"; "FlashMap…" §4 identity P(Y=y) = p(y))."""

import numpy as np
import pytest

import oracle
from helpers import chi2_pvalue, filtered_probs

N_TRIALS = 1_000_000
P_REJECT = 1e-3


def run_trials(t, d, T, top_k, top_p, q_sample, seed, n=N_TRIALS):
    rng = np.random.default_rng(seed)
    k = t.shape[0] - 1
    V = t.shape[1]
    x = np.empty((n, k), np.int32)
    for i in range(k):
        x[:, i] = rng.choice(V, size=n, p=q_sample[i])
    u = rng.random((n, k + 1), dtype=np.float32)
    return oracle.verify_trials(t, d, T, top_k, top_p, x, u)


def positional_pvalues(acc, tok, p):
    k = len(p) - 1
    V = p[0].shape[0]
    out = []
    for j in range(k + 1):
        sel = acc >= j
        counts = np.bincount(tok[sel, j], minlength=V)
        out.append(chi2_pvalue(counts, p[j]))
    return out


@pytest.mark.slow
@pytest.mark.parametrize("V", [8, 64])
def test_chi_square_emitted_tokens_follow_target(V):
    rng = np.random.default_rng(100 + V)
    k = 3
    t = rng.normal(size=(k + 1, V)) * 1.2
    d = t[:k] + rng.normal(size=(k, V)) * 0.8
    T = 0.9
    p = [filtered_probs(r, T, 0, 1.0) for r in t]
    q = [filtered_probs(r, T, 0, 1.0) for r in d]
    acc, tok, _ = run_trials(t, d, T, 0, 1.0, q, seed=V)
    pv = positional_pvalues(acc, tok, p)
    assert min(pv) > P_REJECT, pv
    # acceptance at position 0 has probability sum_y min(p_0, q_0)
    a0 = np.minimum(p[0], q[0]).sum()
    assert abs((acc >= 1).mean() - a0) < 5 * np.sqrt(a0 * (1 - a0) / N_TRIALS)


@pytest.mark.slow
def test_chi_square_with_identical_filters():
    rng = np.random.default_rng(7)
    V, k, T, tk, tp = 64, 3, 1.1, 5, 0.8
    t = rng.normal(size=(k + 1, V)) * 1.5
    d = t[:k] + rng.normal(size=(k, V)) * 0.5
    p = [filtered_probs(r, T, tk, tp) for r in t]
    q = [filtered_probs(r, T, tk, tp) for r in d]
    acc, tok, _ = run_trials(t, d, T, tk, tp, q, seed=8)
    pv = positional_pvalues(acc, tok, p)
    assert min(pv) > P_REJECT, pv


@pytest.mark.slow
def test_negative_control_filter_applied_to_draft_only_is_detected():
    """Sampling parameters applied inconsistently to draft and target (the
    failure mode named in "Speculative decoding and multi-token prediction",
    "Practical guidance"): drafts come from the filtered q, the verifier is
    told there is no filter.  The emitted law must then miss p."""
    rng = np.random.default_rng(7)
    V, k, T, tk, tp = 64, 3, 1.1, 5, 0.8
    t = rng.normal(size=(k + 1, V)) * 1.5
    d = t[:k] + rng.normal(size=(k, V)) * 0.5
    p_unf = [filtered_probs(r, T, 0, 1.0) for r in t]
    q_f = [filtered_probs(r, T, tk, tp) for r in d]
    acc, tok, _ = run_trials(t, d, T, 0, 1.0, q_f, seed=9, n=200_000)
    pv = positional_pvalues(acc, tok, p_unf)
    assert pv[0] < 1e-6


def alpha_rows(alpha, k, V=8):
    r = np.array([.25] * 4 + [0] * 4)
    a = np.array([0] * 4 + [.5, .5, 0, 0])
    b = np.array([0] * 4 + [0, 0, .5, .5])
    p = alpha * r + (1 - alpha) * a
    q = alpha * r + (1 - alpha) * b
    with np.errstate(divide="ignore"):
        return np.log(np.tile(p, (k + 1, 1))), np.log(np.tile(q, (k, 1))), p, q


@pytest.mark.slow
@pytest.mark.parametrize("alpha", [0.3, 0.5, 0.7, 0.8])
def test_closed_form_k15_monte_carlo(alpha):
    k = 15
    t, d, p, q = alpha_rows(alpha, k)
    acc, tok, _ = run_trials(t, d, 1.0, 0, 1.0, [q] * k, seed=int(alpha * 100))
    E = (1 - alpha ** (k + 1)) / (1 - alpha)
    tau = acc + 1.0
    sigma = tau.std() / np.sqrt(len(tau))
    assert abs(tau.mean() - E) < 4 * sigma
    geo = np.array([alpha ** j * (1 - alpha) for j in range(k)] + [alpha ** k])
    assert chi2_pvalue(np.bincount(acc, minlength=k + 1), geo) > P_REJECT
