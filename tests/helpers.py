"""Small test helpers: independent restatements used as references by tests."""

import numpy as np


def softmax64(x, T):
    z = np.asarray(x, np.float64) / np.float64(np.float32(T))
    z = z - z.max()
    e = np.exp(z)
    return e / e.sum()


def filtered_probs(x, T, top_k, top_p):
    """Sort-based restatement of the row filter (temperature, then top-k with
    ties to the lower index, then top-p keeping the crossing token), used only
    as a reference for statistical tests; the filter itself is pinned by hand
    examples in test_oracle_pins.py."""
    x = np.asarray(x, np.float64)
    V = x.shape[0]
    T = np.float64(np.float32(T))
    order = np.lexsort((np.arange(V), -x))
    K = top_k if 0 < top_k < V else V
    keep = order[:K]
    w = np.exp((x[keep] - x[keep[0]]) / T)
    P = w / w.sum()
    if top_p < 1:
        before = np.concatenate([[0.0], np.cumsum(P)[:-1]])
        n = int((before < np.float64(np.float32(top_p))).sum())
        keep, w = keep[:n], w[:n]
    p = np.zeros(V)
    p[keep] = w / w.sum()
    return p


def chi2_pvalue(counts, probs, min_expected=5.0):
    """Pearson chi-square goodness of fit, pooling cells with expected < min_expected."""
    from scipy import stats
    counts = np.asarray(counts, np.float64)
    n = counts.sum()
    exp = np.asarray(probs, np.float64) * n
    big = exp >= min_expected
    c = list(counts[big])
    e = list(exp[big])
    if (~big).any():
        c.append(counts[~big].sum())
        e.append(exp[~big].sum())
    c, e = np.array(c), np.array(e)
    # cells with zero expected mass must also hold zero counts
    if (e == 0).any():
        return 0.0 if c[e == 0].sum() > 0 else stats.chisquare(c[e > 0], e[e > 0]).pvalue
    return stats.chisquare(c, e).pvalue
