"""Pins of the adaptive-k oracle (oracle/adapt.py) against the values printed
in "Speculative decoding and multi-token prediction", section "Acceptance rate
is the whole economics", and against closed forms and simulation."""

import os

import numpy as np
import pytest

from oracle.adapt import adapt_k, expected_tokens, next_k, speedup

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "expected_tokens_per_pass.txt")


def golden_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            a, k, e = line.split()
            rows.append((float(a), int(k), float(e)))
    return rows


@pytest.mark.parametrize("alpha,k,printed", golden_rows())
def test_expected_tokens_match_the_printed_values(alpha, k, printed):
    assert round(expected_tokens(alpha, k), 2) == printed


@pytest.mark.parametrize("alpha,printed", [(0.3, 1.0), (0.5, 1.4), (0.7, 2.0), (0.8, 2.4)])
def test_speedup_at_c_point_one_and_k_four_matches_the_printed_values(alpha, printed):
    # the page rounds E / 1.4 to one decimal ("about 1.0x at alpha 0.3 ...")
    assert round(speedup(alpha, 4, 0.1), 1) == printed


def test_the_pages_worked_length():
    # "about k equal to 6 at alpha 0.7 and c 0.1"
    assert next_k(0.7, 0.1, 1, 32) == 6


def test_next_k_is_where_the_geometric_tail_crosses_c():
    for alpha in np.linspace(0.05, 0.97, 40):
        for c in (0.02, 0.05, 0.1, 0.3):
            k = next_k(alpha, c, 1, 32)
            if alpha > c:
                assert alpha ** k > c * (1 - 1e-12)
                if k < 32:
                    assert alpha ** (k + 1) <= c * (1 + 1e-12)
            else:
                assert k == 1                    # not even one draft pays: k_min


def test_closed_form_matches_its_sum():
    for alpha in (0.1, 0.5, 0.9, 0.999):
        for k in (0, 1, 4, 15):
            assert abs(expected_tokens(alpha, k) - sum(alpha ** i for i in range(k + 1))) < 1e-9


def test_estimate_converges_to_the_acceptance_rate():
    """Accept lengths from the verification rule with i.i.d. acceptance alpha:
    the estimate (no decay) approaches alpha."""
    rng = np.random.default_rng(0)
    for alpha in (0.3, 0.6, 0.85):
        k = 8
        s = f = 0.0
        for _ in range(4000):
            acc = rng.random(k) < alpha
            L = int(np.argmin(acc)) if not acc.all() else k
            _, s2, f2, a = adapt_k([L], [k], [s], [f], 1.0, 0.1, 1, 16)
            s, f = s2[0], f2[0]
        assert abs(a[0] - alpha) < 0.02


def test_failed_requests_keep_their_state_and_k():
    kn, s2, f2, _ = adapt_k([-1, 3], [5, 5], [2.0, 2.0], [1.0, 1.0], 0.9, 0.1, 1, 8)
    assert kn[0] == 5 and s2[0] == 2.0 and f2[0] == 1.0
    assert s2[1] == 0.9 * 2.0 + 3 and f2[1] == 0.9 * 1.0 + 1
