"""Pins of the oracle to facts outside itself (no GPU).

Each test checks the oracle against something the pages or mathematics fix:
library routines for the special cases they cover (softmax, argmax), closed
forms computed by hand, the exact output law obtained by enumerating the
oracle's piecewise-constant dependence on its uniforms (losslessness, "FlashMap…"
§4 identity P(Y=y) = p(y)), and the page's printed expected-tokens-per-pass
values ("Speculative decoding and multi-token prediction", "Acceptance rate is
the whole economics").
"""

import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle
from helpers import filtered_probs

HERE = os.path.dirname(os.path.abspath(__file__))


# --------------------------------------------------------------------------
# Row distributions: library special cases and hand-computed filter examples.
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float64])
@pytest.mark.parametrize("T", [0.3, 0.7, 1.0, 2.5])
def test_softmax_equals_torch_softmax(dtype, T):
    g = torch.Generator().manual_seed(7)
    x = (torch.randn(3000, generator=g) * 3).to(dtype)
    p, m = oracle.row_probs(x, T)
    # the temperature travels as float32, like every per-request parameter
    ref = torch.softmax(x.double() / float(np.float32(T)), dim=0).numpy()
    assert m == math.inf
    np.testing.assert_allclose(p, ref, rtol=1e-12, atol=0)


def test_temperature_changes_distribution():
    x = torch.tensor([2.0, 1.0, 0.0, -1.0], dtype=torch.float64)
    p1, _ = oracle.row_probs(x, 1.0)
    p2, _ = oracle.row_probs(x, 2.0)
    assert abs(p1[0] - math.e**2 / sum(math.e**v for v in (2, 1, 0, -1))) < 1e-15
    assert abs(p2[0] - math.e / sum(math.e**(v / 2) for v in (2, 1, 0, -1))) < 1e-15


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_argmax_equals_torch_argmax_first_index_on_ties(dtype):
    g = torch.Generator().manual_seed(3)
    for _ in range(50):
        x = torch.randint(-3, 3, (257,), generator=g).to(dtype)  # many ties
        assert oracle.argmax(x) == int(torch.argmax(x))
    x = torch.full((9,), -math.inf, dtype=torch.float32)
    assert oracle.argmax(x) == 0
    x[4] = float("nan")
    assert oracle.argmax(x) == -1


DYADIC = np.log(np.array([0.5, 0.25, 0.125, 0.125]))


@pytest.mark.parametrize("top_k,top_p,expected", [
    (2, 1.0, [2 / 3, 1 / 3, 0, 0]),
    (0, 0.7, [2 / 3, 1 / 3, 0, 0]),            # cum before: 0, .5, .75 -> keep 2
    (0, 0.8, [4 / 7, 2 / 7, 1 / 7, 0]),        # .75 < .8 keeps the crossing token
    (0, 0.45, [1, 0, 0, 0]),                   # first token always kept
    (3, 0.6, [2 / 3, 1 / 3, 0, 0]),            # top-p on the top-3-renormalised dist
    (2, 0.6, [1, 0, 0, 0]),                    # renormalised top-2 is (2/3, 1/3): 2/3 >= .6
    (1, 1.0, [1, 0, 0, 0]),                    # top-k = 1 is one-hot at the argmax
    (4, 1.0, [0.5, 0.25, 0.125, 0.125]),       # top-k >= V is off
    (0, 1.0, [0.5, 0.25, 0.125, 0.125]),
])
def test_filter_hand_examples(top_k, top_p, expected):
    p, _ = oracle.row_probs(DYADIC, 1.0, top_k, top_p)
    np.testing.assert_allclose(p, expected, rtol=1e-14, atol=1e-15)


def test_filter_applies_temperature_first():
    # T = 2: p proportional to sqrt(.5, .25, .125, .125) = (.7071, .5, .3536, .3536)/1.9142;
    # cumulative before token 2 is .6306 >= .6 -> keep {0, 1}, renormalise.
    p, _ = oracle.row_probs(DYADIC, 2.0, 0, 0.6)
    s = 1 + math.sqrt(0.5)
    np.testing.assert_allclose(p, [1 / s, math.sqrt(0.5) / s, 0, 0], rtol=1e-14, atol=0)


def test_filter_ties_lower_index_wins():
    p, _ = oracle.row_probs(np.array([1.0, 1.0, 1.0, 0.0]), 1.0, 2, 1.0)
    np.testing.assert_allclose(p, [0.5, 0.5, 0, 0], rtol=1e-15)
    p, _ = oracle.row_probs(np.array([0.0, 1.0, 1.0, 1.0]), 1.0, 2, 1.0)
    np.testing.assert_allclose(p, [0, 0.5, 0.5, 0], rtol=1e-15)


def test_neg_inf_logits_have_zero_mass_and_bad_rows_error():
    x = np.array([0.0, -np.inf, np.log(0.5), -np.inf])
    p, _ = oracle.row_probs(x, 1.0)
    np.testing.assert_allclose(p, [2 / 3, 0, 1 / 3, 0], rtol=1e-15)
    with pytest.raises(ValueError):
        oracle.row_probs(np.full(4, -np.inf), 1.0)
    with pytest.raises(ValueError):
        oracle.row_probs(np.array([0.0, np.nan, 1.0]), 1.0)
    with pytest.raises(ValueError):
        oracle.row_probs(np.array([0.0, np.inf, 1.0]), 1.0)


# --------------------------------------------------------------------------
# The rejection rule: hand-derived cases.
# --------------------------------------------------------------------------

def one_request(trows, drows, x, u, T=1.0, top_k=0, top_p=1.0):
    acc, tok, mg = oracle.verify_trials(np.asarray(trows, np.float64),
                                        None if drows is None else np.asarray(drows, np.float64),
                                        T, top_k, top_p, np.asarray(x, np.int32)[None],
                                        np.asarray(u, np.float32)[None])
    return int(acc[0]), tok[0].tolist(), mg[0]


def test_greedy_longest_prefix_then_target_token():
    t = np.full((3, 5), -1.0)
    t[0, 3] = t[1, 1] = t[2, 2] = 2.0        # argmaxes 3, 1, 2
    L, tok, _ = one_request(t, None, [3, 0], [0.5] * 3, T=0.0)
    assert (L, tok) == (1, [3, 1, -1])
    L, tok, _ = one_request(t, None, [3, 1], [0.5] * 3, T=0.0)
    assert (L, tok) == (2, [3, 1, 2])
    L, tok, _ = one_request(t, None, [0, 1], [0.5] * 3, T=0.0)   # full rejection still emits one
    assert (L, tok) == (0, [3, -1, -1])


def test_inverse_cdf_boundary_convention():
    # Bonus from p = (.5, .5): t = u * S; y* = min{y : C_y > t}.
    t = np.log(np.array([[0.5, 0.5]]))
    assert one_request(t, np.zeros((0, 2)), [], [0.5])[1] == [1]      # C_0 = .5 is not > .5
    assert one_request(t, np.zeros((0, 2)), [], [0.49999997])[1] == [0]
    assert one_request(t, np.zeros((0, 2)), [], [0.0])[1] == [0]
    with np.errstate(divide="ignore"):
        t0 = np.log(np.array([[0.0, 0.5, 0.5]]))                      # zero-width token skipped
    assert one_request(t0, np.zeros((0, 3)), [], [0.0])[1] == [1]


def test_accept_is_strict_u_below_ratio():
    t = np.log(np.array([[0.25, 0.75], [0.5, 0.5]]))
    d = np.log(np.array([[0.5, 0.5]]))
    # ratio for token 0 = .25 / .5 = .5 exactly
    assert one_request(t, d, [0], [0.49999997, 0.3])[0] == 1
    assert one_request(t, d, [0], [0.5, 0.3])[0] == 0
    # residual after the reject is max(0, p - q) = (0, .25) -> token 1
    assert one_request(t, d, [0], [0.5, 0.0])[1] == [1, -1]


def test_zero_target_probability_always_rejected():
    t = np.array([[-np.inf, 0.0, 0.0], [0.0, 0.0, 0.0]])
    d = np.zeros((1, 3))
    L, tok, _ = one_request(t, d, [0], [0.0, 0.2])
    assert L == 0 and tok[0] != 0


def test_identical_p_q_always_accepts():
    rng = np.random.default_rng(0)
    t = rng.normal(size=(4, 16))
    d = t[:3].copy()
    for _ in range(20):
        x = rng.integers(0, 16, 3)
        u = rng.random(4).astype(np.float32)
        L, tok, _ = one_request(t, d, x, u)
        assert L == 3 and tok[:3] == list(x)


def test_top_k_one_is_greedy_when_argmaxes_agree_or_not():
    rng = np.random.default_rng(1)
    for _ in range(20):
        t = rng.normal(size=(3, 12))
        d = t[:2] + rng.normal(size=(2, 12))
        gd = d.argmax(1)
        u = rng.random(3).astype(np.float32)
        L, tok, _ = one_request(t, d, gd, u, T=1.0, top_k=1)
        Lg, tokg, _ = one_request(t, None, gd, u, T=0.0)
        assert (L, tok) == (Lg, tokg)


def test_k_zero_samples_bonus_from_first_target_row():
    t = np.log(np.array([[0.25, 0.25, 0.5]]))
    assert one_request(t, np.zeros((0, 3)), [], [0.6])[1] == [2]
    assert one_request(t, np.zeros((0, 3)), [], [0.3])[1] == [1]


def test_batch_layout_and_data_errors():
    rng = np.random.default_rng(2)
    k = np.array([2, 0, 3], np.int32)
    Rt, Rd = int((k + 1).sum()), int(k.sum())
    V = 6
    t = rng.normal(size=(Rt, V)).astype(np.float32)
    d = rng.normal(size=(Rd, V)).astype(np.float32)
    x = rng.integers(0, V, Rd).astype(np.int32)
    u = rng.random(Rt).astype(np.float32)
    T = np.array([1.0, 0.5, 0.0], np.float32)
    out = oracle.verify(t, d, x, k, T, uniforms=u)
    # each request equals the single-request path on its own rows
    t_off = [0, 3, 4]
    for b in range(3):
        r0, d0 = t_off[b], t_off[b] - b
        acc, tok, _ = oracle.verify_trials(t[r0:r0 + k[b] + 1], d[d0:d0 + k[b]] if k[b] else None,
                                           T[b], 0, 1.0, x[d0:d0 + k[b]][None],
                                           u[r0:r0 + k[b] + 1][None])
        assert out["accept_len"][b] == acc[0]
        assert out["tokens"][r0:r0 + k[b] + 1].tolist() == tok[0].tolist()
    # data errors are per request
    x_bad = x.copy()
    x_bad[0] = V
    out = oracle.verify(t, d, x_bad, k, T, uniforms=u)
    assert out["accept_len"][0] == -1 and out["accept_len"][2] >= 0
    t_bad = t.copy()
    t_bad[3, 2] = np.nan
    out = oracle.verify(t_bad, d, x, k, T, uniforms=u)
    assert out["accept_len"][1] == -1 and out["accept_len"][0] >= 0
    out = oracle.verify(t, d, x, np.array([2, 0, 33], np.int32), T, uniforms=u)
    assert out["rc"] != 0 and (out["accept_len"] == -1).all()
    out = oracle.verify(t, d, x, k, np.array([1.0, -1.0, 0.0], np.float32), uniforms=u)
    assert out["accept_len"][1] == -1
    out = oracle.verify(t, d, x, k, T, top_p=np.array([1.0, 0.0, 1.0], np.float32), uniforms=u)
    assert out["accept_len"][1] == -1


# --------------------------------------------------------------------------
# Exact output law by enumeration (V = 4, k = 2): accepted mass plus residual
# mass recovers p at every position.
# --------------------------------------------------------------------------

def exact_law(trows, drows, T=1.0, top_k=0, top_p=1.0, lib=None):
    """Enumerate draft tuples (weight prod q_i(x_i)) and the cells of the
    oracle's piecewise-constant dependence on (u_0, .., u_k); return the exact
    law of (L, tokens) as a dict of probabilities."""
    k = trows.shape[0] - 1
    V = trows.shape[1]
    p = [filtered_probs(r, T, top_k, top_p) for r in trows]
    q = [filtered_probs(r, T, top_k, top_p) for r in drows]
    # breakpoints of the final draw: every candidate final distribution
    finals = [p[k]] + [np.maximum(0, p[i] - q[i]) for i in range(k)] + [p[i] for i in range(k)]
    fb = {0.0, 1.0}
    for r in finals:
        s = r.sum()
        if s > 0:
            fb.update(np.cumsum(r / s).tolist())
    fb = sorted(b for b in fb if 0 <= b <= 1)
    fcells = [(a, b) for a, b in zip(fb[:-1], fb[1:]) if b - a > 1e-12]
    xs, us, ws = [], [], []
    for tup in itertools.product(range(V), repeat=k):
        wq = np.prod([q[i][tup[i]] for i in range(k)]) if k else 1.0
        if wq == 0:
            continue
        acells = []
        for i in range(k):
            r = p[i][tup[i]] / q[i][tup[i]]
            c = min(1.0, r)
            cells = [(0.0, c), (c, 1.0)] if 0 < c < 1 else [(0.0, 1.0)]
            acells.append(cells)
        for combo in itertools.product(*acells, fcells):
            width = np.prod([b - a for a, b in combo])
            xs.append(tup)
            us.append([(a + b) / 2 for a, b in combo])
            ws.append(wq * width)
    acc, tok, _ = oracle.verify_trials(trows, drows if k else None, T, top_k, top_p,
                                       np.array(xs, np.int32).reshape(-1, k),
                                       np.array(us, np.float32), lib=lib)
    law = {}
    for L, t, w in zip(acc, tok, ws):
        key = (int(L), tuple(int(v) for v in t))
        law[key] = law.get(key, 0.0) + w
    return law, p


def check_lossless(law, p):
    k = len(p) - 1
    total = sum(law.values())
    assert abs(total - 1) < 1e-12
    V = p[0].shape[0]
    # first emitted token ~ p_0
    m0 = np.zeros(V)
    for (L, t), w in law.items():
        m0[t[0]] += w
    np.testing.assert_allclose(m0, p[0], atol=1e-12)
    # given the first j drafts were accepted, the next emitted token ~ p_j
    for j in range(1, k + 1):
        mj = np.zeros(V)
        for (L, t), w in law.items():
            if L >= j:
                mj[t[j]] += w
        assert mj.sum() > 0
        np.testing.assert_allclose(mj / mj.sum(), p[j], atol=1e-12)


DY = np.log  # logits of dyadic probabilities


@pytest.mark.parametrize("case", ["dyadic", "random", "neg_inf", "filtered"])
def test_exact_enumeration_output_law_equals_p(case):
    rng = np.random.default_rng(11)
    if case == "dyadic":
        t = DY(np.array([[.5, .25, .125, .125], [.125, .125, .25, .5], [.25, .25, .25, .25]]))
        d = DY(np.array([[.25, .25, .25, .25], [.5, .125, .125, .25]]))
        args = {}
    elif case == "random":
        t = rng.normal(size=(3, 4)) * 1.5
        d = rng.normal(size=(2, 4)) * 1.5
        args = dict(T=0.8)
    elif case == "neg_inf":
        t = DY(np.array([[.5, 0, .25, .25], [.25, .25, .5, 0], [0, .5, 0, .5]]))
        d = DY(np.array([[0, .5, .5, 0], [.25, .25, .25, .25]]))
        args = {}
    else:
        t = rng.normal(size=(3, 4)) * 1.5
        d = t[:2] + 0.4 * rng.normal(size=(2, 4))     # kept sets overlap
        args = dict(T=1.3, top_k=3, top_p=0.8)
    with np.errstate(divide="ignore"):
        law, p = exact_law(np.asarray(t), np.asarray(d), **args)
    check_lossless(law, p)


# Planted mistakes: each mutated copy of the oracle source must fail the
# exact-enumeration check (which shows the check can see that kind of error).
MUTANTS = [
    ("residual sign", "std::max(0.0, p[L][y] - q[L][y])", "std::max(0.0, q[L][y] - p[L][y])"),
    ("final draw reuses u_L", "inverse_cdf(r, (double)u[k], &mcdf)",
     "inverse_cdf(r, (double)u[L], &mcdf)"),
    ("ratio inverted", "const double ratio = pi / qi;", "const double ratio = qi / pi;"),
    ("bonus from the last draft position", "    r = p[k];\n", "    r = p[k - 1];\n"),
    ("residual not renormalised by q", "std::max(0.0, p[L][y] - q[L][y])", "p[L][y]"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_enumeration_catches_planted_oracle_mistake(tmp_path, name, old, new):
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, name
    mutant = tmp_path / "oracle_mutant.cpp"
    mutant.write_text(src.replace(old, new))
    lib = oracle.load_variant(oracle.compile_source(str(mutant), str(tmp_path / "m.so")))
    t = DY(np.array([[.375, .375, .125, .125], [.125, .125, .25, .5], [.25, .25, .25, .25]]))
    d = DY(np.array([[.25, .25, .25, .25], [.5, .125, .125, .25]]))
    law, p = exact_law(t, d, lib=lib)
    with pytest.raises(AssertionError):
        check_lossless(law, p)
    law, p = exact_law(t, d)                       # the real oracle passes the same check
    check_lossless(law, p)


# --------------------------------------------------------------------------
# Closed form E = (1 - a^(k+1)) / (1 - a) on rows with sum min(p, q) = a.
# --------------------------------------------------------------------------

def alpha_rows(alpha, k, V=8):
    """p = a r + (1-a) u_A, q = a r + (1-a) u_B, r uniform on 0..3, A = {4, 5},
    B = {6, 7} disjoint, so min(p, q) = a r and sum min(p, q) = a exactly."""
    r = np.array([.25] * 4 + [0] * 4)
    a = np.array([0] * 4 + [.5, .5, 0, 0])
    b = np.array([0] * 4 + [0, 0, .5, .5])
    p = alpha * r + (1 - alpha) * a
    q = alpha * r + (1 - alpha) * b
    with np.errstate(divide="ignore"):
        return np.log(np.tile(p, (k + 1, 1))), np.log(np.tile(q, (k, 1)))


def exact_expected_tokens(alpha, k):
    t, d = alpha_rows(alpha, k)
    V = t.shape[1]
    q = np.exp(d[0])
    support = [y for y in range(V) if q[y] > 0]
    xs, us, ws = [], [], []
    pv = np.exp(t[0])
    for tup in itertools.product(support, repeat=k):
        wq = np.prod([q[y] for y in tup])
        cells = []
        for y in tup:
            c = min(1.0, pv[y] / q[y])
            cells.append([(0.0, c), (c, 1.0)] if 0 < c < 1 else [(0.0, 1.0)])
        for combo in itertools.product(*cells):
            xs.append(tup)
            us.append([(a + b) / 2 for a, b in combo] + [0.5])
            ws.append(wq * np.prod([b - a for a, b in combo]))
    acc, _, _ = oracle.verify_trials(t, d, 1.0, 0, 1.0, np.array(xs, np.int32),
                                     np.array(us, np.float32))
    ws = np.array(ws)
    assert abs(ws.sum() - 1) < 1e-12
    return float((ws * (acc + 1)).sum()), acc, ws


def load_golden():
    rows = []
    with open(os.path.join(HERE, "golden", "expected_tokens_per_pass.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                a, k, e = line.split()
                rows.append((float(a), int(k), float(e)))
    return rows


@pytest.mark.parametrize("alpha,k,printed", load_golden())
def test_expected_tokens_per_pass_matches_page(alpha, k, printed):
    E, acc, ws = exact_expected_tokens(alpha, k)
    closed = (1 - alpha ** (k + 1)) / (1 - alpha)
    assert abs(E - closed) < 1e-12
    assert round(E, 2) == printed
    # the law of L is the truncated geometric a^j (1 - a), a^k at j = k
    for j in range(k + 1):
        pj = ws[acc == j].sum()
        want = alpha ** j * (1 - alpha) if j < k else alpha ** k
        assert abs(pj - want) < 1e-12
