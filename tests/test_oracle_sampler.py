"""Pins of the oracle's draft-side sampler ("FlashMap: Flow Map Speculative
Decoding…", §5 draft_block step 5: logits / temperature, softmax, a
multinomial draw; argmax at temperature 0), against facts that do not come
from the oracle itself:

* the exact output law over a grid of uniforms on rows whose probabilities are
  dyadic (so every breakpoint of the inverse CDF falls between grid points);
* the same law for a filtered row against the sort-based restatement in
  helpers.py, within the grid's resolution;
* torch.argmax (first index on ties) for temperature 0;
* a chi-square test against numpy's softmax;
* boundary uniforms, batch layout, data errors, and agreement with the
  verifier's bonus draw on the same row and uniform;
* planted mistakes in copies of the oracle that the law check must catch.
"""

import numpy as np
import pytest
import torch

import oracle
from helpers import chi2_pvalue, filtered_probs, softmax64

GRID = 1 << 16


def grid_uniforms():
    # midpoints (j + 1/2) / 2^16: exact in float32, never on a dyadic breakpoint
    return ((np.arange(GRID, dtype=np.float64) + 0.5) / GRID).astype(np.float32)


def grid_law(row, T=1.0, top_k=0, top_p=1.0, lib_call=None):
    """Tokens drawn from one row for every grid uniform (the row repeated, one
    request of k = GRID rows would exceed the k limit, so GRID requests of k = 1)."""
    row = np.asarray(row, np.float64)
    V = row.shape[0]
    rows = np.broadcast_to(row, (GRID, V)).copy()
    k = np.ones(GRID, np.int32)
    u = grid_uniforms()
    call = lib_call or oracle.draft_sample
    r = call(rows, k, np.full(GRID, T, np.float32), u,
             top_k=np.full(GRID, top_k, np.int32), top_p=np.full(GRID, top_p, np.float32),
             threads=8)
    assert r["rc"] == 0
    return r["tokens"], r["q"], u


DYADIC = [
    np.array([1 / 8, 1 / 4, 0.0, 1 / 2, 1 / 8]),
    np.array([1 / 2, 1 / 2]),
    np.array([1.0]),
    np.array([0.0, 0.0, 3 / 4, 1 / 16, 1 / 16, 1 / 8]),
    np.array([1 / 1024] * 512 + [1 / 2048] * 1024),
]


@pytest.mark.parametrize("p", DYADIC, ids=[f"V{len(p)}" for p in DYADIC])
def test_exact_law_on_dyadic_rows(p):
    """P(x = y) = p(y) exactly: the count of grid uniforms that draw y is
    p(y) * 2^16, and the token is non-decreasing in u (index order)."""
    with np.errstate(divide="ignore"):
        logits = np.log(p)  # zero probability -> -inf logit
    tok, q, _ = grid_law(logits)
    assert (np.diff(tok) >= 0).all()
    counts = np.bincount(tok, minlength=len(p))
    assert (counts == np.round(p * GRID).astype(np.int64)).all()
    np.testing.assert_allclose(q, p[tok], rtol=1e-12)


def test_filtered_law_matches_sort_based_restatement():
    rng = np.random.default_rng(3)
    x = rng.normal(0, 1.5, 40)
    x[7] = x[3]  # a tie across the top-k boundary region
    T, top_k, top_p = 0.7, 12, 0.8
    tok, q, _ = grid_law(x, T, top_k, top_p)
    ref = filtered_probs(x, T, top_k, top_p)
    law = np.bincount(tok, minlength=len(x)) / GRID
    # each breakpoint moves a count by at most one grid cell
    assert np.abs(law - ref).max() <= 1.0 / GRID + 1e-12
    assert set(np.nonzero(law)[0]) <= set(np.nonzero(ref)[0])
    np.testing.assert_allclose(q, ref[tok], rtol=1e-12)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_greedy_is_torch_argmax_first_index(dtype):
    g = torch.Generator().manual_seed(5)
    x = torch.randn(64, 300, generator=g).to(dtype)
    x[::3, 17] = x[::3].max(dim=1).values  # ties with an earlier or later maximum
    x[::5, 250] = x[::5].max(dim=1).values
    k = torch.full((32,), 2, dtype=torch.int32)
    u = torch.rand(64, generator=g)
    r = oracle.draft_sample(x, k, torch.zeros(32), u)
    assert r["rc"] == 0
    assert (r["tokens"] == torch.argmax(x.float(), dim=1).numpy()).all()
    assert np.isnan(r["q"]).all()


def test_chi_square_against_softmax():
    rng = np.random.default_rng(11)
    V, n, T = 64, 40000, 0.8
    x = rng.normal(0, 1, V).astype(np.float32)
    rows = np.broadcast_to(x, (n, V)).copy()
    u = rng.random(n, dtype=np.float32)
    r = oracle.draft_sample(rows, np.ones(n, np.int32), np.full(n, T, np.float32), u, threads=8)
    p = softmax64(x, T)
    assert chi2_pvalue(np.bincount(r["tokens"], minlength=V), p) > 1e-3


def test_top_k_one_draws_the_argmax_for_every_uniform():
    rng = np.random.default_rng(2)
    x = rng.normal(0, 1, 50)
    tok, q, _ = grid_law(x, 1.3, top_k=1)
    assert (tok == int(np.argmax(x))).all()
    assert (q == 1.0).all()


def test_boundary_uniforms_pick_first_and_last_tokens_with_mass():
    p = np.array([0.0, 0.25, 0.0, 0.5, 0.25, 0.0])
    with np.errstate(divide="ignore"):
        x = np.log(p)
    u = np.array([0.0, np.nextafter(np.float32(1), np.float32(0))], np.float32)
    r = oracle.draft_sample(np.stack([x, x]), [2], [1.0], u)
    assert r["tokens"].tolist() == [1, 4]


def test_layout_and_data_errors():
    rng = np.random.default_rng(4)
    V = 20
    k = np.array([2, 0, 3, 1, 2], np.int32)
    x = rng.normal(0, 1, (int(k.sum()), V)).astype(np.float32)
    x[3, 5] = np.nan                          # request 2 (rows 2..4): a NaN logit
    T = np.array([1.0, 1.0, 1.0, -1.0, 0.5], np.float32)  # request 3: bad temperature
    u = rng.random(int(k.sum()), dtype=np.float32)
    r = oracle.draft_sample(x, k, T, u)
    assert r["rc"] == 0
    assert (r["tokens"][2:5] == -1).all() and r["tokens"][5] == -1
    assert np.isnan(r["q"][2:6]).all()
    for row in (0, 1, 6, 7):
        b_T = 1.0 if row < 2 else 0.5
        ref = softmax64(x[row], b_T)
        c = np.cumsum(ref)
        assert r["tokens"][row] == int(np.searchsorted(c, np.float64(u[row]) * c[-1], "right"))
    # row count that does not match sum(k): every token -1
    r2 = oracle.draft_sample(x[:-1], k, np.ones(5, np.float32), u[:-1])
    assert r2["rc"] == 21 and (r2["tokens"] == -1).all()


def test_agrees_with_the_verifiers_bonus_draw():
    """A k = 0 request of the verifier draws its bonus token from p_0 with
    u_0; the sampler's draw on the same row with the same uniform is the same
    token (two entry points, one definition of the draw)."""
    rng = np.random.default_rng(9)
    V, n = 30, 200
    x = rng.normal(0, 2, (n, V)).astype(np.float32)
    u = rng.random(n, dtype=np.float32)
    for top_k, top_p in [(0, 1.0), (7, 0.85)]:
        s = oracle.draft_sample(x, np.ones(n, np.int32), np.full(n, 0.9, np.float32), u,
                                top_k=np.full(n, top_k, np.int32),
                                top_p=np.full(n, top_p, np.float32))
        v = oracle.verify(x, None, None, np.zeros(n, np.int32), np.full(n, 0.9, np.float32),
                          top_k=np.full(n, top_k, np.int32), top_p=np.full(n, top_p, np.float32),
                          uniforms=u)
        assert (s["tokens"] == v["tokens"]).all()


MUTANTS = [
    ("draws with 1 - u", "tok[i] = inverse_cdf(p, (double)uniforms[d0 + i], &mc[i]);",
     "tok[i] = inverse_cdf(p, 1.0 - (double)uniforms[d0 + i], &mc[i]);"),
    ("argmax instead of a draw", "tok[i] = inverse_cdf(p, (double)uniforms[d0 + i], &mc[i]);",
     "tok[i] = argmax_first(x); (void)mc;"),
    ("neighbouring row's uniform", "tok[i] = inverse_cdf(p, (double)uniforms[d0 + i], &mc[i]);",
     "tok[i] = inverse_cdf(p, (double)uniforms[d0 + (i + 1) % k], &mc[i]);"),
]


def run_lib(lib, rows, k, u):
    n = rows.shape[0]
    tok = np.empty(n, np.int32)
    q = np.empty(n)
    mg = np.empty((n, 2))
    rc = lib.oracle_draft_sample(len(k), rows.shape[1], oracle.DT_F64, oracle._ptr(rows), n,
                                 rows.shape[1], oracle._ptr(k),
                                 oracle._ptr(np.ones(len(k), np.float32)), None, None,
                                 oracle._ptr(u), oracle._ptr(tok), oracle._ptr(q), oracle._ptr(mg))
    assert rc == 0
    return tok


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_law_check_catches_planted_sampler_mistake(tmp_path, name, old, new):
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, name
    mutant = tmp_path / "oracle_mutant.cpp"
    mutant.write_text(src.replace(old, new))
    lib = oracle.load_variant(oracle.compile_source(str(mutant), str(tmp_path / "m.so")))
    p = np.array([1 / 8, 1 / 4, 0.0, 1 / 2, 1 / 8])
    with np.errstate(divide="ignore"):
        x = np.log(p)
    # two rows per request, the two uniforms of a request far apart
    rows = np.broadcast_to(x, (GRID, len(p))).copy()
    k = np.full(GRID // 2, 2, np.int32)
    u = grid_uniforms()
    u = np.stack([u[: GRID // 2], u[GRID // 2:]], axis=1).reshape(-1).copy()
    expect = np.searchsorted(np.cumsum(p), u.astype(np.float64), "right")
    # the check: every row's token is the inverse CDF of its own uniform
    assert (run_lib(oracle._lib(), rows, k, u) == expect).all()   # the real oracle passes
    assert not (run_lib(lib, rows, k, u) == expect).all(), name    # the mutant fails
