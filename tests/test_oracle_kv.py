"""Pins of the KV-cache commit oracle (oracle/kv.py).  The commit has a plain
definition; it is pinned by a hand-worked example and by properties computed
another way: each request's logical sequence, gathered from the paged cache
through its block table with torch indexing, must equal its old prefix
followed by the accepted entries; nothing else in the cache changes; rejected
entries are written nowhere; errors write nothing."""

import numpy as np
import pytest
import torch

from oracle.kv import KV_ERR_ACCEPT, KV_ERR_PAGE, kv_commit


def logical(cache, table_row, length, S):
    """Request's entries at positions 0..length-1, gathered by torch indexing."""
    pos = torch.arange(length)
    pages = torch.as_tensor(table_row)[pos // S]
    return torch.as_tensor(cache)[pages, :, :, pos % S, :]  # [length, layers, 2, E]


def make_case(seed, B=6, layers=3, E=5, S=4, kmax=7, n_pages=64):
    rng = np.random.default_rng(seed)
    k = rng.integers(0, kmax + 1, B)
    L = np.array([rng.integers(-1, kk + 1) for kk in k])
    L[0] = -1
    L[1] = k[1]                       # every draft accepted
    n = rng.integers(0, 30, B)
    max_pages = (30 + kmax + S) // S + 1
    perm = rng.permutation(n_pages)
    table = np.full((B, max_pages), -1, np.int32)
    used = 0
    for b in range(B):
        need = (n[b] + k[b] + 1 + S - 1) // S
        table[b, :need] = perm[used:used + need]
        used += need
    cache = rng.normal(size=(n_pages, layers, 2, S, E)).astype(np.float32)
    spec = rng.normal(size=(B, kmax + 1, layers, 2, E)).astype(np.float32) + 100.0  # distinct
    return k, L, n, table, cache, spec, S


@pytest.mark.parametrize("seed", range(5))
def test_logical_view_is_prefix_then_accepted_entries(seed):
    k, L, n, table, cache, spec, S = make_case(seed)
    before = cache.copy()
    new_len, st = kv_commit(spec, L, k, n, table, cache, S)
    assert (st == 0).all()
    for b in range(len(k)):
        if L[b] < 0:
            assert new_len[b] == n[b]
            continue
        assert new_len[b] == n[b] + L[b] + 1
        want = torch.cat([logical(before, table[b], n[b], S),
                          torch.as_tensor(spec[b, :L[b] + 1])])
        assert torch.equal(logical(cache, table[b], new_len[b], S), want)


@pytest.mark.parametrize("seed", range(3))
def test_only_the_committed_slots_change_and_rejected_entries_appear_nowhere(seed):
    k, L, n, table, cache, spec, S = make_case(seed + 10)
    before = cache.copy()
    kv_commit(spec, L, k, n, table, cache, S)
    written = np.zeros(cache.shape[0] * S, bool)
    for b in range(len(k)):
        for p in range(n[b], n[b] + L[b] + 1):
            written[table[b, p // S] * S + p % S] = True
    per_slot = np.moveaxis(cache, 3, 1).reshape(cache.shape[0] * S, -1)
    per_slot0 = np.moveaxis(before, 3, 1).reshape(before.shape[0] * S, -1)
    assert (per_slot[~written] == per_slot0[~written]).all()
    for b in range(len(k)):
        for j in range(max(L[b], -1) + 1, k[b] + 1):   # rejected drafts
            e = spec[b, j].reshape(-1)                # one slot's [layers, 2, E]
            assert not (per_slot == e).all(axis=1).any()


def test_hand_example_across_a_page_boundary():
    S, layers, E = 2, 1, 1
    cache = np.zeros((8, layers, 2, S, E), np.float32)
    spec = np.arange(1 * 4 * layers * 2 * E, dtype=np.float32).reshape(1, 4, layers, 2, E) + 1
    table = np.array([[7, 2, 5, -1]], np.int32)
    new_len, st = kv_commit(spec, [2], [3], [3], table, cache, S)
    assert st.tolist() == [0] and new_len.tolist() == [6]
    # positions 3, 4, 5 -> (page 2, slot 1), (page 5, slot 0), (page 5, slot 1)
    assert cache[2, 0, :, 1, 0].tolist() == [1.0, 2.0]
    assert cache[5, 0, :, 0, 0].tolist() == [3.0, 4.0]
    assert cache[5, 0, :, 1, 0].tolist() == [5.0, 6.0]
    assert np.count_nonzero(cache) == 6       # the draft at j = 3 was rejected


def test_errors_write_nothing():
    k, L, n, table, cache, spec, S = make_case(42)
    b_acc, b_page = 2, 3
    L = L.copy()
    L[b_acc] = k[b_acc] + 1                      # accept length above k
    L[b_page] = k[b_page]
    table = table.copy()
    last = (n[b_page] + L[b_page]) // S
    table[b_page, last] = -1                     # its last destination page is missing
    before = cache.copy()
    new_len, st = kv_commit(spec, L, k, n, table, cache, S)
    assert st[b_acc] == KV_ERR_ACCEPT and st[b_page] == KV_ERR_PAGE
    assert new_len[b_acc] == n[b_acc] and new_len[b_page] == n[b_page]
    # the failed requests' own pages are untouched
    for b in (b_acc, b_page):
        rows = table[b][table[b] >= 0]
        assert (cache[rows] == before[rows]).all()


KV_MUTANTS = [
    ("accepted drafts only (the last emitted token's entry dropped)",
     "        for j in range(L + 1):\n            p = n + j",
     "        for j in range(L):\n            p = n + j"),
    ("rejected draft kept", "        for j in range(L + 1):\n            p = n + j",
     "        for j in range(L + 2):\n            p = n + j"),
    ("slot off by one", "dest.append((page, p % page_size))",
     "dest.append((page, (p + 1) % page_size))"),
]


@pytest.mark.parametrize("name,old,new", KV_MUTANTS, ids=[m[0] for m in KV_MUTANTS])
def test_logical_view_catches_planted_mistake(name, old, new):
    import oracle.kv as kvmod
    src = open(kvmod.__file__).read()
    assert src.count(old) == 1, name
    ns = {}
    exec(compile(src.replace(old, new), "kv_mutant", "exec"), ns)
    k, L, n, table, cache, spec, S = make_case(7)
    L = np.minimum(L, k - 1)          # leave room for a kept rejected draft
    before = cache.copy()
    try:
        new_len, st = ns["kv_commit"](spec, L, k, n, table, cache, S)
    except IndexError:
        return                         # the mutant ran past the block table: caught
    ok = True
    for b in range(len(k)):
        if L[b] < 0:
            continue
        want = torch.cat([logical(before, table[b], n[b], S), torch.as_tensor(spec[b, :L[b] + 1])])
        got = logical(cache, table[b], n[b] + L[b] + 1, S)
        ok &= bool(torch.equal(got, want)) and new_len[b] == n[b] + L[b] + 1
        if L[b] + 1 < k[b] + 1:       # the next slot must not hold the rejected draft
            p = n[b] + L[b] + 1
            ok &= not np.array_equal(cache[table[b, p // S], :, :, p % S], spec[b, L[b] + 1])
    assert not ok, name
