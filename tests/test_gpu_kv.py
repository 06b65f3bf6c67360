"""KV-cache commit on the GPU against the oracle (oracle/kv.py), bit-exact:
the whole cache, the updated lengths and the error record."""

import numpy as np
import pytest
import torch

import speculative_decoding_verification_13_gb300 as sv
from oracle.kv import kv_commit as oracle_commit

pytestmark = pytest.mark.gpu

DEV = "cuda"


def case(seed, B, layers, E, S, kmax, dtype=torch.bfloat16, spare_pages=8):
    rng = np.random.default_rng(seed)
    k = rng.integers(0, kmax + 1, B).astype(np.int32)
    L = np.array([rng.integers(-1, kk + 1) for kk in k], np.int32)
    if B > 1:
        L[0], L[1] = -1, k[1]
    n = rng.integers(0, 3 * S, B).astype(np.int32)
    max_pages = (3 * S + kmax + 1) // S + 2
    need = (n + k + 1 + S - 1) // S
    n_pages = int(need.sum()) + spare_pages
    perm = rng.permutation(n_pages).astype(np.int32)
    table = np.full((B, max_pages), -1, np.int32)
    used = 0
    for b in range(B):
        table[b, :need[b]] = perm[used:used + need[b]]
        used += need[b]
    g = torch.Generator().manual_seed(seed)
    cache = torch.randn(n_pages, layers, 2, S, E, generator=g).to(dtype)
    spec = torch.randn(B, kmax + 1, layers, 2, E, generator=g).to(dtype)
    return k, L, n, table, cache, spec, S


def run_both(k, L, n, table, cache, spec, S):
    cache_d = cache.to(DEV)
    kv_len = torch.as_tensor(n).to(DEV)
    sv.kv_commit(cache_d, spec.to(DEV), torch.as_tensor(L).to(DEV), torch.as_tensor(k).to(DEV),
                 kv_len, torch.as_tensor(table).to(DEV))
    code = sv.kv_commit_error()[0]
    c_ref = cache.view(torch.int16 if cache.element_size() == 2 else torch.int32).numpy().copy()
    s_ref = spec.view(torch.int16 if spec.element_size() == 2 else torch.int32).numpy()
    new_len, st = oracle_commit(s_ref, L, k, n, table, c_ref, S)
    got = cache_d.cpu().view(torch.int16 if cache.element_size() == 2 else torch.int32).numpy()
    assert np.array_equal(got, c_ref), "cache differs from the oracle"
    assert np.array_equal(kv_len.cpu().numpy(), new_len), "kv_len differs"
    return code, st


@pytest.mark.parametrize("B,layers,E,S,kmax,dtype", [
    (40, 4, 1024, 16, 15, torch.bfloat16),   # Qwen3-8B-class rows (8 heads x 128)
    (64, 3, 64, 1, 8, torch.float16),        # one token per page
    (17, 2, 8, 64, 32, torch.float32),       # long pages, the largest k
    (1, 1, 8, 4, 0, torch.bfloat16),         # k = 0: only the last emitted token
])
def test_commit_matches_oracle(B, layers, E, S, kmax, dtype):
    code, st = run_both(*case(B * 7 + S, B, layers, E, S, kmax, dtype))
    assert code == 0 and (st == 0).all()


def test_errors_write_nothing_and_are_reported():
    k, L, n, table, cache, spec, S = case(99, 12, 2, 64, 4, 6)
    L = L.copy()
    table = table.copy()
    L[3] = k[3] + 1                                # accept length above k
    L[5] = k[5]
    table[5, (n[5] + L[5]) // S] = -1              # a destination page missing
    L[7] = k[7]
    table[7, (n[7] + L[7]) // S] = cache.shape[0]  # a page id past the pool
    code, st = run_both(k, L, n, table, cache, spec, S)
    assert st[3] == 26 and st[5] == 27 and st[7] == 27
    assert code in (26, 27)


def test_empty_batch():
    cache = torch.zeros(4, 1, 2, 4, 8, dtype=torch.bfloat16, device=DEV)
    spec = torch.zeros(0, 1, 1, 2, 8, dtype=torch.bfloat16, device=DEV)
    e = torch.zeros(0, dtype=torch.int32, device=DEV)
    sv.kv_commit(cache, spec, e, e, e.clone(), torch.zeros(0, 2, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    assert (cache == 0).all()


@pytest.mark.parametrize("B", [1025, 4097])
def test_batches_past_one_validation_round(B):
    # the validation CTA takes 1024 requests a round: its scan carries the
    # token offsets from round to round
    code, st = run_both(*case(B, B, 1, 8, 4, 15))
    assert code == 0 and (st == 0).all()


def test_calls_of_several_sizes_reuse_one_workspace():
    # a workspace sized for the largest batch first, then smaller batches on
    # the same workspace: nothing of an earlier call leaks into a later one
    for i, (B, layers, E, S, kmax) in enumerate([(300, 2, 64, 16, 15), (40, 4, 1024, 16, 15),
                                                 (7, 1, 8, 4, 3), (1, 1, 8, 4, 0),
                                                 (300, 3, 16, 8, 32)]):
        code, st = run_both(*case(1000 + i, B, layers, E, S, kmax))
        assert code == 0 and (st == 0).all(), (B, code)
