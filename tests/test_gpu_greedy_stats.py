"""Greedy verification from the LM head's argmax: the tcgen05 LM-head GEMM
(spec_lmhead_stats) gives each target row's argmax in its epilogue and
spec_verify_greedy_from_argmax verifies from those alone, so the logits never
exist.  Checked bit for bit against the oracle's greedy verification of the
float64 logits formed from the same hidden states and unembedding, except
for requests whose examined rows have a near tie at the top (two logits
within the f32-accumulation tolerance of the LM-head test), which are
counted; plus the data-error contract."""

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_13_gb300 as sv
from oracle.lmhead import lmhead_stats as oracle_stats

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_verification_13_gb300 import build
    build.build()
    oracle.build()
    torch.cuda.init()


def _offsets(k):
    return np.concatenate([[0], np.cumsum(np.asarray(k) + 1)])


def _drafts_near(arg, k, rng, V):
    """Drafts that follow the given argmax for a random prefix, then deviate."""
    t_off = _offsets(k)
    x = []
    for b, kb in enumerate(k):
        stop = rng.integers(0, kb + 1)
        for i in range(kb):
            a = int(arg[t_off[b] + i])
            x.append(a if i < stop else int((a + 1 + rng.integers(0, V - 1)) % V))
    return np.asarray(x, np.int32)


@pytest.mark.parametrize("B,V,d", [(40, 32000, 512), (12, 151936, 1024)])
def test_lmhead_then_greedy_verify_matches_oracle(B, V, d):
    rng = np.random.default_rng(B + V)
    k = rng.integers(0, 9, B)
    k[0], k[-1] = 0, 8
    Rt = int((k + 1).sum())
    g = torch.Generator().manual_seed(V + d)
    H = torch.randn(Rt, d, generator=g).to(torch.bfloat16)
    W = (torch.randn(V, d, generator=g) / np.sqrt(d) * 4).to(torch.bfloat16)
    o = oracle_stats(H, W, np.zeros(Rt), np.full(Rt, -1))
    z = o["z"]
    x = _drafts_near(o["arg"], k, rng, V)
    _, _, arg, _ = sv.lmhead_stats(H.to(DEV), W.to(DEV), torch.zeros(Rt, device=DEV))
    acc, tok = sv.verify_greedy_from_argmax(arg, torch.from_numpy(x).to(DEV),
                                            torch.from_numpy(k.astype(np.int32)).to(DEV), V)
    assert sv.verify_greedy_error()[0] == 0
    acc, tok = acc.cpu().numpy(), tok.cpu().numpy()
    # the oracle's greedy verification of the float64 logits (draft logits
    # are never read at temperature 0)
    ov = oracle.verify(z, None, x, k.astype(np.int32), np.zeros(B, np.float32),
                       None, None, np.zeros(Rt, np.float32), threads=16)
    bound = (np.abs(H.double().numpy()) @ np.abs(W.double().numpy()).T).max(axis=1)
    tol = 4 * 2.0 ** -23 * bound + 1e-6
    top2 = np.sort(z, axis=1)[:, -2:]
    near_tie = (top2[:, 1] - top2[:, 0]) < 2 * tol
    t_off = _offsets(k)
    exempt = 0
    for b in range(B):
        rows = slice(t_off[b], t_off[b] + min(int(ov["accept_len"][b]), int(k[b])) + 1)
        if near_tie[rows].any():
            exempt += 1
            continue
        assert acc[b] == ov["accept_len"][b], b
        assert (tok[t_off[b]:t_off[b + 1]] == ov["tokens"][t_off[b]:t_off[b + 1]]).all(), b
    assert exempt <= B // 10, exempt
    assert len(set(acc.tolist())) > 3  # accept lengths actually vary


def test_greedy_from_argmax_edges_and_errors():
    V = 1000
    k = np.array([0, 32, 3, 5], np.int32)
    Rt = int((k + 1).sum())
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((Rt, V)).astype(np.float32)
    arg = np.argmax(logits, axis=1).astype(np.int32)
    x = _drafts_near(arg, k, rng, V)
    args = [torch.from_numpy(a).to(DEV) for a in (arg, x, k)]
    acc, tok = sv.verify_greedy_from_argmax(*args, V)
    ov = oracle.verify(logits, None, x, k,
                       np.zeros(len(k), np.float32), None, None, np.zeros(Rt, np.float32))
    assert (acc.cpu().numpy() == ov["accept_len"]).all()
    assert (tok.cpu().numpy() == ov["tokens"]).all()
    # a draft token outside [0, V) fails its request only
    x_bad = x.copy()
    x_bad[int(k[0])] = V + 5  # first draft of request 1
    acc, tok = sv.verify_greedy_from_argmax(args[0], torch.from_numpy(x_bad).to(DEV), args[2], V)
    code, req, _ = sv.verify_greedy_error()
    assert code == 20 and req == 1
    a = acc.cpu().numpy()
    assert a[1] == -1 and (a[[0, 2, 3]] == ov["accept_len"][[0, 2, 3]]).all()
    # row counts that do not match k fail the whole batch
    k_bad = k.copy()
    k_bad[2] = 4
    acc, tok = sv.verify_greedy_from_argmax(args[0], args[1], torch.from_numpy(k_bad).to(DEV), V)
    assert sv.verify_greedy_error()[0] == 21
    assert (acc.cpu().numpy() == -1).all() and (tok.cpu().numpy() == -1).all()
