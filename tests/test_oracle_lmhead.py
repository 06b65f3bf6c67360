"""Pins of the LM-head statistics oracle (oracle/lmhead.py) against library
routines on the same logits and a hand-worked example."""

import numpy as np
import pytest
import torch

from oracle.lmhead import lmhead_stats


def test_hand_example():
    H = np.array([[1.0, 2.0], [0.5, -1.0]])
    W = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0], [-1.0, 0.5]])
    # z row 0 = [1, 2, 3, 0], row 1 = [0.5, -1, -0.5, -1]
    r = lmhead_stats(H, W, [1.0, 0.5], [1, 3])
    assert r["m"].tolist() == [3.0, 0.5]
    assert r["arg"].tolist() == [2, 0]
    assert r["xt"].tolist() == [2.0, -1.0]
    s0 = np.exp(-2) + np.exp(-1) + 1 + np.exp(-3)
    s1 = 1 + np.exp(-3) + np.exp(-2) + np.exp(-3)
    np.testing.assert_allclose(r["s"], [s0, s1], rtol=1e-15)


@pytest.mark.parametrize("T", [1.0, 0.6, 1.7])
def test_stats_equal_torch_logsumexp_and_softmax(T):
    g = torch.Generator().manual_seed(3)
    H = torch.randn(20, 64, generator=g).to(torch.bfloat16)
    W = torch.randn(300, 64, generator=g).to(torch.bfloat16)
    tok = torch.randint(0, 300, (20,), generator=g)
    r = lmhead_stats(H, W, [T] * 20, tok.numpy())
    z = H.double() @ W.double().T
    lse = torch.logsumexp(z / T, dim=1).numpy()
    np.testing.assert_allclose(r["m"] / T + np.log(r["s"]), lse, rtol=1e-13)
    p = torch.softmax(z / T, dim=1)[torch.arange(20), tok].numpy()
    np.testing.assert_allclose(np.exp((r["xt"] - r["m"]) / T) / r["s"], p, rtol=1e-12)
    assert (r["arg"] == torch.argmax(z, dim=1).numpy()).all()


def test_ties_first_index_and_greedy_rows():
    H = np.ones((2, 4))
    W = np.array([[1, 0, 0, 0], [0.5, 0.5, 0, 0], [0, 0, 0, 1], [0, 0, 0.25, 0.75]], float)
    r = lmhead_stats(H, W, [0.0, 0.0], [-1, 2])
    assert r["arg"].tolist() == [0, 0]          # four equal logits: the first index
    assert np.isnan(r["xt"][0]) and r["xt"][1] == 1.0
    np.testing.assert_allclose(r["s"], [4.0, 4.0])   # temperature 0 sums at T = 1
