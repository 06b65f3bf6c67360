"""Adaptive k on the GPU against the oracle, bit for bit (counts, alpha, k),
over several passes of accept lengths from the verification rule."""

import numpy as np
import pytest
import torch

import speculative_decoding_verification_13_gb300 as sv
from oracle.adapt import adapt_k as oracle_adapt

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("decay,c,k_min,k_max", [(0.9, 0.1, 1, 16), (1.0, 0.05, 2, 32),
                                                 (0.5, 0.3, 0, 8)])
def test_matches_oracle_over_passes(decay, c, k_min, k_max):
    rng = np.random.default_rng(int(decay * 10) + k_max)
    B = 1000
    alpha_true = rng.uniform(0.05, 0.98, B)
    k = np.full(B, max(k_min, 4), np.int32)
    s_o, f_o = np.zeros(B), np.zeros(B)
    succ = torch.zeros(B, dtype=torch.float64, device="cuda")
    fail = torch.zeros(B, dtype=torch.float64, device="cuda")
    for _ in range(12):
        acc = rng.random((B, 33)) < alpha_true[:, None]
        L = np.array([int(np.argmin(acc[b, :k[b]])) if k[b] and not acc[b, :k[b]].all() else k[b]
                      for b in range(B)], np.int32)
        L[rng.random(B) < 0.02] = -1                       # failed verifications
        kn_o, s_o, f_o, a_o = oracle_adapt(L, k, s_o, f_o, decay, c, k_min, k_max)
        kn, al = sv.adapt_k(torch.as_tensor(L, device="cuda"), torch.as_tensor(k, device="cuda"),
                            succ, fail, decay, c, k_min, k_max, with_alpha=True)
        assert np.array_equal(kn.cpu().numpy(), kn_o)
        assert np.array_equal(succ.cpu().numpy(), s_o) and np.array_equal(fail.cpu().numpy(), f_o)
        assert np.array_equal(al.cpu().numpy(), a_o.astype(np.float32))
        k = kn_o


def test_rejects_bad_arguments():
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = torch.zeros(1, dtype=torch.float64, device="cuda")
    with pytest.raises(sv.SpecVerifyError):
        sv.adapt_k(e, e, d, d.clone(), k_min=5, k_max=3)
