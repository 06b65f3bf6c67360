"""LM-head GEMM with fused verification statistics (tcgen05) against the
oracle (float64 product of the same bf16 inputs).  Tolerances follow from f32
accumulation: a logit may differ by a few f32 rounding steps of the row's
|h| . |w| magnitude; the argmax must match unless the oracle's top two logits
are closer than that."""

import numpy as np
import pytest
import torch

import speculative_decoding_verification_13_gb300 as sv
from oracle.lmhead import lmhead_stats as oracle_stats

pytestmark = pytest.mark.gpu

DEV = "cuda"


def run(M, V, d, seed, scale=1.0, greedy_frac=0.25, tokens=True):
    g = torch.Generator().manual_seed(seed)
    H = (torch.randn(M, d, generator=g) * scale).to(torch.bfloat16)
    W = (torch.randn(V, d, generator=g) / np.sqrt(d) * 4).to(torch.bfloat16)
    T = torch.rand(M, generator=g) * 1.5 + 0.3
    T[torch.rand(M, generator=g) < greedy_frac] = 0.0
    tok = torch.randint(0, V, (M,), generator=g, dtype=torch.int32) if tokens else None
    m, s, a, x = sv.lmhead_stats(H.to(DEV), W.to(DEV), T.to(DEV),
                                 tok.to(DEV) if tok is not None else None)
    torch.cuda.synchronize()
    assert sv.lmhead_stats_error()[0] == 0
    o = oracle_stats(H, W, T.numpy(), tok.numpy() if tok is not None else np.full(M, -1))
    bound = (np.abs(H.double().numpy()) @ np.abs(W.double().numpy()).T).max(axis=1)
    tol = 4 * 2.0 ** -23 * bound + 1e-6
    m, s, a, x = (t.cpu().numpy() for t in (m, s, a, x))
    assert (np.abs(m - o["m"]) <= tol).all(), np.abs(m - o["m"]).max()
    Ts = np.where(T.numpy() > 0, T.numpy(), 1.0)
    # the sum's relative error follows the logits' absolute error over T
    assert (np.abs(s / o["s"] - 1) <= 2 * tol / Ts + 1e-5).all(), np.abs(s / o["s"] - 1).max()
    z = o["z"]
    top2 = np.sort(z, axis=1)[:, -2:] if z.shape[1] > 1 else np.concatenate([z, z], 1)
    close = (top2[:, 1] - top2[:, 0]) < 2 * tol
    bad = (a != o["arg"]) & ~close
    assert not bad.any(), f"argmax mismatch rows {np.nonzero(bad)[0][:10]}"
    if tokens:
        assert (np.abs(x - o["xt"]) <= tol).all()
    else:
        assert np.isnan(x).all()
    return int(close.sum())


@pytest.mark.parametrize("M,V,d", [
    (128, 256, 64),        # one tile, one K block
    (200, 1000, 256),      # ragged row and column tiles
    (130, 3000, 520),      # K not a multiple of the 64-wide K block
    (256, 151936, 1024),   # the Qwen3 vocabulary, many column chunks (8 W tiles a unit)
    (512, 151936, 128),    # 16 W tiles a work unit on a 152-SM GPU
    (1024, 151936, 128),   # 32 W tiles a work unit on a 152-SM GPU
])
def test_matches_oracle(M, V, d):
    run(M, V, d, seed=M + V + d)


def test_greedy_rows_and_no_tokens():
    run(300, 5000, 128, seed=5, greedy_frac=1.0, tokens=False)


def test_large_logits():
    run(128, 2048, 512, seed=6, scale=8.0)
