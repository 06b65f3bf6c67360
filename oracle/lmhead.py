"""Oracle of the LM-head GEMM with a fused verification-statistics epilogue.

TEST INFRASTRUCTURE ONLY: the plain definition in numpy (float64).  Only
tests/, __graft_entry__.smoke() and bench.py's CPU baseline may use it.

The target's logits are the last hidden states times the unembedding matrix,
z = h W^T ("FlashMap: Flow Map Speculative Decoding…", section 1: the target
yields a distribution over the vocabulary from its final hidden state), and
verification needs of each logit row only its softmax statistics at the
row's temperature, its argmax and the logit of the row's token
("FlashMap…" §5 draft_block step 5: logits / T, softmax, argmax at T = 0;
§4: p(x) of the drafted token).  Computing them in the GEMM's epilogue means
the logits never reach memory.  Per row r with temperature T_r (1 when
T_r = 0) and token x_r (-1 for none):

  m_r   = max_y z[r, y]
  s_r   = sum_y exp((z[r, y] - m_r) / T_r)
  arg_r = min{ y : z[r, y] = m_r }
  xt_r  = z[r, x_r]  (NaN when x_r < 0)

so that p_r(x_r) = exp((xt_r - m_r) / T_r) / s_r.  A matmul serves as the first
step (the float64 product of bfloat16-exact inputs).
"""

from __future__ import annotations

import numpy as np


def as_f64(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, np.float64)


def lmhead_stats(H, W, temperature, tokens):
    """Returns dict m [M], s [M], arg [M] int32, xt [M], z [M, V] (the logits)."""
    h, w = as_f64(H), as_f64(W)
    T = np.asarray(temperature, np.float64).reshape(-1)
    tok = np.asarray(tokens, np.int64).reshape(-1)
    z = h @ w.T
    M = z.shape[0]
    m = z.max(axis=1) if z.shape[1] else np.full(M, -np.inf)
    arg = np.argmax(z, axis=1).astype(np.int32)   # first index among equal maxima
    Ts = np.where(T > 0, T, 1.0)
    s = np.exp((z - m[:, None]) / Ts[:, None]).sum(axis=1)
    xt = np.full(M, np.nan)
    ok = tok >= 0
    xt[ok] = z[np.nonzero(ok)[0], tok[ok]]
    return dict(m=m, s=s, arg=arg, xt=xt, z=z)
