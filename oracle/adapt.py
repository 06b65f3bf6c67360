"""Oracle of the per-request speculation-length update (adaptive k).

TEST INFRASTRUCTURE ONLY: the plain definition in Python.  Only tests/ and
bench.py's CPU baseline may use it.

"Speculative decoding and multi-token prediction", section "Acceptance rate
is the whole economics": with acceptance rate alpha (the probability that one
drafted token survives verification) a pass yields E = (1 - alpha^(k+1)) /
(1 - alpha) tokens and costs about 1 + k c target steps (c: a draft step's
cost as a fraction of a target step); a position beyond k is worth alpha^k
tokens for a cost of c, so speculation pays while alpha^k stays above c (the
section's own example: about k = 6 at alpha 0.7 and c 0.1; its checklist:
"raise k only while alpha^k stays above the draft cost fraction").  The
section also says to measure alpha, and that it varies within a response.
Readings where the pages stop:

  A1  alpha is estimated per request from its verification outcomes: a pass
      with accept length L out of k drafts is L accepted positions and, when
      L < k, one rejected position (the verification rule stops at the
      first rejection, so later positions are not observed);
  A2  the counts decay geometrically, by d per pass (recent passes weigh
      more, as alpha drifts within a response), and start from one accepted
      and one rejected position (a uniform prior): alpha = (S + 1) / (S + F + 2);
  A3  the next k is the largest k in [k_min, k_max] with alpha^k > c, and
      k_min when even alpha^k_min <= c;
  A4  a request whose accept length is -1 (failed verification) keeps its
      counts and its k.
"""

from __future__ import annotations

import math

import numpy as np


def expected_tokens(alpha, k):
    """E = 1 + alpha + ... + alpha^k."""
    if alpha == 1.0:
        return k + 1.0
    return (1.0 - alpha ** (k + 1)) / (1.0 - alpha)


def speedup(alpha, k, c):
    """Tokens per pass over the pass cost in target steps, E / (1 + k c)."""
    return expected_tokens(alpha, k) / (1.0 + k * c)


def next_k(alpha, c, k_min, k_max):
    """Largest k in [k_min, k_max] with alpha^k > c (A3); alpha^k is the
    product of k factors alpha, taken in order (each product rounded)."""
    k = k_min
    p = 1.0
    for j in range(1, k_max + 1):
        p = p * alpha
        if j >= k_min and p > c:
            k = j
    return k


def adapt_k(accept_len, k_used, succ, fail, decay, c, k_min, k_max):
    """One update.  Returns (k_next [B] int32, succ' [B], fail' [B], alpha [B])."""
    B = len(accept_len)
    kn = np.empty(B, np.int32)
    s2 = np.array(succ, np.float64).copy()
    f2 = np.array(fail, np.float64).copy()
    al = np.empty(B)
    for b in range(B):
        L, k = int(accept_len[b]), int(k_used[b])
        if L >= 0:
            s2[b] = decay * s2[b] + L
            f2[b] = decay * f2[b] + (1.0 if L < k else 0.0)
        a = (s2[b] + 1.0) / (s2[b] + f2[b] + 2.0)
        al[b] = a
        kn[b] = next_k(a, c, k_min, k_max) if L >= 0 else k
    return kn, s2, f2, al
