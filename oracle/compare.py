"""The parity rule: a verification result compared with the oracle's, request
by request.

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle/``): used by ``tests/`` and
by ``bench.py``'s oracle leg; the CUDA library never imports it.  Pure numpy,
no method arithmetic: it compares outputs and reads the margins the oracle
returns.

The rule follows the problem statement of the verification path:

* accept lengths and emitted tokens must be bit-exact, except for requests
  whose oracle margin shows that a floating-point implementation may
  legitimately take a decision the other way: |u - ratio| < 1e-5 at an
  evaluated position, or a CDF-boundary margin < 1e-5.  Two decisions of the
  method compare a cumulative distribution with a threshold: the final
  inverse-CDF draw (against u * S) and the top-p cut (the cumulative
  probability, in sorted order, against top_p; "Speculative decoding and
  multi-token prediction", "Why the output is identical").  The CDF-boundary
  margin is the smaller of the two;
* such requests are "exempt"; an exempt request whose output differs is an
  "excused mismatch".  A request whose output differs counts as one
  mismatched row (the decision where its outputs diverge).  An excused
  mismatch must be explained by rounding: its smallest oracle margin must lie
  below 1e-6 (EXPLAINED), ten times and more the error of float-accurate
  weights in a cumulative sum (a few 1e-8 for draws, below 1e-6 for a top-p
  cut over a nucleus of thousands of tokens), so a mismatch at a margin the
  arithmetic does resolve fails as a bug.  Their count must stay at or under
  ``max_excused_frac`` (1e-4) of the verified rows, with a floor of one (an
  exempt draw whose CDF boundary lies within 1e-8 of u S, about one exempt
  draw in a thousand, cannot be resolved by float-accurate weights);
* every request with a valid result must be structurally valid (accepted
  prefix equal to the drafts, one emitted token in [0, V), -1 after it);
* p_i(x_i), q_i(x_i) must match within 1e-5 relative (float32 logits) or
  2e-3 (bfloat16) at every position the decision examined.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

MARGIN = 1e-5          # |u - ratio| and CDF-boundary margins (draw and top-p cut)
MAX_EXCUSED_FRAC = 1e-4
EXPLAINED = 1e-6       # an excused mismatch's oracle margin must lie below this
PQ_RTOL = {"float32": 1e-5, "bfloat16": 2e-3}


def t_offsets(k):
    k = np.asarray(k, np.int64)
    return np.concatenate([[0], np.cumsum(k + 1)])


@dataclass
class Report:
    name: str
    requests: int
    rows: int
    exempt: int = 0                 # exempt requests
    exempt_rows: int = 0            # verified rows of exempt requests
    exempt_by: dict = field(default_factory=dict)  # cause -> requests
    mismatched: list = field(default_factory=list)          # non-exempt
    mismatched_exempt: list = field(default_factory=list)   # excused
    excused_margins: list = field(default_factory=list)     # their smallest oracle margin
    structural: list = field(default_factory=list)
    pq_max_rel: float = 0.0
    pq_bad: int = 0

    @property
    def excused_frac(self) -> float:
        return len(self.mismatched_exempt) / max(self.rows, 1)

    def excused_allowed(self, max_excused_frac: float = MAX_EXCUSED_FRAC) -> int:
        return max(1, int(max_excused_frac * self.rows))

    def excused_explained(self) -> bool:
        return all(m < EXPLAINED for m in self.excused_margins)

    def ok(self, max_excused_frac: float = MAX_EXCUSED_FRAC) -> bool:
        return (not self.structural and not self.mismatched and self.pq_bad == 0
                and self.excused_explained()
                and len(self.mismatched_exempt) <= self.excused_allowed(max_excused_frac))

    def summary(self) -> dict:
        return {"requests": self.requests, "verified_rows": self.rows,
                "exempt_requests": self.exempt, "exempt_rows": self.exempt_rows,
                "exempt_by": dict(self.exempt_by),
                "non_exempt_mismatches": len(self.mismatched),
                "excused_mismatches": len(self.mismatched_exempt),
                "excused_frac": self.excused_frac,
                "excused_margins": [float(m) for m in self.excused_margins],
                "structural_errors": len(self.structural),
                "pq_max_rel_err": self.pq_max_rel, "pq_out_of_tolerance": self.pq_bad}

    def line(self):
        return (f"{self.name}: {self.requests} requests, {self.rows} verified rows, "
                f"exempt {self.exempt} requests / {self.exempt_rows} rows "
                f"({self.exempt_rows / max(self.rows, 1):.2e} of rows; by cause "
                f"{self.exempt_by}), mismatches non-exempt {len(self.mismatched)} "
                f"excused {len(self.mismatched_exempt)} "
                f"({self.excused_frac:.2e} of rows, oracle margins "
                f"{['%.1e' % m for m in self.excused_margins]}), "
                f"pq max rel err {self.pq_max_rel:.2e}")


def exempt_mask(margins):
    """(exempt [B] bool, causes dict) from the oracle's per-request margins
    (columns: |u - ratio|, CDF margin of the draw, top-p cut margin)."""
    mg = np.asarray(margins, np.float64)
    acc, cdf, topp = mg[:, 0] < MARGIN, mg[:, 1] < MARGIN, mg[:, 2] < MARGIN
    causes = {"ratio": int(acc.sum()), "draw_cdf": int(cdf.sum()), "top_p_cdf": int(topp.sum())}
    return acc | cdf | topp, causes


def compare(k_per_req, temperature, vocab, draft_tokens, logit_dtype, g, o, name=""):
    """Compare a GPU result ``g`` (dict: acc [B], tok [R_t], pq [R_d, 2] or None)
    with the oracle's ``o`` (dict: accept_len, tokens, pq, margins)."""
    k = np.asarray(k_per_req, np.int64)
    T = np.asarray(temperature)
    V = int(vocab)
    B = len(k)
    t_off = t_offsets(k)
    d_off = t_off[:-1] - np.arange(B)
    x = np.asarray(draft_tokens)
    exempt, causes = exempt_mask(o["margins"])
    rep = Report(name, B, int(t_off[-1]), int(exempt.sum()),
                 int(sum(k[b] + 1 for b in np.nonzero(exempt)[0])), causes)
    for b in range(B):
        r0, r1 = t_off[b], t_off[b + 1]
        same = g["acc"][b] == o["accept_len"][b] and (g["tok"][r0:r1] == o["tokens"][r0:r1]).all()
        if not same:
            if exempt[b]:
                rep.mismatched_exempt.append(b)
                rep.excused_margins.append(float(np.nanmin(np.asarray(o["margins"][b], float))))
            else:
                rep.mismatched.append(b)
        L = g["acc"][b]
        if L >= 0:
            toks = g["tok"][r0:r1]
            ok = (0 <= L <= k[b]) and (toks[:L] == x[d_off[b]:d_off[b] + L]).all() \
                and 0 <= toks[L] < V and (toks[L + 1:] == -1).all()
            if not ok:
                rep.structural.append(b)
    if g.get("pq") is not None and len(x):
        tol = PQ_RTOL[logit_dtype]
        # positions the decision examined: 0 .. min(L, k - 1); the library may
        # leave later positions unevaluated (NaN)
        rows = np.concatenate([np.arange(d_off[b], d_off[b] + min(int(g["acc"][b]) + 1, k[b]))
                               for b in range(B)
                               if T[b] > 0 and o["accept_len"][b] >= 0 and g["acc"][b] >= 0]
                              or [np.zeros(0, int)])
        if len(rows):
            gp, op = g["pq"][rows], o["pq"][rows]
            pos = op > 0
            rel = np.zeros_like(op)
            rel[pos] = np.abs(gp[pos] - op[pos]) / op[pos]
            rel[~pos] = np.where(gp[~pos] == 0, 0.0, np.inf)
            rep.pq_max_rel = float(rel.max())
            rep.pq_bad = int((rel > tol).sum())
    return rep
