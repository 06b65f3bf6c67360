"""Helpers for the GPU-vs-oracle parity tests: run both sides on the same
seeded inputs and compare element by element.

Comparison rule: accept lengths and emitted tokens must be bit-exact for every
request except those whose oracle margin says a floating-point implementation
may legitimately round the other way: |u - ratio| < 1e-5 or CDF-boundary
margin < 1e-5 (the tolerances of the verification path), or top-p decision
margin < 1e-12 (both sides take that decision in double precision).  Those
requests are counted and reported; every request must still be structurally
valid.  p_i(x_i) and q_i(x_i) must match within 1e-5 relative for float32
logits and 2e-3 for bfloat16 logits at every position the decision examined
(up to the first rejection).
"""

from __future__ import annotations

import os
from dataclasses import dataclass, field

import numpy as np
import torch

import oracle
import speculative_decoding_verification_13_gb300 as sv

MARGIN = 1e-5
TOPP_MARGIN = 1e-12
PQ_RTOL = {torch.float32: 1e-5, torch.bfloat16: 2e-3}


def t_offsets(k):
    k = np.asarray(k, np.int64)
    return np.concatenate([[0], np.cumsum(k + 1)])


def run_gpu(batch, verifier=None, with_pq=True):
    dev = batch.target.device
    v = verifier or sv.Verifier(dev)
    Rd = batch.draft_rows
    pq = torch.full((max(Rd, 1), 2), float("nan"), dtype=torch.float64, device=dev) \
        if with_pq else None
    acc, tok = v(batch.target, batch.draft, batch.draft_tokens, batch.k_per_req,
                 batch.temperature, batch.uniforms, batch.top_k, batch.top_p, out_pq=pq)
    err = v.error()
    return dict(acc=acc.cpu().numpy(), tok=tok.cpu().numpy(),
                pq=pq[:Rd].cpu().numpy() if with_pq else None, err=err, verifier=v)


def run_oracle(batch_cpu, threads=None):
    threads = threads or min(32, os.cpu_count() or 1)
    return oracle.verify(batch_cpu.target, batch_cpu.draft, batch_cpu.draft_tokens,
                         batch_cpu.k_per_req, batch_cpu.temperature, batch_cpu.top_k,
                         batch_cpu.top_p, batch_cpu.uniforms, threads=threads)


@dataclass
class Report:
    name: str
    requests: int
    rows: int
    exempt: int
    mismatched: list = field(default_factory=list)
    mismatched_exempt: list = field(default_factory=list)
    structural: list = field(default_factory=list)
    pq_max_rel: float = 0.0
    pq_bad: int = 0

    def line(self):
        return (f"{self.name}: {self.requests} requests, {self.rows} verified rows, "
                f"exempt {self.exempt} ({self.exempt / max(self.rows, 1):.2e} of rows), "
                f"mismatches non-exempt {len(self.mismatched)} exempt "
                f"{len(self.mismatched_exempt)}, pq max rel err {self.pq_max_rel:.2e}")


def compare(batch_cpu, g, o, name=""):
    k = batch_cpu.k_per_req.numpy().astype(np.int64)
    T = batch_cpu.temperature.numpy()
    V = batch_cpu.vocab
    B = len(k)
    t_off = t_offsets(k)
    d_off = t_off[:-1] - np.arange(B)
    x = batch_cpu.draft_tokens.numpy()
    mg = o["margins"]
    exempt = (mg[:, 0] < MARGIN) | (mg[:, 1] < MARGIN) | (mg[:, 2] < TOPP_MARGIN)
    rep = Report(name, B, int(t_off[-1]), int(exempt.sum()))
    for b in range(B):
        r0, r1 = t_off[b], t_off[b + 1]
        same = g["acc"][b] == o["accept_len"][b] and (g["tok"][r0:r1] == o["tokens"][r0:r1]).all()
        if not same:
            (rep.mismatched_exempt if exempt[b] else rep.mismatched).append(b)
        L = g["acc"][b]
        if L >= 0:
            toks = g["tok"][r0:r1]
            ok = (0 <= L <= k[b]) and (toks[:L] == x[d_off[b]:d_off[b] + L]).all() \
                and 0 <= toks[L] < V and (toks[L + 1:] == -1).all()
            if not ok:
                rep.structural.append(b)
    if g["pq"] is not None and batch_cpu.draft_rows:
        tol = PQ_RTOL[batch_cpu.target.dtype]
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
