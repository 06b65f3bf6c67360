"""Helpers for the GPU-vs-oracle parity tests: run both sides on the same
seeded inputs and compare element by element.

The comparison rule lives in ``oracle/compare.py`` (shared with bench.py's
oracle leg): accept lengths and emitted tokens bit-exact except for requests
whose oracle margin is below 1e-5 (|u - ratio|, or a CDF-boundary margin: the
final draw's or the top-p cut's); such excused mismatches may not exceed 1e-4
of the verified rows; p_i(x_i), q_i(x_i) within 1e-5 relative (float32
logits) or 2e-3 (bfloat16) at every position the decision examined.
"""

from __future__ import annotations

import os

import torch

import oracle
import speculative_decoding_verification_13_gb300 as sv
from oracle.compare import MARGIN, MAX_EXCUSED_FRAC, Report, t_offsets  # noqa: F401
from oracle.compare import compare as _compare

PQ_RTOL = {torch.float32: 1e-5, torch.bfloat16: 2e-3}


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


def compare(batch_cpu, g, o, name="") -> Report:
    dt = "bfloat16" if batch_cpu.target.dtype == torch.bfloat16 else "float32"
    return _compare(batch_cpu.k_per_req.numpy(), batch_cpu.temperature.numpy(),
                    batch_cpu.vocab, batch_cpu.draft_tokens.numpy(), dt, g, o, name)
