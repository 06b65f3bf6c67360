"""The bounded-wait timeout path on the GPU, in the form that faults nothing:
with the test option set, one wait of the row pass (on a barrier nothing
arrives on) runs out after its short limit.  The library must record
SV_ERR_TIMEOUT, fail only the request whose row that CTA held (accept length
-1, tokens -1), verify every other request exactly as a normal call does, let
its own copies land, and leave the context usable for the next call."""

import time

import numpy as np
import pytest
import torch

import speculative_decoding_verification_13_gb300 as sv
from speculative_decoding_verification_13_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda"
SV_ERR_TIMEOUT = 24


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_verification_13_gb300 import build
    build.build()
    torch.cuda.init()


def _run(b, v, **kw):
    acc, tok = v(b.target, b.draft, b.draft_tokens, b.k_per_req, b.temperature, b.uniforms,
                 b.top_k, b.top_p, **kw)
    err = v.error()
    return acc.cpu().numpy().copy(), tok.cpu().numpy().copy(), err


@pytest.mark.parametrize("cfg,batch", [("c3", 8), ("c4", 8), ("c5", 24)])
def test_expired_wait_fails_one_request_and_the_context_recovers(cfg, batch):
    b = W.make_batch(cfg, device=DEV, batch=batch)
    v = sv.Verifier(DEV)
    acc0, tok0, err0 = _run(b, v)
    assert err0[0] == 0
    t0 = time.perf_counter()
    acc1, tok1, err1 = _run(b, v, test_expire_wait=True)
    elapsed = time.perf_counter() - t0
    assert err1[0] == SV_ERR_TIMEOUT, err1
    bad = err1[1]
    k = b.k_per_req.cpu().numpy()
    t_off = np.concatenate([[0], np.cumsum(k + 1)])
    assert 0 <= bad < b.batch
    assert acc1[bad] == -1 and (tok1[t_off[bad]:t_off[bad + 1]] == -1).all()
    others = np.arange(b.batch) != bad
    assert (acc1[others] == acc0[others]).all()
    for r in np.nonzero(others)[0]:
        assert (tok1[t_off[r]:t_off[r + 1]] == tok0[t_off[r]:t_off[r + 1]]).all()
    assert elapsed < 5.0  # the expiring wait is short (1 ms)
    # the context is usable and a normal call verifies everything again
    acc2, tok2, err2 = _run(b, v)
    assert err2[0] == 0
    assert (acc2 == acc0).all() and (tok2 == tok0).all()
