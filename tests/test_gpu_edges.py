"""Edge cases at the limits of the boundary, against the oracle element by
element: the largest vocabulary, the largest k with the largest top-k and a
top-p cut, a batch large enough for the setup kernel to work in several
chunks, and an empty batch on the device."""

import numpy as np
import pytest
import torch

import speculative_decoding_verification_13_gb300 as sv
from speculative_decoding_verification_13_gb300 import workloads as W
from test_gpu_parity import check

pytestmark = pytest.mark.gpu

DEV = "cuda"


def test_largest_vocabulary():
    """V = SV_VOCAB_MAX (2^22): a filtered request (top-k 256 keeps more
    survivors than the row pass's speculative buffer, so every row takes the
    certified path), an unfiltered sampled request and a greedy request."""
    V = sv.SV_VOCAB_MAX
    b = W.make_batch_from_params("V=2^22", [2, 2, 2], [1.0, 0.8, 0.0], [1.0, 1.0, 1.0], V,
                                 torch.bfloat16, 77, device=DEV, top_k=[256, 0, 0],
                                 top_p=[0.95, 1.0, 1.0])
    check(b, "V=2^22")


def test_largest_k_and_top_k_with_top_p():
    """k = SV_MAX_K with top-k = SV_TOPK_MAX and several top-p cuts; low draft
    noise so that many positions are accepted (several decision waves)."""
    b = W.make_batch_from_params("k=32 top-k 256", [32, 32, 17, 32], [1.0, 1.0, 0.7, 0.4],
                                 [0.3, 0.05, 0.3, 0.02], 50000, torch.bfloat16, 78, device=DEV,
                                 top_k=[256, 256, 100, 256], top_p=[0.9, 0.5, 0.99, 1.0])
    g, _, _ = check(b, "k=32 top-k 256")
    assert int(g["acc"].max()) >= 8  # the late waves were exercised


def test_filtered_full_acceptance_at_wave_multiples():
    """Draft logits equal to the target's make p = q, so every draft is
    accepted and the bonus row is drawn from.  k a multiple of the decision
    wave (8 positions) leaves that wave no spare warp for the bonus row, which
    then takes a wave of its own; k = 0 and k = 7 bracket it."""
    ks = [8, 16, 24, 32, 0, 7]
    b = W.make_batch_from_params("full acceptance", ks, [1.0, 0.9, 1.2, 0.7, 1.0, 1.0],
                                 [0.0] * len(ks), 32000, torch.bfloat16, 80, device=DEV,
                                 top_k=[64, 256, 40, 128, 10, 200],
                                 top_p=[0.9, 1.0, 0.8, 0.95, 1.0, 0.7])
    g, _, _ = check(b, "full acceptance")
    assert g["acc"].tolist() == ks


def test_many_requests_several_setup_chunks():
    """2500 requests (the setup kernel handles 1024 per chunk) mixing greedy,
    unfiltered and filtered sampling, k from 0 to 6."""
    rng = np.random.default_rng(79)
    B = 2500
    k = rng.integers(0, 7, B)
    kind = rng.integers(0, 3, B)
    T = np.where(kind == 0, 0.0, rng.uniform(0.5, 1.5, B))
    tk = np.where(kind == 2, rng.integers(1, 60, B), 0)
    tp = np.where(kind == 2, rng.uniform(0.5, 1.0, B), 1.0)
    b = W.make_batch_from_params("B=2500", k.tolist(), T.tolist(), [0.8] * B, 2048,
                                 torch.float32, 79, device=DEV, top_k=tk.tolist(),
                                 top_p=tp.tolist())
    check(b, "B=2500")


@pytest.mark.parametrize("B", [1024, 1025])
def test_setup_chunk_boundary(B):
    """B = 1024 is the largest batch the setup kernel handles in one chunk
    (eight CTAs sharing the row-list writes); B = 1025 takes two chunks (one
    CTA).  Mixed greedy, unfiltered and filtered requests, k from 0 to 4."""
    rng = np.random.default_rng(B)
    k = rng.integers(0, 5, B)
    kind = rng.integers(0, 3, B)
    T = np.where(kind == 0, 0.0, rng.uniform(0.5, 1.5, B))
    tk = np.where(kind == 2, rng.integers(1, 40, B), 0)
    tp = np.where(kind == 2, rng.uniform(0.5, 1.0, B), 1.0)
    b = W.make_batch_from_params(f"B={B}", k.tolist(), T.tolist(), [0.8] * B, 512,
                                 torch.float32, B, device=DEV, top_k=tk.tolist(),
                                 top_p=tp.tolist())
    check(b, f"B={B}")


def test_empty_batch_on_device():
    V = 1000
    target = torch.zeros(0, V, dtype=torch.bfloat16, device=DEV)
    draft = torch.zeros(0, V, dtype=torch.bfloat16, device=DEV)
    e_i = torch.zeros(0, dtype=torch.int32, device=DEV)
    e_f = torch.zeros(0, dtype=torch.float32, device=DEV)
    acc, tok = sv.verify(target, draft, e_i, e_i, e_f, e_f)
    torch.cuda.synchronize()
    assert acc.numel() == 0 and tok.numel() == 0
