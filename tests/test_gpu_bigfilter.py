"""GPU parity for rows filtered by top-p alone or by a top-k above
SV_TOPK_MAX: the kept set is a threshold on the composite key (logit
descending, index ascending) found in the row pass, and draws use it as a
mask.  Checked against the oracle element by element (tokens and accept
lengths; p(x), q(x)), plus every row's kept-set size, last kept token and the
row's kept mass, at full size on Qwen3-vocabulary rows and on edge cases
(ties, -inf, sorted rows, tiny and huge top-k, fp32)."""

from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_13_gb300 as sv
from speculative_decoding_verification_13_gb300 import workloads as W
from parity import MARGIN, t_offsets
from test_gpu_parity import _rows_with, check, custom, padded

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_verification_13_gb300 import build
    build.build()
    oracle.build()
    torch.cuda.init()


def _row_params(b):
    """Per logit row (target rows, then draft rows): temperature, top-k, top-p."""
    k = b.k_per_req.cpu().numpy()
    B = len(k)
    T, tk, tp = (t.cpu().numpy() for t in (b.temperature, b.top_k, b.top_p))
    own = np.concatenate([np.repeat(np.arange(B), k + 1), np.repeat(np.arange(B), k)])
    return T[own], tk[own], tp[own]


def check_kept_sets(b, v, rows=None, threads=16):
    """Every filtered row's kept-set size and last kept token (in the composite
    order) against the oracle's kept set, unless the oracle's own top-p cut is
    within the CDF margin (then the sets may differ by the crossing token)."""
    B, Rt, Rd = b.batch, b.target_rows, b.draft_rows
    d = v.dump(B, Rt, Rd)
    T, tk, tp = _row_params(b)
    allrows = torch.cat([b.target, b.draft]).cpu()
    V = b.vocab
    big = np.nonzero((T > 0) & ((tp < 1) | ((tk > 0) & (tk < V))) &
                     ~((tk > 0) & (tk <= sv.SV_TOPK_MAX)))[0]
    if rows is not None:
        big = big[:rows]
    assert len(big) > 0

    def one(r):
        p, margin = oracle.row_probs(allrows[r], float(T[r]), int(tk[r]), float(tp[r]))
        return r, p, margin

    with ThreadPoolExecutor(threads) as ex:
        res = list(ex.map(one, big))
    close = 0
    for r, p, margin in res:
        nz = np.nonzero(p)[0]
        if margin < MARGIN:
            close += 1
            assert abs(int(d["kept_count"][r]) - len(nz)) <= 1, r
            continue
        assert int(d["kept_count"][r]) == len(nz), (r, int(d["kept_count"][r]), len(nz))
        x = allrows[r].double().numpy()[nz]
        last = nz[np.lexsort((-nz, x))[0]]  # smallest logit, then the largest index
        assert int(d["stats"][r, 4]) == last, r
        # the kept mass, relative to the row max: sum over the kept set of
        # exp((x - max) / T), float-accurate on the GPU
        want = np.exp((x - float(allrows[r].double().max())) / np.float64(np.float32(T[r]))).sum()
        assert abs(float(d["stats"][r, 1]) - want) <= 5e-6 * want, r
    print(f"kept sets: {len(res)} rows, {close} within the top-p margin")
    return len(res)


def test_top_p_alone_full_size():
    """c4 with top-p 0.9 and no top-k: nuclei of thousands of tokens."""
    b = W.make_batch("c4p", device=DEV)
    v = sv.Verifier(DEV)
    g, o, rep = check(b, "c4p", verifier=v)
    check_kept_sets(b, v, rows=600)


def test_top_p_with_large_top_k_full_size():
    B = 32
    b = W.make_batch_from_params("tk1000", [15] * B, [1.0] * B, [1.0] * B, W.VOCAB_QWEN3,
                                 torch.bfloat16, 11, device=DEV, top_k=[1000] * B,
                                 top_p=[0.95] * B)
    v = sv.Verifier(DEV)
    check(b, "top-k 1000 + top-p 0.95", verifier=v)
    check_kept_sets(b, v)


def test_top_k_vocab_minus_one():
    V = W.VOCAB_QWEN3
    b = W.make_batch_from_params("tkV-1", [7] * 8, [1.0, 0.3, 1.5, 1.0] * 2, [1.0] * 8, V,
                                 torch.bfloat16, 12, device=DEV, top_k=[V - 1] * 8,
                                 top_p=[1.0] * 4 + [0.99] * 4)
    v = sv.Verifier(DEV)
    check(b, "top-k V-1", verifier=v)
    check_kept_sets(b, v)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_mixed_filters_in_one_batch(dtype):
    """Greedy, unfiltered, small top-k (candidate path) and threshold rows
    (top-p alone, top-k 257 and 5000, top-k with top-p) side by side."""
    k = [3, 5, 2, 6, 4, 1, 7, 3, 0, 5]
    T = [1.0, 0.0, 0.8, 1.2, 0.3, 1.0, 0.6, 1.0, 1.0, 1.5]
    tk = [0, 0, 50, 0, 257, 5000, 0, 300, 2000, 0]
    tp = [1.0, 1.0, 0.9, 0.8, 1.0, 1.0, 0.95, 0.5, 0.99, 0.2]
    b = custom(k, T, 20000, dtype, top_k=tk, top_p=tp)
    v = sv.Verifier(DEV)
    check(b, f"mixed filters {dtype}", verifier=v)
    check_kept_sets(b, v)


@pytest.mark.parametrize("top_p", [0.3, 0.999])
def test_all_equal_logits_top_p(top_p):
    """Every logit equal: the crossing bin holds the whole row (the exact radix
    path), and ties go to the lower index."""
    b = _rows_with(custom([3, 2], [1.0, 0.8], 9000, torch.bfloat16, top_p=[top_p] * 2),
                   lambda x: torch.zeros_like(x))
    v = sv.Verifier(DEV)
    check(b, f"ties top_p={top_p}", verifier=v)
    check_kept_sets(b, v)


def test_heavy_ties_large_top_k():
    """Logits on 16 levels: big tie groups at the top-k boundary."""
    b = _rows_with(custom([4, 3], [1.0, 0.7], 30000, torch.bfloat16, top_k=[4000, 12000],
                          top_p=[1.0, 0.9]),
                   lambda x: torch.round(x.float() * 1.5).clamp(-15, 0).to(x.dtype))
    v = sv.Verifier(DEV)
    check(b, "heavy ties", verifier=v)
    check_kept_sets(b, v)


def test_negative_infinity_with_top_p():
    def mask(x):
        y = x.clone()
        y[:, 1::2] = float("-inf")
        return y
    b = _rows_with(custom([3, 4], [1.0, 0.6], 7000, torch.float32, top_k=[0, 3000],
                          top_p=[0.9, 1.0]), mask)
    v = sv.Verifier(DEV)
    check(b, "-inf top-p", verifier=v)
    check_kept_sets(b, v)


@pytest.mark.parametrize("direction", ["ascending", "descending"])
def test_sorted_rows_top_p(direction):
    def sorted_rows(x):
        s = torch.sort(x.float(), dim=1, descending=(direction == "descending")).values
        return s.to(x.dtype)
    b = _rows_with(custom([4, 3], [1.0, 0.7], 60000, torch.bfloat16, top_k=[0, 700],
                          top_p=[0.9, 0.95]), sorted_rows)
    v = sv.Verifier(DEV)
    check(b, f"sorted {direction} top-p", verifier=v)
    check_kept_sets(b, v)


def test_top_p_alone_is_no_longer_a_data_error():
    b = custom([2, 3, 1], [1.0, 1.0, 0.0], 500, torch.float32, top_k=[0, 0, 0],
               top_p=[0.5, 1.0, 1.0])
    g, _, _ = check(b, "top-p alone, small")
    assert (g["acc"] >= 0).all()


# ---------------------------------------------------------------- sampler

def _sampler_check(x, k, T, tk, tp, u, name):
    s = sv.DraftSampler(DEV)
    tok, q = s(x, k, T, u, tk, tp, with_q=True)
    torch.cuda.synchronize()
    assert s.error()[0] == 0
    o = oracle.draft_sample(x.cpu(), k.cpu(), T.cpu(), u.cpu(), tk.cpu(), tp.cpu(), threads=16)
    tok, q = tok.cpu().numpy(), q.cpu().numpy()
    exempt = (o["margins"][:, 0] < MARGIN) | (o["margins"][:, 1] < MARGIN)
    mism = tok != o["tokens"]
    bad = np.nonzero(mism & ~exempt)[0]
    print(f"{name}: {len(tok)} rows, exempt {int(exempt.sum())}, non-exempt mismatches "
          f"{len(bad)}, excused {int((mism & exempt).sum())}")
    assert len(bad) == 0, bad[:10]
    exc = mism & exempt
    assert int(exc.sum()) <= max(1, int(1e-4 * len(tok)))
    if exc.any():
        assert (np.nanmin(o["margins"][exc], axis=1) < 1e-6).all()
    same = ~mism & ~np.isnan(o["q"])
    rel = np.abs(q[same] - o["q"][same]) / np.maximum(o["q"][same], 1e-30)
    tol = 2e-3 if x.dtype == torch.bfloat16 else 1e-5
    assert rel.max() <= tol


@pytest.mark.parametrize("case", ["c4p", "tk1000", "tkV-1"])
def test_sampler_threshold_rows(case):
    V = W.VOCAB_QWEN3
    B = 48
    tk = {"c4p": 0, "tk1000": 1000, "tkV-1": V - 1}[case]
    tp = {"c4p": 0.9, "tk1000": 0.95, "tkV-1": 1.0}[case]
    b = W.make_batch_from_params(case, [15] * B, [1.0] * (B // 2) + [0.7] * (B // 2), [1.0] * B,
                                 V, torch.bfloat16, 21, device=DEV, top_k=[tk] * B,
                                 top_p=[tp] * B)
    g = torch.Generator(device=DEV)
    g.manual_seed(31)
    u = torch.rand(b.draft_rows, generator=g, device=DEV)
    _sampler_check(b.draft, b.k_per_req, b.temperature, b.top_k, b.top_p, u, f"sampler {case}")
