"""GPU parity: the sm_103a path (through the C ABI) against the oracle on the
same seeded inputs, element by element, on the five workloads at full size and
on edge cases; plus checks against library routines (torch.argmax,
torch.logsumexp) and the data-error contract."""

import math

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_13_gb300 as sv
from speculative_decoding_verification_13_gb300 import workloads as W
from parity import MARGIN, MAX_EXCUSED_FRAC, compare, run_gpu, run_oracle, t_offsets

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_verification_13_gb300 import build
    build.build()
    oracle.build()
    torch.cuda.init()


def check(batch_gpu, name, verifier=None, max_excused_frac=MAX_EXCUSED_FRAC):
    """GPU result against the oracle: non-exempt requests bit-exact; excused
    mismatches (exempt requests whose output differs) only at oracle margins
    below 1e-6 and at most max(1, max_excused_frac x verified rows); (p, q)
    within tolerance."""
    g = run_gpu(batch_gpu, verifier)
    assert g["err"][0] == 0, f"device error {g['err']}"
    cpu = batch_gpu.to("cpu")
    o = run_oracle(cpu)
    rep = compare(cpu, g, o, name)
    print(rep.line())
    assert not rep.structural, f"structurally invalid requests {rep.structural[:10]}"
    assert not rep.mismatched, f"non-exempt mismatches {rep.mismatched[:10]}: " + rep.line()
    assert rep.pq_bad == 0, rep.line()
    assert rep.excused_explained(), \
        f"excused mismatches at margins the arithmetic resolves: " + rep.line()
    assert len(rep.mismatched_exempt) <= rep.excused_allowed(max_excused_frac), \
        f"excused mismatches {rep.mismatched_exempt[:10]}: " + rep.line()
    return g, o, rep


# ---------------------------------------------------------------- workloads

CASES = [("c1", "t1"), ("c1", "greedy"), ("c2", "t0.7"), ("c2", "greedy"),
         ("c3", "s0.5"), ("c3", "s1"), ("c3", "s2"), ("c4", "default"), ("c5", "default")]


@pytest.mark.parametrize("cfg,variant", CASES, ids=[f"{c}:{v}" for c, v in CASES])
def test_workload_parity_full_size(cfg, variant):
    gen_dev = "cpu" if cfg in ("c1", "c2") else DEV
    batch = W.make_batch(cfg, variant, device=gen_dev).to(DEV)
    check(batch, f"{cfg}:{variant}")


def test_greedy_requests_match_torch_argmax_at_full_size():
    """Independent of the oracle: greedy decisions from torch.argmax (first
    index on ties) over every greedy request of the ragged workload."""
    batch = W.make_batch("c5", device=DEV)
    g = run_gpu(batch, with_pq=False)
    k = batch.k_per_req.cpu().numpy()
    T = batch.temperature.cpu().numpy()
    t_off = t_offsets(k)
    arg = torch.argmax(batch.target.float(), dim=1).cpu().numpy()
    x = batch.draft_tokens.cpu().numpy()
    n = 0
    for b in np.nonzero(T == 0)[0]:
        d0 = t_off[b] - b
        L = 0
        while L < k[b] and x[d0 + L] == arg[t_off[b] + L]:
            L += 1
        want = list(x[d0:d0 + L]) + [arg[t_off[b] + L]] + [-1] * (k[b] - L)
        assert g["acc"][b] == L
        assert g["tok"][t_off[b]:t_off[b + 1]].tolist() == want
        n += 1
    assert n > 200


def test_softmax_statistics_match_torch_logsumexp():
    """Row max and normaliser of unfiltered sampled rows against
    torch.logsumexp in float64 (library special case of the softmax)."""
    batch = W.make_batch("c3", "s1", device=DEV)
    v = sv.Verifier(DEV)
    run_gpu(batch, v)
    B, Rt, Rd = batch.batch, batch.target_rows, batch.draft_rows
    d = v.dump(B, Rt, Rd)
    stats = d["stats"]
    T = float(batch.temperature[0])
    rows = torch.cat([batch.target, batch.draft]).double()
    m = rows.max(dim=1).values
    lse = torch.logsumexp((rows - m[:, None]) / T, dim=1).cpu()
    np.testing.assert_array_equal(stats[:, 0].numpy(), m.cpu().numpy())
    rel = (stats[:, 1].log() - lse).abs() / 1.0
    assert float(rel.max()) < 1e-6


def test_no_filter_arrays_equal_switched_off_filters():
    """top_k = top_p = NULL (no threshold row pass is launched) gives the
    same results as arrays of switched-off values."""
    for cfg, var in (("c3", "s1"), ("c5", None), ("c1", "t1")):
        batch = W.make_batch(cfg, var, device=DEV, batch=None if cfg == "c1" else 24)
        v = sv.Verifier(DEV)
        args = (batch.target, batch.draft, batch.draft_tokens, batch.k_per_req,
                batch.temperature, batch.uniforms)
        a0, t0 = (x.cpu() for x in v(*args, batch.top_k, batch.top_p))
        a1, t1 = (x.cpu() for x in v(*args, None, None))
        assert v.error()[0] == 0
        assert torch.equal(a0, a1) and torch.equal(t0, t1), cfg


def test_filtered_kept_sets_match_oracle():
    batch = W.make_batch("c4", device=DEV, batch=16)
    v = sv.Verifier(DEV)
    g = run_gpu(batch, v)
    B, Rt, Rd = batch.batch, batch.target_rows, batch.draft_rows
    d = v.dump(B, Rt, Rd)
    rows = torch.cat([batch.target, batch.draft]).cpu()
    # rows the verification needed: positions up to the first rejection (the
    # bonus row after k acceptances); later rows are never filtered
    acc = g["acc"]
    k = batch.k_per_req.cpu().numpy()
    t_off = t_offsets(k)
    needed = []
    for b in range(B):
        L = int(acc[b])
        needed += [t_off[b] + i for i in range(L + 1)]
        needed += [Rt + t_off[b] - b + i for i in range(min(L + 1, k[b]))]
    assert len(needed) > 0
    for r in needed:
        p, _ = oracle.row_probs(rows[r], 1.0, 50, 0.9)
        nz = np.nonzero(p)[0]
        n = int(d["kept_count"][r])
        idx = d["kept_idx"][r, :n].numpy()
        assert sorted(idx.tolist()) == nz.tolist(), r
        # float-accurate weights (a few 1e-7 relative), well inside the 1e-5
        # relative bound on softmax probabilities
        np.testing.assert_allclose(d["kept_p"][r, :n].numpy(), p[idx], rtol=1e-6, atol=0)
        # kept order is (logit desc, index asc)
        vals = rows[r].float().numpy()[idx]
        assert all((vals[i] > vals[i + 1]) or (vals[i] == vals[i + 1] and idx[i] < idx[i + 1])
                   for i in range(n - 1))


# ---------------------------------------------------------------- edge cases

def padded(x):
    """Same values in a [rows, V] view whose row stride is a multiple of 16
    bytes (the library's alignment contract for TMA row copies)."""
    per = 16 // x.element_size()
    Vp = (x.shape[1] + per - 1) // per * per
    if Vp == x.shape[1]:
        return x
    y = torch.full((x.shape[0], Vp), float("nan"), dtype=x.dtype, device=x.device)
    y[:, :x.shape[1]] = x
    return y[:, :x.shape[1]]


def custom(k, T, V, dtype=torch.bfloat16, top_k=None, top_p=None, sig=1.0, seed=5):
    B = len(k)
    b = W.make_batch_from_params("edge", k, T, [sig] * B, V, dtype, seed, device=DEV,
                                 top_k=top_k, top_p=top_p)
    b.target, b.draft = padded(b.target), padded(b.draft)
    return b


@pytest.mark.parametrize("V", [1, 3, 7, 8, 9, 1000, 4097, 8193, 40000])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_vocab_sizes_and_ragged_tails(V, dtype):
    k = [0, 1, 3, 5, 2]
    T = [1.0, 0.0, 0.9, 1.3, 0.0]
    check(custom(k, T, V, dtype), f"V={V}")
    if V > 8:
        tk = [min(5, V - 1)] * 5
        check(custom(k, [1.0, 0.7, 1.0, 2.0, 0.0], V, dtype, top_k=tk, top_p=[0.9] * 5),
              f"V={V} filtered")


@pytest.mark.parametrize("V", [2048, 2049])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_draws_either_side_of_the_in_warp_draw(V, dtype):
    # up to 2048 elements the deciding warp takes the final draw itself; from
    # 2049 the draw pass and the locate kernel do: residuals and bonus draws,
    # unfiltered and by a kept-set threshold (top-p alone), on both sides
    k = [0, 1, 3, 5, 2, 7, 4, 6]
    T = [1.0, 0.0, 0.9, 1.3, 0.6, 1.0, 2.0, 0.8]
    check(custom(k, T, V, dtype, sig=0.5, seed=V), f"V={V}")
    check(custom(k, T, V, dtype, top_p=[0.9, 1.0, 0.5, 0.95, 0.3, 0.99, 0.9, 0.7], sig=0.5,
                 seed=V + 1), f"V={V} top-p alone")


def test_unaligned_row_stride_is_rejected_on_the_host():
    b = W.make_batch_from_params("edge", [1], [1.0], [1.0], 3, torch.float32, 5, device=DEV)
    with pytest.raises(sv.SpecVerifyError, match="UNSUPPORTED"):
        run_gpu(b)


def test_k_extremes_and_ragged_mix():
    k = [0, 32, 1, 31, 0, 16, 32]
    T = [1.0, 1.0, 0.0, 0.5, 0.0, 1.0, 0.0]
    check(custom(k, T, 5000, torch.bfloat16, sig=0.3), "k extremes")
    check(custom(k, [1.0] * 7, 5000, torch.bfloat16, top_k=[256, 1, 50, 17, 3, 256, 100],
                 top_p=[1.0, 1.0, 0.5, 0.95, 0.01, 0.9, 1.0], sig=0.3), "k extremes filtered")


def test_identical_target_and_draft_accepts_everything():
    b = custom([7, 7, 7], [1.0, 0.6, 1.0], 3000, torch.float32, top_k=[0, 0, 40],
               top_p=[1.0, 1.0, 0.8])
    k = b.k_per_req.cpu().numpy()
    t_off = t_offsets(k)
    for r in range(3):
        for i in range(7):
            b.draft[t_off[r] - r + i] = b.target[t_off[r] + i]
            # the argmax survives every filter, so p(x) = q(x) > 0
            b.draft_tokens[t_off[r] - r + i] = torch.argmax(b.target[t_off[r] + i])
    g, o, _ = check(b, "p == q")
    assert (g["acc"] == 7).all()


def _rows_with(b, fn):
    b.target.copy_(fn(b.target))
    b.draft.copy_(fn(b.draft))
    return b


@pytest.mark.parametrize("top_k", [1, 2, 50, 256])
def test_all_equal_logits_ties(top_k):
    b = _rows_with(custom([3, 2, 4], [1.0, 0.0, 0.8], 9000, torch.bfloat16,
                          top_k=[top_k] * 3, top_p=[0.9, 1.0, 1.0]),
                   lambda x: torch.zeros_like(x))
    check(b, f"ties top_k={top_k}")


@pytest.mark.parametrize("direction", ["ascending", "descending"])
def test_sorted_rows_adversarial_for_threshold(direction):
    def sorted_rows(x):
        s = torch.sort(x.float(), dim=1, descending=(direction == "descending")).values
        return s.to(x.dtype)
    for tk in (1, 64, 256):
        b = _rows_with(custom([4, 3], [1.0, 0.7], 60000, torch.bfloat16, top_k=[tk] * 2,
                              top_p=[1.0, 0.95]), sorted_rows)
        check(b, f"sorted {direction} top_k={tk}")


def test_negative_infinity_logits_are_legal():
    def mask(x):
        y = x.clone()
        y[:, ::3] = float("-inf")
        return y
    b = _rows_with(custom([3, 2, 2, 1], [1.0, 0.0, 0.5, 1.0], 7000, torch.float32,
                          top_k=[0, 0, 30, 0], top_p=[1.0, 1.0, 0.9, 1.0]), mask)
    check(b, "-inf")
    # a row that is -inf everywhere but one token
    b = custom([2], [1.0], 600, torch.float32)
    b.target[1] = float("-inf")
    b.target[1, 77] = 0.0
    check(b, "single finite token")


def test_one_hot_draft_like_ngram_proposal():
    b = custom([4, 4], [1.0, 0.8], 2000, torch.float32)
    x = b.draft_tokens.clone()
    b.draft.fill_(float("-inf"))
    b.draft[torch.arange(8, device=DEV), x.long()] = 0.0
    check(b, "one-hot draft")


def test_determinism_bitwise():
    b = W.make_batch("c3", "s1", device=DEV, batch=8)
    g1 = run_gpu(b)
    g2 = run_gpu(b)
    assert (g1["acc"] == g2["acc"]).all() and (g1["tok"] == g2["tok"]).all()
    assert np.array_equal(g1["pq"].view(np.int64), g2["pq"].view(np.int64))


def test_workspace_reuse_across_shapes():
    v = sv.Verifier(DEV)
    for cfg, B in (("c4", 8), ("c3", 4), ("c4", 2), ("c5", 12)):
        b = W.make_batch(cfg, device=DEV, batch=B)
        check(b, f"reuse {cfg}:{B}", verifier=v)


# ---------------------------------------------------------------- data errors

def _expect(b, code, bad_requests):
    v = sv.Verifier(DEV)
    g = run_gpu(b, v)
    assert g["err"][0] == code, g["err"]
    acc = g["acc"]
    for r in range(b.batch):
        if r in bad_requests:
            assert acc[r] == -1
        else:
            assert acc[r] >= 0
    return g


def test_data_errors_are_reported_per_request():
    b = custom([2, 3, 1], [1.0, 1.0, 0.0], 500, torch.float32)
    b.target[4, 10] = float("nan")
    _expect(b, 22, {1})
    b = custom([2, 3, 1], [1.0, 1.0, 0.0], 500, torch.float32)
    b.draft[0, 3] = float("inf")
    _expect(b, 22, {0})
    b = custom([2, 3, 1], [1.0, 1.0, 0.0], 500, torch.float32)
    b.draft_tokens[3] = 500
    _expect(b, 20, {1})
    b = custom([2, 3, 1], [1.0, 1.0, 0.0], 500, torch.float32)
    b.temperature[2] = -1.0
    _expect(b, 17, {2})
    b = custom([2, 3, 1], [1.0, 1.0, 0.0], 500, torch.float32, top_p=[1.0, 0.0, 1.0])
    _expect(b, 18, {1})
    b = custom([2, 3, 1], [1.0, 1.0, 0.0], 500, torch.float32, top_k=[0, -3, 0])
    _expect(b, 19, {1})
    b = custom([2, 3, 1], [1.0, 1.0, 0.0], 500, torch.float32)
    b.draft[:] = float("-inf")
    _expect(b, 22, {0, 1})


def test_every_request_failing_validation():
    """No row is streamed (every request fails the setup kernel's checks): the
    row pass's CTAs find only the end of the row list."""
    b = custom([2, 3, 1, 4], [1.0, 1.0, 0.0, 0.7], 500, torch.bfloat16)
    b.temperature[:] = -1.0
    g = _expect(b, 17, {0, 1, 2, 3})
    assert (g["tok"] == -1).all()


def test_batch_level_errors():
    b = custom([2, 3], [1.0, 1.0], 300, torch.float32)
    b.k_per_req[0] = 33
    g = run_gpu(b)
    assert g["err"][0] == 16 and (g["acc"] == -1).all() and (g["tok"] == -1).all()
    b = custom([2, 3], [1.0, 1.0], 300, torch.float32)
    b.k_per_req.copy_(torch.tensor([1, 3], dtype=torch.int32))   # sum(k) != draft rows
    g = run_gpu(b)
    assert g["err"][0] == 21 and (g["acc"] == -1).all()


def test_greedy_without_draft_logits():
    b = custom([3, 0, 2], [0.0, 0.0, 0.0], 800, torch.bfloat16)
    v = sv.Verifier(DEV)
    acc, tok = v(b.target, None, b.draft_tokens, b.k_per_req, b.temperature, b.uniforms)
    assert v.error()[0] == 0
    o = run_oracle(b.to("cpu"))
    assert acc.cpu().numpy().tolist() == o["accept_len"].tolist()
    assert tok.cpu().numpy().tolist() == o["tokens"].tolist()
    b2 = custom([3, 1], [0.0, 1.0], 800, torch.bfloat16)
    acc, tok = v(b2.target, None, b2.draft_tokens, b2.k_per_req, b2.temperature, b2.uniforms)
    assert v.error()[0] == 23 and int(acc[1]) == -1 and int(acc[0]) >= 0
