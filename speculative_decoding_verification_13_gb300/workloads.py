"""Seeded synthetic inputs for speculative-decoding verification.

This module only *makes inputs*; it holds none of the verification
arithmetic and imports neither the oracle nor the CUDA library.  Both sides
consume the tensors it returns.

Recipe (stand-in for the pages' workloads: the Qwen3 vocabulary V = 151936 of
"FlashMap…" §5, DFlash's block of 16 including the anchor, "DFlash" §2.3 and
§6 Table 1, and the typical speculation length 3-8 of "Speculative decoding and
multi-token prediction", "Draft and verify"):

* target logit of token v in a row: ``-1.1 * ln(1 + pi(v)) + N(0, 0.5^2)``
  with ``pi`` a fresh uniformly random permutation of 0..V-1 per row (a Zipf
  profile over ranks, placed at random token ids);
* draft row i of a request: target row i of that request ``+ N(0, sigma^2)``;
* drafted tokens: sampled from the drafter's own distribution, i.e. softmax of
  the (stored-precision) draft row at the request temperature with the
  request's top-k / top-p applied (drawn with torch's softmax / topk /
  multinomial, standing in for a drafter); argmax of the draft row at T = 0;
* uniforms: ``U[0, 1)``, one per target row (row t_off[b] + i drives draft i,
  row t_off[b] + k_b the final residual / bonus draw).

All draws come from one ``torch.Generator`` seeded with ``seed``, in a fixed
order: per-request parameters, permutations, target noise, draft noise, draft
tokens, uniforms.  Logits are rounded to the storage dtype at generation, so
every consumer reads identical values.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import torch

VOCAB_QWEN3 = 151936


@dataclass
class Batch:
    name: str
    target: torch.Tensor          # [R_t, V] float32 or bfloat16
    draft: torch.Tensor           # [R_d, V] same dtype
    draft_tokens: torch.Tensor    # [R_d] int32
    k_per_req: torch.Tensor       # [B] int32
    temperature: torch.Tensor     # [B] float32 (0 = greedy)
    top_k: torch.Tensor           # [B] int32 (0 = off)
    top_p: torch.Tensor           # [B] float32 (1 = off)
    uniforms: torch.Tensor        # [R_t] float32
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.k_per_req.shape[0])

    @property
    def vocab(self) -> int:
        return int(self.target.shape[1])

    @property
    def target_rows(self) -> int:
        return int(self.target.shape[0])

    @property
    def draft_rows(self) -> int:
        return int(self.draft.shape[0])

    def filters(self):
        """(top_k, top_p) for a call: None for both when the workload has no
        filter (its arrays hold only the switched-off values), which tells
        the library that no row can need the kept-set threshold pass."""
        if self.meta.get("filtered", True):
            return self.top_k, self.top_p
        return None, None

    def logit_bytes(self) -> int:
        es = self.target.element_size()
        return (self.target_rows + self.draft_rows) * self.vocab * es

    def to(self, device, non_blocking=False) -> "Batch":
        f = lambda t: t.to(device, non_blocking=non_blocking)
        return Batch(self.name, f(self.target), f(self.draft), f(self.draft_tokens),
                     f(self.k_per_req), f(self.temperature), f(self.top_k), f(self.top_p),
                     f(self.uniforms), dict(self.meta))

    def requests(self, idx) -> "Batch":
        """Sub-batch of the given request indices (rows copied, order kept)."""
        k = self.k_per_req.cpu().long()
        t_off = torch.cat([torch.zeros(1, dtype=torch.long), torch.cumsum(k + 1, 0)])
        trows, drows = [], []
        for b in idx:
            b = int(b)
            trows.append(torch.arange(t_off[b], t_off[b + 1]))
            d0 = int(t_off[b]) - b
            drows.append(torch.arange(d0, d0 + int(k[b])))
        tr = torch.cat(trows).to(self.target.device)
        dr = torch.cat(drows).to(self.target.device) if drows else tr[:0]
        bi = torch.as_tensor([int(b) for b in idx], device=self.k_per_req.device)
        return Batch(self.name + "[sub]", self.target[tr], self.draft[dr],
                     self.draft_tokens[dr], self.k_per_req[bi], self.temperature[bi],
                     self.top_k[bi], self.top_p[bi], self.uniforms[tr], dict(self.meta))


# The five workloads.  Sizes and distributions follow the configurations the
# verification path is measured on; ``variant`` picks the temperature / sigma
# run where a configuration has several.
CONFIGS = {
    "c1": dict(B=1, k=4, V=1024, dtype=torch.float32, sigma=1.0, seed=1301,
               variants={"t1": 1.0, "greedy": 0.0}),
    "c2": dict(B=8, k=7, V=32000, dtype=torch.float32, sigma=0.7, seed=1302,
               variants={"t0.7": 0.7, "greedy": 0.0}),
    "c3": dict(B=32, k=15, V=VOCAB_QWEN3, dtype=torch.bfloat16, temp=1.0, seed=1303,
               variants={"s0.5": 0.5, "s1": 1.0, "s2": 2.0}),
    "c4": dict(B=256, k=15, V=VOCAB_QWEN3, dtype=torch.bfloat16, temp=1.0, sigma=1.0,
               top_k=50, top_p=0.9, seed=1304, variants={"default": None}),
    # c4 with top-p alone (no top-k): the nucleus of a Zipf row then holds
    # thousands of tokens
    "c4p": dict(B=256, k=15, V=VOCAB_QWEN3, dtype=torch.bfloat16, temp=1.0, sigma=1.0,
                top_k=0, top_p=0.9, seed=1306, variants={"default": None}),
    "c5": dict(B=1024, k=None, V=VOCAB_QWEN3, dtype=torch.bfloat16, seed=1305,
               variants={"default": None}),
}


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _zipf_rows(n, V, g, device, chunk):
    """``-1.1 ln(1 + pi(v)) + N(0, 0.5^2)`` rows in float32, pi a random permutation per row."""
    out = torch.empty(n, V, dtype=torch.float32, device=device)
    for r0 in range(0, n, chunk):
        r1 = min(n, r0 + chunk)
        keys = torch.rand(r1 - r0, V, generator=g, device=device)
        perm = torch.argsort(keys, dim=1)
        del keys
        out[r0:r1] = -1.1 * torch.log1p(perm.to(torch.float32))
        del perm
    for r0 in range(0, n, chunk):
        r1 = min(n, r0 + chunk)
        out[r0:r1] += 0.5 * torch.randn(r1 - r0, V, generator=g, device=device)
    return out


def _sample_draft_tokens(draft, temps, top_k, top_p, owner, g, chunk):
    """Drafter stand-in: x_i ~ softmax(draft_i / T) with the request's top-k /
    top-p, or argmax at T = 0 (library calls only)."""
    n, V = draft.shape
    out = torch.empty(n, dtype=torch.int64, device=draft.device)
    for r0 in range(0, n, chunk):
        r1 = min(n, r0 + chunk)
        x = draft[r0:r1].float()
        T = temps[owner[r0:r1]]
        tk = top_k[owner[r0:r1]]
        tp = top_p[owner[r0:r1]]
        greedy = T == 0
        Ts = torch.where(greedy, torch.ones_like(T), T)
        z = x / Ts[:, None]
        on = (tk > 0) & (tk < V)
        n_on = int(on.sum().item())
        samp = None
        if n_on < r1 - r0:  # rows without top-k: the whole softmax, then top-p
            pr = torch.softmax(z, dim=1)
            if bool(((tp < 1) & ~on).any()):
                # nucleus over the whole row: sort (logit desc, index asc),
                # keep while the mass before a token is below top_p
                order = torch.argsort(z, dim=1, descending=True, stable=True)
                ps = pr.gather(1, order)
                before = torch.cumsum(ps, dim=1) - ps
                # the first token always stays (also for an invalid top_p of a
                # data-error test, so that the draw is defined)
                first = torch.arange(V, device=x.device)[None] == 0
                keep = (before < tp[:, None]) | first
                ps = torch.where(keep, ps, torch.zeros_like(ps))
                pr = torch.zeros_like(pr).scatter_(1, order, ps)
                del order, ps, before, keep
            samp = torch.multinomial(pr, 1, generator=g).squeeze(1)
        if n_on:
            kk = int(torch.where(on, tk, torch.zeros_like(tk)).max().item())
            vals, idx = torch.topk(z, kk, dim=1)
            # each row's own top-k first (renormalised over it), then top-p
            # (rows without top-k keep slot 0 here; their token comes from above)
            col = torch.arange(kk, device=x.device)[None]
            in_k = (col < tk[:, None]) & on[:, None] | (col == 0) & ~on[:, None]
            pr = torch.softmax(vals.masked_fill(~in_k, float("-inf")), dim=1)
            before = torch.cumsum(pr, dim=1) - pr
            keep = ((before < tp[:, None]) | (col == 0)) & in_k
            pr = torch.where(keep, pr, torch.zeros_like(pr))
            pick = torch.multinomial(pr, 1, generator=g).squeeze(1)
            samp_k = idx.gather(1, pick[:, None]).squeeze(1)
            samp = samp_k if samp is None else torch.where(on, samp_k, samp)
        out[r0:r1] = torch.where(greedy, torch.argmax(x, dim=1), samp)
    return out.to(torch.int32)


def make_batch_from_params(name, k_list, temps, sigmas, V, dtype, seed, device="cpu",
                           top_k=None, top_p=None, chunk=None, g=None) -> Batch:
    """Build a batch from explicit per-request parameters (lists or tensors)."""
    device = torch.device(device)
    g = g if g is not None else _gen(device, seed)
    k = torch.as_tensor(k_list, dtype=torch.int32)
    B = int(k.shape[0])
    T = torch.as_tensor(temps, dtype=torch.float32).reshape(B)
    sig = torch.as_tensor(sigmas, dtype=torch.float32).reshape(B)
    tk = torch.zeros(B, dtype=torch.int32) if top_k is None else \
        torch.as_tensor(top_k, dtype=torch.int32).reshape(B)
    tp = torch.ones(B, dtype=torch.float32) if top_p is None else \
        torch.as_tensor(top_p, dtype=torch.float32).reshape(B)
    kl = k.long()
    Rt, Rd = int((kl + 1).sum()), int(kl.sum())
    if chunk is None:
        chunk = max(1, min(512, (1 << 27) // max(V, 1)))
    target32 = _zipf_rows(Rt, V, g, device, chunk)
    # Draft row i of request b pairs with target row i of request b.
    t_off = torch.cat([torch.zeros(1, dtype=torch.long), torch.cumsum(kl + 1, 0)])
    owner_d = torch.repeat_interleave(torch.arange(B), kl)
    pos_d = torch.arange(Rd) - torch.repeat_interleave(t_off[:-1] - torch.arange(B), kl) \
        if Rd else torch.zeros(0, dtype=torch.long)
    src = (t_off[:-1][owner_d] + pos_d) if Rd else torch.zeros(0, dtype=torch.long)
    draft32 = torch.empty(Rd, V, dtype=torch.float32, device=device)
    src_d, own_d = src.to(device), owner_d.to(device)
    sig_d = sig.to(device)
    for r0 in range(0, Rd, chunk):
        r1 = min(Rd, r0 + chunk)
        noise = torch.randn(r1 - r0, V, generator=g, device=device)
        draft32[r0:r1] = target32[src_d[r0:r1]] + sig_d[own_d[r0:r1], None] * noise
    target = target32.to(dtype)
    del target32
    draft = draft32.to(dtype)
    del draft32
    if Rd:
        tokens = _sample_draft_tokens(draft, T.to(device), tk.to(device), tp.to(device),
                                      own_d, g, chunk)
    else:
        tokens = torch.zeros(0, dtype=torch.int32, device=device)
    uniforms = torch.rand(Rt, generator=g, device=device)
    meta = dict(seed=seed, sigmas=sig.tolist() if B <= 64 else None, V=V,
                filtered=top_k is not None or top_p is not None)
    return Batch(name, target, draft, tokens, k.to(device), T.to(device), tk.to(device),
                 tp.to(device), uniforms, meta)


def make_batch(config: str, variant: str | None = None, device="cpu", batch: int | None = None,
               seed_offset: int = 0) -> Batch:
    """One of the five workloads.  ``batch`` overrides B (smaller parity cases,
    larger replicas); ``seed_offset`` gives independent replicas (one per rank)."""
    c = CONFIGS[config]
    if variant is None:
        variant = next(iter(c["variants"]))
    B = c["B"] if batch is None else batch
    seed = c["seed"] + seed_offset
    name = f"{config}:{variant}" + (f":B{B}" if batch is not None else "")
    V, dtype = c["V"], c["dtype"]
    if config in ("c1", "c2"):
        T = c["variants"][variant]
        return make_batch_from_params(name, [c["k"]] * B, [T] * B, [c["sigma"]] * B, V, dtype,
                                      seed, device)
    if config == "c3":
        sigma = c["variants"][variant]
        return make_batch_from_params(name, [c["k"]] * B, [c["temp"]] * B, [sigma] * B, V,
                                      dtype, seed, device)
    if config in ("c4", "c4p"):
        return make_batch_from_params(name, [c["k"]] * B, [c["temp"]] * B, [c["sigma"]] * B,
                                      V, dtype, seed, device, top_k=[c["top_k"]] * B,
                                      top_p=[c["top_p"]] * B)
    if config == "c5":
        # Ragged: k ~ U{1..15}; 25% greedy, else T ~ U[0.3, 1.2]; sigma ~ U[0.3, 2].
        g = _gen(torch.device(device), seed)
        k = torch.randint(1, 16, (B,), generator=g, device=device).cpu()
        greedy = torch.rand(B, generator=g, device=device).cpu() < 0.25
        T = 0.3 + 0.9 * torch.rand(B, generator=g, device=device).cpu()
        T = torch.where(greedy, torch.zeros_like(T), T)
        sig = 0.3 + 1.7 * torch.rand(B, generator=g, device=device).cpu()
        return make_batch_from_params(name, k, T, sig, V, dtype, seed, device, g=g)
    raise KeyError(config)


def workload_bytes(config: str) -> int:
    """Logit bytes the spec formula counts for the fixed-k workloads."""
    c = CONFIGS[config]
    es = 4 if c["dtype"] == torch.float32 else 2
    if c["k"] is None:
        raise ValueError("ragged workload: bytes follow from the drawn k")
    return c["B"] * (2 * c["k"] + 1) * c["V"] * es


__all__ = ["Batch", "CONFIGS", "make_batch", "make_batch_from_params", "workload_bytes",
           "VOCAB_QWEN3"]
