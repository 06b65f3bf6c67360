"""Oracle of the KV-cache commit after verification.

TEST INFRASTRUCTURE ONLY: the plain definition, in numpy loops, of what the
commit computes.  Only tests/, __graft_entry__.smoke() and bench.py's CPU
baseline may use it; the CUDA library never does.

The pages state the operation in one line each: the serving pipeline of
"FlashMap: Flow Map Speculative Decoding…" (section "Architecture", the target
verification stage) updates the paged KV cache with the accepted tokens, and
"Speculative decoding and multi-token prediction" (section "Practical
guidance") names a KV-cache rollback that does not truncate on rejection as a
bug that breaks the equality of outputs with and without speculation.  They
define no layout, so this one is chosen (the same in the CUDA library):

* the paged cache is ``cache[num_pages, n_layers, 2, page_size, E]`` (K then V,
  E elements per token per layer, e.g. kv_heads * head_dim);
* request b's logical position p lives in page ``block_table[b, p // page_size]``
  at slot ``p % page_size``;
* the verification pass wrote the K/V of its k_b + 1 inputs (the last emitted
  token, whose K/V was not in the cache yet, then the k_b drafts) to
  ``spec[b, j, n_layers, 2, E]``, j = 0..k_b.

Commit with accept length L_b >= 0 appends spec[b, 0..L_b] at positions
kv_len[b] .. kv_len[b] + L_b and sets kv_len[b] += L_b + 1: the rejected
drafts' entries are never written (the rollback truncates).  L_b = -1 (a
request that failed verification) leaves the request untouched.  A request
whose L_b exceeds k_b, or whose destination pages are missing from its block
table (entry < 0 or >= num_pages, or past max_pages), is a data error: nothing
of it is written and its kv_len is unchanged.
"""

from __future__ import annotations

import numpy as np

KV_OK = 0
KV_ERR_ACCEPT = 26   # accept length above k
KV_ERR_PAGE = 27     # a destination page missing from the block table


def kv_commit(spec, accept_len, k_per_req, kv_len, block_table, cache, page_size):
    """Commit in place.  Returns (new kv_len [B] int32, status [B] int32)."""
    spec = np.asarray(spec)
    B = len(accept_len)
    n_pages = cache.shape[0]
    max_pages = block_table.shape[1] if block_table.ndim == 2 else 0
    new_len = np.array(kv_len, dtype=np.int64).copy()
    status = np.zeros(B, np.int32)
    for b in range(B):
        L = int(accept_len[b])
        if L < 0:
            continue
        if L > int(k_per_req[b]):
            status[b] = KV_ERR_ACCEPT
            continue
        n = int(kv_len[b])
        dest = []
        for j in range(L + 1):
            p = n + j
            col = p // page_size
            page = int(block_table[b, col]) if col < max_pages else -1
            if page < 0 or page >= n_pages:
                status[b] = KV_ERR_PAGE
                break
            dest.append((page, p % page_size))
        if status[b]:
            continue
        for j, (page, slot) in enumerate(dest):
            cache[page, :, :, slot, :] = spec[b, j]
        new_len[b] = n + L + 1
    return new_len.astype(np.int32), status
