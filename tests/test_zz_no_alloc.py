"""spec_verify_noalloc (library-owned fixed workspace) against spec_verify
(caller workspace) on the same inputs, through the C ABI.  The two run the same
kernels, so emitted tokens and accept lengths must agree exactly and (p, q)
within the floating-point tolerance of the parity tests; each case makes two
allocation-free calls in a row so that state left in the shared buffer by one
call cannot leak into the next, and the buffer is filled with 0xFF bytes
before the first of them (nothing in it has to start at zero).  Collected
last on purpose: it must pass alone and after every other test in the
session."""

import pytest
import torch

import speculative_decoding_verification_13_gb300 as sv
from speculative_decoding_verification_13_gb300 import workloads

pytestmark = pytest.mark.gpu

PQ_RTOL = {torch.float32: 1e-5, torch.bfloat16: 2e-3}


def _outputs(b, device):
    B = b.k_per_req.numel()
    return (torch.full((B,), -7, dtype=torch.int32, device=device),
            torch.full((b.target.shape[0],), -7, dtype=torch.int32, device=device),
            torch.full((b.draft.shape[0], 2), -7.0, dtype=torch.float64, device=device))


CASES = [("c1", "t1", None), ("c2", "t0.7", None), ("c2", "greedy", None), ("c3", "s1", 8),
         ("c4", "default", 16), ("c5", "default", 40)]


@pytest.mark.parametrize("config,variant,batch", CASES)
def test_noalloc_matches_workspace_path(config, variant, batch):
    dev = torch.device("cuda")
    b = workloads.make_batch(config, variant, device=dev, batch=batch)
    args = (b.target, b.draft, b.draft_tokens, b.k_per_req, b.temperature, b.uniforms,
            b.top_k, b.top_p)
    acc0, tok0, pq0 = _outputs(b, dev)
    sv.Verifier(dev)(*args, out_accept_len=acc0, out_tokens=tok0, out_pq=pq0)
    torch.cuda.synchronize()
    # the buffer is documented to need no zeroing: fill it with junk first
    _fill_scratch(0xFF)
    for _ in range(2):
        acc1, tok1, pq1 = _outputs(b, dev)
        sv.verify_noalloc(*args, out_accept_len=acc1, out_tokens=tok1, out_pq=pq1)
        torch.cuda.synchronize()
        ptr, nbytes = sv.noalloc_scratch()
        assert nbytes == sv.SV_NOALLOC_SCRATCH_BYTES and ptr % 256 == 0
        code, _, _ = sv.get_error(_ScratchView(ptr))
        assert code == 0
        assert torch.equal(acc0, acc1)
        assert torch.equal(tok0, tok1)
        nan0, nan1 = torch.isnan(pq0), torch.isnan(pq1)
        assert torch.equal(nan0, nan1)
        tol = PQ_RTOL[b.target.dtype]
        ok = ~nan0
        assert torch.allclose(pq1[ok], pq0[ok], rtol=tol, atol=0.0)


def _fill_scratch(byte):
    """Overwrite the library's whole buffer, seen through its device address
    as a byte tensor (the CUDA array interface wraps the address; nothing is
    allocated)."""
    ptr, nbytes = sv.noalloc_scratch()

    class _Raw:
        __cuda_array_interface__ = {"shape": (nbytes,), "typestr": "|u1",
                                    "data": (ptr, False), "version": 3}

    view = torch.as_tensor(_Raw(), device="cuda")
    assert view.data_ptr() == ptr and view.numel() == nbytes
    view.fill_(byte)
    torch.cuda.synchronize()


class _ScratchView:
    """Stands in for a workspace tensor: get_error only needs data_ptr()."""

    def __init__(self, ptr):
        self.ptr = ptr

    def data_ptr(self):
        return self.ptr


def test_noalloc_rejects_batches_beyond_its_buffer():
    dev = torch.device("cuda")
    B, k, V = 64, 31, 64  # 64 * 32 + 64 * 31 rows need more than the fixed buffer
    Rt, Rd = B * (k + 1), B * k
    assert sv.workspace_size(B, Rt, Rd) > sv.SV_NOALLOC_SCRATCH_BYTES
    target = torch.zeros(Rt, V, dtype=torch.bfloat16, device=dev)
    draft = torch.zeros(Rd, V, dtype=torch.bfloat16, device=dev)
    kk = torch.full((B,), k, dtype=torch.int32, device=dev)
    acc = torch.full((B,), -7, dtype=torch.int32, device=dev)
    tok = torch.full((Rt,), -7, dtype=torch.int32, device=dev)
    with pytest.raises(sv.SpecVerifyError) as e:
        sv.verify_noalloc(target, draft, torch.zeros(Rd, dtype=torch.int32, device=dev), kk,
                          torch.ones(B, device=dev), torch.rand(Rt, device=dev),
                          out_accept_len=acc, out_tokens=tok)
    assert e.value.code == 4  # SV_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert (acc == -7).all() and (tok == -7).all()  # nothing was enqueued
