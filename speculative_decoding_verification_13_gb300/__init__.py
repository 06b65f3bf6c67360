"""GB300-native batched speculative-decoding verification.

Python binding of ``libspecverify.so`` (C ABI declared in
``include/specverify.h``).  This module only marshals arguments: every step of
verification runs in the library's sm_103a kernels.  PyTorch supplies device
memory and streams.  There is no CPU fallback: if the library has not been
built, importing the binding's entry points raises.

Typical use::

    import speculative_decoding_verification_13_gb300 as sv
    accept_len, tokens = sv.verify(target, draft, draft_tokens, k_per_req,
                                   temperature, uniforms, top_k=top_k, top_p=top_p)

Row layout (see the header): request b owns target rows t_off[b]..t_off[b]+k_b
(t_off[b] = sum_{j<b}(k_j+1)) and draft rows t_off[b]-b..; ``uniforms`` and the
returned ``tokens`` use the target-row layout.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = ["verify", "Verifier", "workspace_size", "get_error", "dump_rows", "strerror",
           "library_path", "SpecVerifyError", "SV_TOPK_MAX", "SV_MAX_K", "verify_noalloc",
           "noalloc_scratch", "SV_NOALLOC_SCRATCH_BYTES", "DraftSampler", "draft_sample", "kv_commit",
           "kv_commit_error", "lmhead_stats", "lmhead_stats_error",
           "adapt_k", "verify_greedy_from_argmax", "verify_greedy_error"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_lib", "libspecverify.so")

SV_OK = 0
SV_F32, SV_BF16 = 0, 1
SV_MAX_K = 32
SV_TOPK_MAX = 256
SV_VOCAB_MAX = 1 << 22
SV_NOALLOC_SCRATCH_BYTES = 16 << 20

ERROR_NAMES = {
    0: "SV_OK", 1: "SV_ERR_ARG", 2: "SV_ERR_UNSUPPORTED", 3: "SV_ERR_CUDA",
    4: "SV_ERR_WORKSPACE", 16: "SV_ERR_DATA_K", 17: "SV_ERR_DATA_TEMPERATURE",
    18: "SV_ERR_DATA_TOP_P", 19: "SV_ERR_DATA_TOP_K", 20: "SV_ERR_DATA_TOKEN",
    21: "SV_ERR_DATA_ROWS", 22: "SV_ERR_DATA_LOGIT", 23: "SV_ERR_DATA_NO_DRAFT",
    24: "SV_ERR_TIMEOUT", 25: "SV_ERR_INTERNAL",
}


class SpecVerifyError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}{': ' if what else ''}{ERROR_NAMES.get(code, code)} "
                         f"({strerror(code)})")


class _Logits(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("rows", ctypes.c_int64),
                ("row_stride", ctypes.c_int64)]


class _Options(ctypes.Structure):
    _fields_ = [("out_pq", ctypes.c_void_p), ("event_rowpass_begin", ctypes.c_void_p),
                ("event_rowpass_end", ctypes.c_void_p), ("test_expire_wait", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class _KvCache(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("num_pages", ctypes.c_int64),
                ("n_layers", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("entry_elems", ctypes.c_int32), ("elem_bytes", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libspecverify.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"{_LIB_PATH} is missing: build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'` "
                    "(the CUDA library is required; there is no fallback)")
            lib = ctypes.CDLL(_LIB_PATH)
            P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
            lib.spec_verify_workspace_size.restype = sz
            lib.spec_verify_workspace_size.argtypes = [i32, i64, i64]
            lib.spec_verify.restype = ctypes.c_int
            lib.spec_verify.argtypes = [ctypes.POINTER(_Logits), ctypes.POINTER(_Logits),
                                        P, P, P, P, P, P, P, P, P, i32, P, sz,
                                        ctypes.POINTER(_Options)]
            lib.spec_verify_get_error.restype = ctypes.c_int
            lib.spec_verify_get_error.argtypes = [P, P, P, P, P]
            lib.spec_verify_dump_rows.restype = ctypes.c_int
            lib.spec_verify_dump_rows.argtypes = [P, sz, i32, i64, i64, P, P, P, P, P]
            lib.spec_verify_strerror.restype = ctypes.c_char_p
            lib.spec_verify_strerror.argtypes = [ctypes.c_int]
            lib.spec_verify_version.restype = ctypes.c_int
            lib.spec_verify_version.argtypes = []
            lib.spec_draft_sample_workspace_size.restype = sz
            lib.spec_draft_sample_workspace_size.argtypes = [i32, i64]
            lib.spec_draft_sample.restype = ctypes.c_int
            lib.spec_draft_sample.argtypes = [ctypes.POINTER(_Logits), P, P, P, P, P, P, P, P,
                                              i32, P, sz, ctypes.POINTER(_Options)]
            lib.spec_lmhead_stats_workspace_size.restype = sz
            lib.spec_lmhead_stats_workspace_size.argtypes = [i32, i32]
            lib.spec_lmhead_stats.restype = ctypes.c_int
            lib.spec_lmhead_stats.argtypes = [P, P, i32, i32, i32, P, P, P, P, P, P, P, P, sz]
            lib.spec_adapt_k.restype = ctypes.c_int
            lib.spec_adapt_k.argtypes = [P, P, P, P, ctypes.c_double, ctypes.c_double, i32, i32,
                                         P, P, P, i32]
            lib.spec_kv_commit_workspace_size.restype = sz
            lib.spec_kv_commit_workspace_size.argtypes = [i32]
            lib.spec_kv_commit.restype = ctypes.c_int
            lib.spec_kv_commit.argtypes = [ctypes.POINTER(_KvCache), P, i32, P, P, P, P, i32, P,
                                           i32, P, sz]
            _lib = lib
    return _lib


def strerror(code: int) -> str:
    return load_library().spec_verify_strerror(int(code)).decode()


def workspace_size(batch: int, target_rows: int, draft_rows: int) -> int:
    return int(load_library().spec_verify_workspace_size(int(batch), int(target_rows),
                                                         int(draft_rows)))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _event_handle(ev, stream):
    """cudaEvent_t of a torch.cuda.Event (torch creates the event lazily on its
    first record; the library re-records it where the row pass starts / ends)."""
    if ev is None:
        return None
    if ev.cuda_event == 0:
        ev.record(stream if stream is not None else torch.cuda.current_stream())
    return ctypes.c_void_p(ev.cuda_event)


def _check(t, name, dtype, ndim=1):
    if t is None:
        return
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimension(s)")
    if ndim == 1 and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _check_verify_args(target, draft, draft_tokens, k_per_req, temperature, uniforms, top_k,
                       top_p, out_accept_len, out_tokens, out_pq, Rt, Rd):
    """Lengths, dtypes and devices of spec_verify's arguments, checked before
    the call: the library reads and writes these buffers on the GPU with the
    lengths that B, R_t and R_d imply, so a short or misplaced tensor would be
    read or written past its end."""
    B = int(k_per_req.numel())
    dev = target.device
    need = {"k_per_req": (k_per_req, B), "temperature": (temperature, B),
            "uniforms": (uniforms, Rt), "draft_tokens": (draft_tokens, Rd),
            "top_k": (top_k, B), "top_p": (top_p, B),
            "out_accept_len": (out_accept_len, B), "out_tokens": (out_tokens, Rt)}
    for name, (t, n) in need.items():
        if t is None:
            if name == "draft_tokens" and Rd == 0:
                continue
            if name in ("top_k", "top_p"):
                continue
            raise ValueError(f"{name} is required")
        if t.device != dev:
            raise ValueError(f"{name} is on {t.device}, the logits on {dev}")
        if t.numel() < n:
            raise ValueError(f"{name} holds {t.numel()} elements, {n} are needed")
    if draft is not None and draft.device != dev:
        raise ValueError(f"draft logits are on {draft.device}, the target logits on {dev}")
    if out_pq is not None:
        if not isinstance(out_pq, torch.Tensor) or out_pq.device != dev:
            raise ValueError("out_pq must be a CUDA tensor on the logits' device")
        if out_pq.dtype != torch.float64 or not out_pq.is_contiguous():
            raise TypeError("out_pq must be a contiguous float64 tensor")
        if out_pq.numel() < 2 * Rd:
            raise ValueError(f"out_pq holds {out_pq.numel()} elements, {2 * Rd} are needed")


def _logits_desc(x, V=None):
    if x is None:
        return _Logits(None, SV_BF16, V or 0, 0, V or 0)
    if not isinstance(x, torch.Tensor) or not x.is_cuda or x.dim() != 2:
        raise TypeError("logits must be 2-D CUDA tensors")
    if x.dtype == torch.bfloat16:
        dt = SV_BF16
    elif x.dtype == torch.float32:
        dt = SV_F32
    else:
        raise TypeError(f"logits must be float32 or bfloat16, got {x.dtype}")
    if x.stride(1) != 1:
        raise ValueError("logit rows must be contiguous")
    rows, V = x.shape
    stride = x.stride(0) if rows > 1 else V
    return _Logits(x.data_ptr() if x.numel() else None, dt, V, rows, stride)


class Verifier:
    """Reusable caller-side state: a workspace sized for the largest batch seen
    and the output buffers.  One Verifier per stream (workspaces must not be
    shared by calls that can overlap)."""

    def __init__(self, device=None):
        self.device = torch.device(device or "cuda")
        self.workspace = None

    def _workspace(self, B, Rt, Rd):
        need = workspace_size(B, Rt, Rd)
        if need == 0 and (B or Rt or Rd):
            raise SpecVerifyError(1, "workspace_size")
        if self.workspace is None or self.workspace.numel() < need:
            self.workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=self.device)
        return self.workspace

    def __call__(self, target, draft, draft_tokens, k_per_req, temperature, uniforms,
                 top_k=None, top_p=None, *, out_accept_len=None, out_tokens=None,
                 out_pq=None, stream=None, rowpass_events=None, test_expire_wait=False):
        """test_expire_wait: test of the timeout path only (one bounded wait of
        the row pass expires; the first listed row's request fails with
        SV_ERR_TIMEOUT)."""
        lib = load_library()
        B = int(k_per_req.shape[0])
        _check(k_per_req, "k_per_req", torch.int32)
        _check(temperature, "temperature", torch.float32)
        _check(uniforms, "uniforms", torch.float32)
        _check(draft_tokens, "draft_tokens", torch.int32)
        _check(top_k, "top_k", torch.int32)
        _check(top_p, "top_p", torch.float32)
        td = _logits_desc(target)
        dd = _logits_desc(draft, td.vocab)
        if draft is None:
            dd.rows = td.rows - B
            dd.dtype = td.dtype
        Rt, Rd = int(td.rows), int(dd.rows)
        if out_accept_len is None:
            out_accept_len = torch.empty(B, dtype=torch.int32, device=target.device)
        if out_tokens is None:
            out_tokens = torch.empty(Rt, dtype=torch.int32, device=target.device)
        _check(out_accept_len, "out_accept_len", torch.int32)
        _check(out_tokens, "out_tokens", torch.int32)
        _check_verify_args(target, draft, draft_tokens, k_per_req, temperature, uniforms, top_k,
                           top_p, out_accept_len, out_tokens, out_pq, Rt, Rd)
        if self.workspace is not None and self.workspace.device != target.device:
            raise ValueError(f"this Verifier's workspace is on {self.workspace.device}, "
                             f"the logits on {target.device}")
        with torch.cuda.device(target.device):
            ws = self._workspace(B, Rt, Rd)
            opts = None
            if out_pq is not None or rowpass_events is not None or test_expire_wait:
                ev0, ev1 = rowpass_events if rowpass_events is not None else (None, None)
                opts = _Options(_ptr(out_pq), _event_handle(ev0, stream),
                                _event_handle(ev1, stream), 1 if test_expire_wait else 0, 0)
            rc = lib.spec_verify(ctypes.byref(td), ctypes.byref(dd), _ptr(draft_tokens),
                                 _ptr(k_per_req), _ptr(temperature), _ptr(top_k), _ptr(top_p),
                                 _ptr(uniforms), _ptr(out_accept_len), _ptr(out_tokens),
                                 _stream_handle(stream), B, _ptr(ws), ws.numel(),
                                 ctypes.byref(opts) if opts is not None else None)
        if rc != SV_OK:
            raise SpecVerifyError(rc, "spec_verify")
        return out_accept_len, out_tokens

    def error(self, stream=None):
        return get_error(self.workspace, stream)

    def dump(self, batch, target_rows, draft_rows, stream=None):
        return dump_rows(self.workspace, batch, target_rows, draft_rows, stream)


class DraftSampler:
    """Draft-side sampler (the drafter's token choice whose drafts Verifier
    checks): x_i drawn from the temperature softmax of drafter row i, filtered
    by the request's top-k / top-p as verification filters, by inverse CDF in
    index order with u_i; argmax at temperature 0.  Rows are laid out like the
    verifier's draft rows.  One DraftSampler per stream."""

    def __init__(self, device=None):
        self.device = torch.device(device or "cuda")
        self.workspace = None

    def _workspace(self, B, R):
        need = int(load_library().spec_draft_sample_workspace_size(int(B), int(R)))
        if need == 0 and (B or R):
            raise SpecVerifyError(1, "spec_draft_sample_workspace_size")
        if self.workspace is None or self.workspace.numel() < need:
            self.workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=self.device)
        return self.workspace

    def __call__(self, logits, k_per_req, temperature, uniforms, top_k=None, top_p=None, *,
                 out_tokens=None, out_q=None, with_q=False, stream=None, rowpass_events=None):
        """Returns ``(tokens [R] int32, q [R] float32 or None)`` on the device."""
        lib = load_library()
        B = int(k_per_req.shape[0])
        _check(k_per_req, "k_per_req", torch.int32)
        _check(temperature, "temperature", torch.float32)
        _check(uniforms, "uniforms", torch.float32)
        _check(top_k, "top_k", torch.int32)
        _check(top_p, "top_p", torch.float32)
        xd = _logits_desc(logits)
        R = int(xd.rows)
        if out_tokens is None:
            out_tokens = torch.empty(R, dtype=torch.int32, device=logits.device)
        _check(out_tokens, "out_tokens", torch.int32)
        if out_q is None and with_q:
            out_q = torch.empty(R, dtype=torch.float32, device=logits.device)
        _check(out_q, "out_q", torch.float32)
        ws = self._workspace(B, R)
        opts = None
        if rowpass_events is not None:
            ev0, ev1 = rowpass_events
            opts = _Options(None, _event_handle(ev0, stream), _event_handle(ev1, stream), 0, 0)
        rc = lib.spec_draft_sample(ctypes.byref(xd), _ptr(k_per_req), _ptr(temperature),
                                   _ptr(top_k), _ptr(top_p), _ptr(uniforms), _ptr(out_tokens),
                                   _ptr(out_q), _stream_handle(stream), B, _ptr(ws), ws.numel(),
                                   ctypes.byref(opts) if opts is not None else None)
        if rc != SV_OK:
            raise SpecVerifyError(rc, "spec_draft_sample")
        return out_tokens, out_q

    def error(self, stream=None):
        return get_error(self.workspace, stream)


_default = {}
_default_sampler = {}


_greedy_ws = {}


def verify_greedy_from_argmax(target_argmax, draft_tokens, k_per_req, vocab, *,
                              out_accept_len=None, out_tokens=None, stream=None):
    """Greedy verification from each target row's argmax (e.g. the out_argmax
    of :func:`lmhead_stats`), so that the logits need not exist.  Returns
    ``(accept_len [B] int32, tokens [R_t] int32)`` on the device."""
    lib = load_library()
    f = lib.spec_verify_greedy_from_argmax
    if f.argtypes is None:
        P = ctypes.c_void_p
        f.restype = ctypes.c_int
        f.argtypes = [P, P, P, P, P, P, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, P,
                      ctypes.c_size_t]
        lib.spec_verify_greedy_workspace_size.restype = ctypes.c_size_t
        lib.spec_verify_greedy_workspace_size.argtypes = []
    _check(target_argmax, "target_argmax", torch.int32)
    _check(draft_tokens, "draft_tokens", torch.int32)
    _check(k_per_req, "k_per_req", torch.int32)
    B, Rt = int(k_per_req.numel()), int(target_argmax.numel())
    dev = target_argmax.device
    for t, n, name in ((draft_tokens, Rt - B, "draft_tokens"), (k_per_req, B, "k_per_req")):
        if t.device != dev or t.numel() < n:
            raise ValueError(f"{name} must be on {dev} with at least {n} elements")
    if out_accept_len is None:
        out_accept_len = torch.empty(B, dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty(Rt, dtype=torch.int32, device=dev)
    _check(out_accept_len, "out_accept_len", torch.int32)
    _check(out_tokens, "out_tokens", torch.int32)
    if out_accept_len.numel() < B or out_tokens.numel() < Rt:
        raise ValueError("output tensors are too short")
    key = dev.index if dev.index is not None else torch.cuda.current_device()
    need = int(lib.spec_verify_greedy_workspace_size())
    ws = _greedy_ws.get(key)
    if ws is None or ws.numel() < need:
        ws = _greedy_ws[key] = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        rc = f(_ptr(target_argmax), _ptr(draft_tokens), _ptr(k_per_req), _ptr(out_accept_len),
               _ptr(out_tokens), _stream_handle(stream), B, Rt, int(vocab), _ptr(ws), ws.numel())
    if rc != SV_OK:
        raise SpecVerifyError(rc, "spec_verify_greedy_from_argmax")
    return out_accept_len, out_tokens


def verify_greedy_error(stream=None, device=None):
    """First data error of the last verify_greedy_from_argmax on this device."""
    d = torch.device(device or "cuda")
    return get_error(_greedy_ws[d.index if d.index is not None else torch.cuda.current_device()],
                     stream)


def adapt_k(accept_len, k_used, succ, fail, decay=0.9, c=0.1, k_min=1, k_max=16,
            with_alpha=False, stream=None):
    """Next speculation length per request from its measured acceptance
    (updates succ / fail in place).  Returns (k_next [B] int32, alpha or None)."""
    lib = load_library()
    _check(accept_len, "accept_len", torch.int32)
    _check(k_used, "k_used", torch.int32)
    _check(succ, "succ", torch.float64)
    _check(fail, "fail", torch.float64)
    B = int(accept_len.shape[0])
    k_next = torch.empty(B, dtype=torch.int32, device=accept_len.device)
    alpha = torch.empty(B, dtype=torch.float32, device=accept_len.device) if with_alpha else None
    rc = lib.spec_adapt_k(_ptr(accept_len), _ptr(k_used), _ptr(succ), _ptr(fail), float(decay),
                          float(c), int(k_min), int(k_max), _ptr(k_next), _ptr(alpha),
                          _stream_handle(stream), B)
    if rc != SV_OK:
        raise SpecVerifyError(rc, "spec_adapt_k")
    return k_next, alpha


_lm_ws = {}


def lmhead_stats(hidden, unembed, temperature, tokens=None, stream=None):
    """Verification statistics of the logits hidden @ unembed.T, computed in the
    tensor-core GEMM's epilogue (the logits are never stored).  hidden [M, d]
    and unembed [V, d] bf16 CUDA tensors; temperature [M] float32; tokens [M]
    int32 or None.  Returns (max [M] f32, sum [M] f64, argmax [M] i32,
    token logit [M] f32)."""
    lib = load_library()
    for t, n in ((hidden, "hidden"), (unembed, "unembed")):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.bfloat16 \
                or t.dim() != 2 or not t.is_contiguous():
            raise TypeError(f"{n} must be a contiguous 2-D bfloat16 CUDA tensor")
    _check(temperature, "temperature", torch.float32)
    _check(tokens, "tokens", torch.int32)
    M, d = hidden.shape
    V = unembed.shape[0]
    if unembed.shape[1] != d:
        raise ValueError("hidden and unembed must share d")
    dev = hidden.device
    out_m = torch.empty(M, dtype=torch.float32, device=dev)
    out_s = torch.empty(M, dtype=torch.float64, device=dev)
    out_a = torch.empty(M, dtype=torch.int32, device=dev)
    out_x = torch.empty(M, dtype=torch.float32, device=dev)
    need = int(lib.spec_lmhead_stats_workspace_size(M, V))
    key = dev.index if dev.index is not None else torch.cuda.current_device()
    ws = _lm_ws.get(key)
    if ws is None or ws.numel() < need:
        ws = _lm_ws[key] = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    rc = lib.spec_lmhead_stats(_ptr(hidden), _ptr(unembed), M, V, d, _ptr(temperature),
                               _ptr(tokens), _ptr(out_m), _ptr(out_s), _ptr(out_a), _ptr(out_x),
                               _stream_handle(stream), _ptr(ws), ws.numel())
    if rc != SV_OK:
        raise SpecVerifyError(rc, "spec_lmhead_stats")
    return out_m, out_s, out_a, out_x


def lmhead_stats_error(stream=None, device=None):
    d = torch.device(device or "cuda")
    return get_error(_lm_ws[d.index if d.index is not None else torch.cuda.current_device()],
                     stream)


_kv_ws = {}


def kv_commit(cache, spec, accept_len, k_per_req, kv_len, block_table, stream=None):
    """Append the accepted K/V entries after verification (in place).

    cache: [num_pages, n_layers, 2, page_size, E] CUDA tensor (2- or 4-byte
    elements); spec: [B, spec_slots, n_layers, 2, E], same dtype; accept_len,
    k_per_req: [B] int32 (accept_len from verify, -1 = leave untouched);
    kv_len: [B] int32, updated in place; block_table: [B, max_pages] int32."""
    lib = load_library()
    for t, n in ((accept_len, "accept_len"), (k_per_req, "k_per_req"), (kv_len, "kv_len")):
        _check(t, n, torch.int32)
    _check(block_table, "block_table", torch.int32, ndim=2)
    if block_table is not None and not block_table.is_contiguous():
        raise ValueError("block_table must be contiguous")
    if cache.dim() != 5 or spec.dim() != 5 or not cache.is_contiguous() or not spec.is_contiguous():
        raise ValueError("cache and spec must be contiguous 5-D tensors")
    if cache.dtype != spec.dtype or cache.element_size() not in (2, 4):
        raise TypeError("cache and spec must share a 2- or 4-byte dtype")
    P_, L_, two, S_, E_ = cache.shape
    B, slots = int(spec.shape[0]), int(spec.shape[1])
    if two != 2 or tuple(spec.shape[2:]) != (L_, 2, E_):
        raise ValueError("spec must be [B, slots, n_layers, 2, E] matching the cache")
    desc = _KvCache(cache.data_ptr(), P_, L_, S_, E_, cache.element_size())
    dev = cache.device.index if cache.device.index is not None else torch.cuda.current_device()
    need = int(lib.spec_kv_commit_workspace_size(B))
    ws = _kv_ws.get(dev)
    if ws is None or ws.numel() < need:
        ws = _kv_ws[dev] = torch.empty(max(need, 256), dtype=torch.uint8, device=cache.device)
    rc = lib.spec_kv_commit(ctypes.byref(desc), _ptr(spec), slots, _ptr(accept_len),
                            _ptr(k_per_req), _ptr(kv_len), _ptr(block_table),
                            int(block_table.shape[1]) if block_table is not None else 0,
                            _stream_handle(stream), B, _ptr(ws), ws.numel())
    if rc != SV_OK:
        raise SpecVerifyError(rc, "spec_kv_commit")
    return kv_len


def kv_commit_error(stream=None, device=None):
    """First data error of the last kv_commit on this device."""
    d = torch.device(device or "cuda")
    return get_error(_kv_ws[d.index if d.index is not None else torch.cuda.current_device()],
                     stream)


def draft_sample(logits, k_per_req, temperature, uniforms, top_k=None, top_p=None, **kw):
    """One-shot draft-side sampling with a per-device cached DraftSampler."""
    dev = logits.device
    s = _default_sampler.get(dev)
    if s is None:
        s = _default_sampler[dev] = DraftSampler(dev)
    return s(logits, k_per_req, temperature, uniforms, top_k, top_p, **kw)


def verify(target, draft, draft_tokens, k_per_req, temperature, uniforms, top_k=None,
           top_p=None, **kw):
    """One-shot verification with a per-device cached Verifier.  Returns
    ``(accept_len [B] int32, tokens [R_t] int32)`` on the device."""
    dev = target.device
    v = _default.get(dev)
    if v is None:
        v = _default[dev] = Verifier(dev)
    return v(target, draft, draft_tokens, k_per_req, temperature, uniforms, top_k, top_p, **kw)


def get_error(workspace, stream=None):
    """Synchronise and return ``(code, request, row)`` of the first data error."""
    code, req, row = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int64()
    rc = load_library().spec_verify_get_error(_ptr(workspace), _stream_handle(stream),
                                              ctypes.byref(code), ctypes.byref(req),
                                              ctypes.byref(row))
    if rc != SV_OK:
        raise SpecVerifyError(rc, "spec_verify_get_error")
    return code.value, req.value, row.value


def dump_rows(workspace, batch, target_rows, draft_rows, stream=None):
    """Per-row intermediate results of the last call (host tensors)."""
    R = target_rows + draft_rows
    stats = torch.empty(R, 5, dtype=torch.float64)
    kept = torch.empty(R, dtype=torch.int32)
    kidx = torch.empty(R, SV_TOPK_MAX, dtype=torch.int32)
    kp = torch.empty(R, SV_TOPK_MAX, dtype=torch.float64)
    rc = load_library().spec_verify_dump_rows(_ptr(workspace), workspace.numel(), batch,
                                              target_rows, draft_rows, _stream_handle(stream),
                                              _ptr(stats), _ptr(kept), _ptr(kidx), _ptr(kp))
    if rc != SV_OK:
        raise SpecVerifyError(rc, "spec_verify_dump_rows")
    return dict(stats=stats, kept_count=kept, kept_idx=kidx, kept_p=kp)


def _noalloc_lib():
    lib = load_library()
    f = lib.spec_verify_noalloc
    if f.argtypes is None:
        P = ctypes.c_void_p
        f.restype = ctypes.c_int
        f.argtypes = [ctypes.POINTER(_Logits), ctypes.POINTER(_Logits), P, P, P, P, P, P, P, P,
                      P, ctypes.c_int32, ctypes.POINTER(_Options)]
        g = lib.spec_verify_noalloc_scratch
        g.restype = ctypes.c_int
        g.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_size_t)]
    return lib


def noalloc_scratch():
    """``(device address, bytes)`` of the current device's library-owned buffer
    used by :func:`verify_noalloc`."""
    ptr, nbytes = ctypes.c_void_p(), ctypes.c_size_t()
    rc = _noalloc_lib().spec_verify_noalloc_scratch(ctypes.byref(ptr), ctypes.byref(nbytes))
    if rc != SV_OK:
        raise SpecVerifyError(rc, "spec_verify_noalloc_scratch")
    return ptr.value, nbytes.value


def verify_noalloc(target, draft, draft_tokens, k_per_req, temperature, uniforms, top_k=None,
                   top_p=None, *, out_accept_len, out_tokens, out_pq=None, stream=None):
    """spec_verify_noalloc: verification with the library's own fixed buffer as
    workspace.  The outputs are caller-provided (nothing is allocated here);
    calls that can overlap on one device race on the shared buffer."""
    lib = _noalloc_lib()
    B = int(k_per_req.shape[0])
    for t, name, dt in ((k_per_req, "k_per_req", torch.int32),
                        (temperature, "temperature", torch.float32),
                        (uniforms, "uniforms", torch.float32),
                        (draft_tokens, "draft_tokens", torch.int32),
                        (top_k, "top_k", torch.int32), (top_p, "top_p", torch.float32),
                        (out_accept_len, "out_accept_len", torch.int32),
                        (out_tokens, "out_tokens", torch.int32)):
        _check(t, name, dt)
    td = _logits_desc(target)
    dd = _logits_desc(draft, td.vocab)
    if draft is None:
        dd.rows = td.rows - B
        dd.dtype = td.dtype
    _check_verify_args(target, draft, draft_tokens, k_per_req, temperature, uniforms, top_k,
                       top_p, out_accept_len, out_tokens, out_pq, int(td.rows), int(dd.rows))
    opts = _Options(_ptr(out_pq), None, None, 0, 0) if out_pq is not None else None
    # the library looks up the buffer of the current device: make it the
    # logits' device
    with torch.cuda.device(target.device):
        rc = lib.spec_verify_noalloc(ctypes.byref(td), ctypes.byref(dd), _ptr(draft_tokens),
                                     _ptr(k_per_req), _ptr(temperature), _ptr(top_k),
                                     _ptr(top_p), _ptr(uniforms), _ptr(out_accept_len),
                                     _ptr(out_tokens), _stream_handle(stream), B,
                                     ctypes.byref(opts) if opts is not None else None)
    if rc != SV_OK:
        raise SpecVerifyError(rc, "spec_verify_noalloc")
    return out_accept_len, out_tokens
