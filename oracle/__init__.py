"""Oracle for batched speculative-decoding verification and for the draft-side
sampler that produces the tokens it verifies.

TEST INFRASTRUCTURE ONLY.  ``oracle.cpp`` states, in plain single-threaded
double-precision C++, what verification computes (the rejection rule of
"FlashMap: Flow Map Speculative Decoding…" §4, "DFlash" §4 and "Speculative
decoding and multi-token prediction", sections "Draft and verify" and "Why the
output is identical").  This module compiles it with the host C++ compiler and
exposes it through ctypes.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference arm may import it; the CUDA library
never does, and the two share no code.

Logit arrays are 2-D C-contiguous ``[rows, V]`` arrays: numpy float32 /
float64, numpy uint16 holding bfloat16 bit patterns, or CPU torch tensors of
dtype float32 / bfloat16 / float64.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB_DIR = os.path.join(_HERE, "_lib")
_LIB_PATH = os.path.join(_LIB_DIR, "liboracle.so")

DT_F32, DT_BF16, DT_F64 = 0, 1, 2

_lock = threading.Lock()
_handle = None


def build(force: bool = False) -> str:
    """Compile ``oracle.cpp`` into ``_lib/liboracle.so`` (plain -O2, no -ffast-math)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    compile_source(_SRC, tmp)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_variant(path: str):
    """Load a shared library built from (a copy of) ``oracle.cpp`` and declare
    its entry points.  Tests use this to run deliberately mutated copies."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32, i64, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    lib.oracle_verify.restype = i32
    lib.oracle_verify.argtypes = [i32, i32, i32, P, i64, i64, P, i64, i64,
                                  P, P, P, P, P, P, P, P, P, P]
    lib.oracle_verify_trials.restype = i32
    lib.oracle_verify_trials.argtypes = [i32, i32, i32, P, P, f32, i32, f32,
                                         i64, P, P, P, P, P]
    lib.oracle_row_probs.restype = i32
    lib.oracle_row_probs.argtypes = [i32, i32, P, f32, i32, f32, P, P]
    lib.oracle_argmax.restype = i32
    lib.oracle_argmax.argtypes = [i32, i32, P]
    lib.oracle_draft_sample.restype = i32
    lib.oracle_draft_sample.argtypes = [i32, i32, i32, P, i64, i64, P, P, P, P, P, P, P, P]
    return lib


def compile_source(src: str, out: str) -> str:
    """Compile a C++ oracle source file into a shared library at ``out``."""
    subprocess.run(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-fno-fast-math",
                    "-ffp-contract=off", "-o", out, src], check=True)
    return out


def _lib():
    global _handle
    with _lock:
        if _handle is None:
            _handle = load_variant(build())
    return _handle


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def as_logits(x):
    """Return ``(C-contiguous numpy array, dtype code)`` for a logit array."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), DT_BF16
            if x.dtype == torch.float32:
                return x.numpy(), DT_F32
            if x.dtype == torch.float64:
                return x.numpy(), DT_F64
            raise TypeError(f"unsupported logit dtype {x.dtype}")
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, DT_F32
    if x.dtype == np.float64:
        return x, DT_F64
    if x.dtype == np.uint16:
        return x, DT_BF16
    raise TypeError(f"unsupported logit dtype {x.dtype}")


def _np(a, dtype):
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def verify(target, draft, draft_tokens, k_per_req, temperature, top_k=None, top_p=None,
           uniforms=None, threads: int = 1):
    """Verify a whole batch.  Returns a dict with ``accept_len`` [B] int32,
    ``tokens`` [R_t] int32 (-1 padded), ``pq`` [R_d, 2] float64
    (p_i(x_i), q_i(x_i)) and ``margins`` [B, 3] float64 (m_acc, m_cdf, m_topp).

    Request b owns target rows t_off[b]..t_off[b]+k_b, t_off[b] = sum_{j<b}(k_j+1),
    and draft rows t_off[b]-b onwards.  ``threads > 1`` splits the batch into
    contiguous groups of requests evaluated concurrently by the same code.
    """
    tl, dt = as_logits(target)
    dl = None
    if draft is not None:
        dl, dt2 = as_logits(draft)
        if dt2 != dt:
            raise TypeError("target and draft logits must share a dtype")
        if dl.shape[0] == 0:
            dl = None
    k = _np(k_per_req, np.int32)
    T = _np(temperature, np.float32)
    B = int(k.shape[0])
    tk = _np(top_k, np.int32) if top_k is not None else np.zeros(B, np.int32)
    tp = _np(top_p, np.float32) if top_p is not None else np.ones(B, np.float32)
    u = _np(uniforms, np.float32)
    x = _np(draft_tokens, np.int32) if draft_tokens is not None else np.zeros(0, np.int32)
    V = int(tl.shape[1])
    Rt, Rd = int(tl.shape[0]), int(x.shape[0])
    acc = np.full(B, -1, np.int32)
    tok = np.full(max(Rt, 1), -1, np.int32)
    pq = np.full((max(Rd, 1), 2), np.nan)
    mg = np.full((max(B, 1), 3), np.nan)
    lib = _lib()
    t_off = np.concatenate([[0], np.cumsum(k.astype(np.int64) + 1)])
    if t_off[-1] != Rt or (dl is not None and dl.shape[0] != Rd) or int(k.sum()) != Rd:
        rc = lib.oracle_verify(B, V, dt, _ptr(tl), Rt, V, _ptr(dl),
                               Rd, V, _ptr(x), _ptr(k), _ptr(T), _ptr(tk), _ptr(tp),
                               _ptr(u), _ptr(acc), _ptr(tok), _ptr(pq), _ptr(mg))
        return dict(rc=rc, accept_len=acc, tokens=tok[:Rt], pq=pq[:Rd], margins=mg[:B])

    def run(lo, hi):
        r0, r1 = int(t_off[lo]), int(t_off[hi])
        d0, d1 = r0 - lo, r1 - hi
        return lib.oracle_verify(
            hi - lo, V, dt, _ptr(tl[r0:r1]), r1 - r0, V,
            _ptr(dl[d0:d1]) if dl is not None else None, d1 - d0, V,
            _ptr(x[d0:d1]), _ptr(k[lo:hi]), _ptr(T[lo:hi]), _ptr(tk[lo:hi]),
            _ptr(tp[lo:hi]), _ptr(u[r0:r1]), _ptr(acc[lo:hi]), _ptr(tok[r0:r1]),
            _ptr(pq[d0:d1]), _ptr(mg[lo:hi]))

    if threads <= 1 or B <= 1:
        rc = run(0, B)
    else:
        bounds = np.linspace(0, B, min(threads, B) + 1).astype(int)
        with ThreadPoolExecutor(len(bounds) - 1) as ex:
            rcs = list(ex.map(lambda ab: run(*ab), zip(bounds[:-1], bounds[1:])))
        rc = max(rcs)
    return dict(rc=rc, accept_len=acc, tokens=tok[:Rt], pq=pq[:Rd], margins=mg[:B])


def verify_trials(target, draft, temperature, top_k, top_p, draft_tokens, uniforms, lib=None):
    """One request (target [k+1, V], draft [k, V]) against many independent
    trials: ``draft_tokens`` [n, k], ``uniforms`` [n, k+1].  Returns
    ``(accept_len [n], tokens [n, k+1], margins [n, 3])``."""
    tl, dt = as_logits(target)
    k = int(tl.shape[0]) - 1
    dl = None
    if draft is not None and k > 0:
        dl, _ = as_logits(draft)
    x = _np(draft_tokens, np.int32).reshape(-1, k) if k > 0 else \
        np.zeros((np.asarray(uniforms).shape[0], 0), np.int32)
    u = _np(uniforms, np.float32).reshape(-1, k + 1)
    n = int(u.shape[0])
    acc = np.empty(n, np.int32)
    tok = np.empty((n, k + 1), np.int32)
    mg = np.empty((n, 3))
    rc = (lib or _lib()).oracle_verify_trials(int(tl.shape[1]), dt, k, _ptr(tl), _ptr(dl),
                                     float(temperature), int(top_k), float(top_p), n,
                                     _ptr(x), _ptr(u), _ptr(acc), _ptr(tok), _ptr(mg))
    if rc != 0:
        raise ValueError(f"oracle_verify_trials failed with code {rc}")
    return acc, tok, mg


def row_probs(row, temperature, top_k=0, top_p=1.0):
    """Distribution of one row; returns ``(p [V] float64, top-p margin)``."""
    x, dt = as_logits(np.asarray(row)[None] if not hasattr(row, "dim") else row.reshape(1, -1))
    V = int(x.shape[-1])
    p = np.empty(V)
    m = np.empty(1)
    rc = _lib().oracle_row_probs(V, dt, _ptr(x), float(temperature), int(top_k),
                                 float(top_p), _ptr(p), _ptr(m))
    if rc != 0:
        raise ValueError(f"oracle_row_probs failed with code {rc}")
    return p, float(m[0])


def draft_sample(logits, k_per_req, temperature, uniforms, top_k=None, top_p=None,
                 threads: int = 1):
    """Draft-side sampling over drafter rows laid out like the verifier's draft
    rows (request b owns rows d_off[b]..d_off[b]+k_b-1).  Returns a dict with
    ``tokens`` [R] int32 (-1 for failed requests), ``q`` [R] float64
    (q_i(x_i), NaN for greedy / failed rows) and ``margins`` [R, 2]
    (m_cdf, m_topp).  ``threads > 1`` evaluates groups of requests
    concurrently with the same code."""
    xl, dt = as_logits(logits)
    k = _np(k_per_req, np.int32)
    B = int(k.shape[0])
    T = _np(temperature, np.float32)
    tk = _np(top_k, np.int32) if top_k is not None else np.zeros(B, np.int32)
    tp = _np(top_p, np.float32) if top_p is not None else np.ones(B, np.float32)
    u = _np(uniforms, np.float32)
    R, V = int(xl.shape[0]), int(xl.shape[1])
    tok = np.full(max(R, 1), -1, np.int32)
    q = np.full(max(R, 1), np.nan)
    mg = np.full((max(R, 1), 2), np.nan)
    lib = _lib()
    d_off = np.concatenate([[0], np.cumsum(k.astype(np.int64))])

    def run(lo, hi):
        r0, r1 = int(d_off[lo]), int(d_off[hi])
        return lib.oracle_draft_sample(hi - lo, V, dt, _ptr(xl[r0:r1]), r1 - r0, V,
                                       _ptr(k[lo:hi]), _ptr(T[lo:hi]), _ptr(tk[lo:hi]),
                                       _ptr(tp[lo:hi]), _ptr(u[r0:r1]), _ptr(tok[r0:r1]),
                                       _ptr(q[r0:r1]), _ptr(mg[r0:r1]))

    if d_off[-1] != R or threads <= 1 or B <= 1 or (k < 0).any() or (k > 32).any():
        rc = lib.oracle_draft_sample(B, V, dt, _ptr(xl), R, V, _ptr(k), _ptr(T), _ptr(tk),
                                     _ptr(tp), _ptr(u), _ptr(tok), _ptr(q), _ptr(mg))
    else:
        bounds = np.linspace(0, B, min(threads, B) + 1).astype(int)
        with ThreadPoolExecutor(len(bounds) - 1) as ex:
            rc = max(ex.map(lambda ab: run(*ab), zip(bounds[:-1], bounds[1:])))
    return dict(rc=rc, tokens=tok[:R], q=q[:R], margins=mg[:R])


def argmax(row) -> int:
    x, dt = as_logits(np.asarray(row)[None] if not hasattr(row, "dim") else row.reshape(1, -1))
    return int(_lib().oracle_argmax(int(x.shape[-1]), dt, _ptr(x)))
