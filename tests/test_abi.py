"""The C ABI library (no GPU): it builds for sm_103a, loads, exports every
function include/specverify.h declares, and rejects bad arguments on the host
before touching the device."""

import ctypes
import os
import re

import pytest

import speculative_decoding_verification_13_gb300 as sv
from speculative_decoding_verification_13_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specverify.h")


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return sv.load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_verify\w*)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    assert "spec_verify" in names and "spec_verify_workspace_size" in names
    assert len(names) >= 6


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_strerror_and_version(lib):
    assert sv.strerror(0) == "ok"
    for code in sv.ERROR_NAMES:
        assert sv.strerror(code) != "unknown status"
    assert lib.spec_verify_version() >= 100


def test_workspace_size():
    a = sv.workspace_size(256, 4096, 3840)
    b = sv.workspace_size(256, 4096, 3840 * 2)
    assert a > 0 and b > a and a % 256 == 0
    assert sv.workspace_size(-1, 0, 0) == 0
    assert sv.workspace_size(0, 0, 0) > 0
    # grows with the candidate lists: at least SV_TOPK_MAX (int32 + double) per row
    assert a >= (4096 + 3840) * sv.SV_TOPK_MAX * 12


def _logits(data, dtype, vocab, rows, stride):
    return sv._Logits(data, dtype, vocab, rows, stride)


def _call(lib, t, d, B, ws=None, nbytes=0, **ptrs):
    P = ctypes.c_void_p
    fake = P(0x1000)  # never dereferenced: every case below fails host-side checks
    args = dict(draft_tokens=fake, k=fake, T=fake, top_k=None, top_p=None, u=fake,
                acc=fake, tok=fake)
    args.update(ptrs)
    return lib.spec_verify(ctypes.byref(t), ctypes.byref(d), args["draft_tokens"], args["k"],
                           args["T"], args["top_k"], args["top_p"], args["u"], args["acc"],
                           args["tok"], None, B, ws, nbytes, None)


def test_host_side_argument_errors(lib):
    P = ctypes.c_void_p
    ok_t = _logits(P(0x10000), 1, 64, 5, 64)
    ok_d = _logits(P(0x20000), 1, 64, 4, 64)
    # unsupported dtype
    assert _call(lib, _logits(P(0x10000), 7, 64, 5, 64), ok_d, 1) == 2
    # mixed dtypes
    assert _call(lib, ok_t, _logits(P(0x20000), 0, 64, 4, 64), 1) == 2
    # vocab mismatch / too large
    assert _call(lib, ok_t, _logits(P(0x20000), 1, 32, 4, 64), 1) == 1
    assert _call(lib, _logits(P(0x10000), 1, (1 << 22) + 1, 5, (1 << 22) + 8),
                 _logits(P(0x20000), 1, (1 << 22) + 1, 4, (1 << 22) + 8), 1) == 2
    # rows inconsistent with the batch: R_t must equal B + R_d
    assert _call(lib, ok_t, ok_d, 2) == 1
    # negative batch
    assert _call(lib, ok_t, ok_d, -1) == 1
    # misaligned data / stride
    assert _call(lib, _logits(P(0x10002), 1, 64, 5, 64), ok_d, 1) == 2
    assert _call(lib, _logits(P(0x10000), 1, 60, 5, 60),
                 _logits(P(0x20000), 1, 60, 4, 60), 1) == 2
    # stride shorter than a row
    assert _call(lib, _logits(P(0x10000), 1, 64, 5, 32), ok_d, 1) == 1
    # missing required pointers
    assert _call(lib, ok_t, ok_d, 1, k=None) == 1
    assert _call(lib, ok_t, ok_d, 1, draft_tokens=None) == 1
    # workspace: missing, misaligned, too small
    assert _call(lib, ok_t, ok_d, 1) == 4
    assert _call(lib, ok_t, ok_d, 1, ws=P(0x30010), nbytes=1 << 30) == 4
    assert _call(lib, ok_t, ok_d, 1, ws=P(0x30000), nbytes=64) == 4
    # an empty batch is a no-op once the workspace is valid
    assert _call(lib, _logits(None, 1, 64, 0, 64), _logits(None, 1, 64, 0, 64), 0,
                 ws=P(0x30000), nbytes=sv.workspace_size(0, 0, 0)) == 0


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    monkeypatch.setattr(sv, "_LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(sv, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        sv.load_library()
