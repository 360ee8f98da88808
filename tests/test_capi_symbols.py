"""CPU checks of the C ABI: the library builds, loads, exports every symbol
that include/specng.h declares, and rejects bad arguments on the host
before any CUDA work (these calls never reach the device)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specng.h")


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_draft_ngram_gb300 import build as b
    from speculative_decoding_draft_ngram_gb300 import capi
    b.build()
    return capi.load()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s+([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("ngram_update", "ngram_draft", "spec_verify", "spec_append", "specng_get_status"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from speculative_decoding_draft_ngram_gb300 import capi
    for n in _declared():
        assert hasattr(lib, n), n
    assert sorted(capi.EXPORTED) == _declared()


def test_strerror_and_workspace_query(lib):
    assert lib.specng_strerror(0) == b"ok"
    assert b"invalid" in lib.specng_strerror(-1)
    assert lib.spec_verify_workspace_bytes(0, 4, 10) == 0
    n1 = lib.spec_verify_workspace_bytes(64, 4, 262144)
    n2 = lib.spec_verify_workspace_bytes(256, 4, 151936)
    assert n1 > 0 and n2 > 0 and n1 % 256 == 0
    assert lib.spec_verify_workspace_bytes(64, 17, 100) == 0


def test_host_argument_checks(lib):
    from speculative_decoding_draft_ngram_gb300 import capi
    t = ctypes.c_void_p()
    assert lib.specng_ngram_create(ctypes.byref(t), 0, 10, 100, None) == -1
    assert lib.specng_ngram_create(ctypes.byref(t), 4, 1 << 19, 100, None) == -1
    assert b"V outside" in lib.specng_last_error()
    assert lib.ngram_update(None, 8, None, None, None) == -1
    assert lib.ngram_draft(None, None, 8, None, 4, None, None, None, None, None) == -1
    p = capi.VerifyParams(temperature=-1.0).to_c()
    fake = ctypes.c_void_p(0x1000)
    rc = lib.spec_verify(fake, 1, 1, 4, 32, fake, None, fake, None, 0, None, ctypes.byref(p),
                         fake, fake, fake, fake, fake, 1 << 20, None)
    assert rc == -1 and b"temperature" in lib.specng_last_error()
    p = capi.VerifyParams().to_c()
    rc = lib.spec_verify(fake, 1, 1, 4, 32, fake, None, fake, None, 0, None, ctypes.byref(p),
                         fake, fake, fake, fake, ctypes.c_void_p(0x1010), 1 << 20, None)
    assert rc == -2                                           # workspace alignment
    rc = lib.spec_verify(fake, 1, 1, 4, 32, fake, None, fake, None, 0, None, ctypes.byref(p),
                         fake, fake, fake, fake, fake, 16, None)
    assert rc == -5                                           # workspace too small
    rc = lib.spec_verify(fake, 7, 1, 4, 32, fake, None, fake, None, 0, None, ctypes.byref(p),
                         fake, fake, fake, fake, fake, 1 << 20, None)
    assert rc == -1                                           # dtype
    p = capi.VerifyParams(rep_penalty=1.1, rep_window=64).to_c()
    rc = lib.spec_verify(fake, 1, 1, 4, 32, fake, None, fake, None, 0, None, ctypes.byref(p),
                         fake, fake, fake, fake, fake, 1 << 20, None)
    assert rc == -1 and b"penalty" in lib.specng_last_error()
    assert lib.spec_append(None, 8, None, 8, None, None, 1, 4, None) == -1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from speculative_decoding_draft_ngram_gb300 import capi
    monkeypatch.setattr(capi, "_LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(capi, "_lib", None)
    with pytest.raises(capi.SpecngError):
        capi.load()
