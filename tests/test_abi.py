"""The C-ABI library builds for sm_103a, loads, and exports every entry point
that include/cas.h declares. No compute call: this runs without a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", fn)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(cas_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def libcas():
    from bit_level_weight_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_entry_points():
    names = declared_functions()
    for required in ("cas_encode_weights", "cas_encode_kv_append", "cas_draft_gemv", "cas_verify_gemm",
                     "cas_draft_attn_decode", "cas_verify_attn", "cas_decode_draft", "cas_reconstruct"):
        assert required in names


def test_library_exports_every_declared_symbol(libcas):
    missing = [n for n in declared_functions() if not hasattr(libcas, n)]
    assert not missing, missing


def test_host_only_entry_points(libcas):
    libcas.cas_status_str.restype = ctypes.c_char_p
    libcas.cas_status_str.argtypes = [ctypes.c_int]
    assert libcas.cas_status_str(0) == b"ok"
    assert b"128" in libcas.cas_status_str(-2)
    libcas.cas_keep_from_ratio.argtypes = [ctypes.c_double]
    libcas.cas_keep_from_ratio.restype = ctypes.c_int32
    assert libcas.cas_keep_from_ratio(0.5) == 64
    assert libcas.cas_keep_from_ratio(0.3) == 38
    assert libcas.cas_keep_from_ratio(0.0) == 0
    assert libcas.cas_keep_from_ratio(1.0) == 128
    libcas.cas_encode_workspace_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
    libcas.cas_encode_workspace_bytes.restype = ctypes.c_uint64
    assert libcas.cas_encode_workspace_bytes(4096, 4096) > 4 * 4096 * 4 * 4


def test_struct_layout_matches_binding():
    import bit_level_weight_gb300 as cas
    assert ctypes.sizeof(cas.cas_params) == 12
    assert cas.cas_weights.base.offset == 544
    assert ctypes.sizeof(cas.cas_weights) == 784
    assert ctypes.sizeof(cas.cas_kv) == 64 + 256


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import bit_level_weight_gb300 as cas
    monkeypatch.setattr(cas, "_lib", None)
    monkeypatch.setattr(cas, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        cas.lib()
