"""The C ABI library loads and exports every symbol include/kime_attn.h declares
(no compute calls: these run without a GPU), and the Python binding mirrors it."""
import os
import re

import pytest

import packed_varlen_attention_kime_gb300 as kime
from packed_varlen_attention_kime_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kime_attn.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kime_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return kime.load_library()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("kime_attn_varlen", "kime_kv_append", "kime_attn_decode", "kime_attn_workspace_bytes"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_exposes_the_same_names():
    for name in declared_functions():
        if name in ("kime_attn_last_cuda_error", "kime_attn_status_string"):
            continue
        assert callable(getattr(kime, name)), name
    assert set(kime.EXPORTED_SYMBOLS) == set(declared_functions())


def test_package_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "packed_varlen_attention_kime_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f
                assert "kime_oracle" not in src, f
