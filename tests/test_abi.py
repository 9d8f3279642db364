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


def test_binding_constants_match_the_header():
    # the dtype codes and status bits the binding passes and reads are the
    # header's own values
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    enum = dict((k, int(v)) for k, v in re.findall(r"\b(KIME_[A-Z0-9_]+)\s*=\s*(-?\d+)", text))
    for name in ("KIME_F32", "KIME_BF16", "KIME_F32_F16OUT", "KIME_F32_BF16OUT", "KIME_F32_3XTF32"):
        assert getattr(kime, name) == enum[name], name
    defines = dict((k, int(v)) for k, v in re.findall(r"#define\s+(KIME_DEV_[A-Z_]+)\s+(\d+)", text))
    for name, value in defines.items():
        assert getattr(kime, name[len("KIME_"):]) == value, name


def test_package_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "packed_varlen_attention_kime_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f
                assert "kime_oracle" not in src, f


def test_workspace_sizes_are_host_arithmetic(lib):
    # host-only entry point (no GPU): op 3 is op 0 at a 1 KB boundary plus the
    # prepared rows [total, 64 * (heads + 2 * kv_heads)] f16; malformed sizes give 0
    for n, T, H, Hkv in [(1, 1, 1, 1), (64, 20249, 12, 12), (16, 18272, 9, 3), (8, 38690, 16, 16)]:
        op0 = kime.kime_attn_workspace_bytes(0, n, T)
        op3 = kime.kime_attn_workspace_bytes(3, n, T, H, Hkv)
        assert op0 > 0 and op3 == ((op0 + 1023) // 1024) * 1024 + T * 64 * (H + 2 * Hkv) * 2
        assert kime.kime_attn_workspace_bytes(2, n, T) == op0
    assert kime.kime_attn_workspace_bytes(3, 4, 100, 6, 4) == 0  # heads not a multiple of kv_heads
    # op 4 (3xTF32 FP32): the size of op 0 (the kernel reads the qkv rows as
    # they are), with heads and kv_heads checked
    for n, T, H, Hkv in [(1, 1, 1, 1), (2, 20, 2, 2), (64, 20249, 12, 12), (16, 18272, 9, 3)]:
        assert kime.kime_attn_workspace_bytes(4, n, T, H, Hkv) == kime.kime_attn_workspace_bytes(0, n, T)
    assert kime.kime_attn_workspace_bytes(4, 4, 100, 6, 4) == 0
    # op 5 (chunked prefill over prepared rows): op 2 at a 1 KB boundary, the
    # chunk's query rows [total, 64 * heads] f16, a 1 KB boundary, then the
    # widened cache rows [n * kv_heads * cap rounded up to 128, 128] f16
    for n, T, H, Hkv, cap in [(1, 1, 1, 1, 1), (8, 1000, 9, 3, 1600), (32, 17600, 9, 3, 8192), (3, 5, 8, 1, 1000)]:
        op2 = kime.kime_attn_workspace_bytes(2, n, T)
        q_end = ((op2 + 1023) // 1024) * 1024 + T * 64 * H * 2
        cap_pad = (cap + 127) // 128 * 128
        want = ((q_end + 1023) // 1024) * 1024 + n * Hkv * cap_pad * 256
        assert kime.kime_attn_workspace_bytes(5, n, T, H, Hkv, cap) == want
    assert kime.kime_attn_workspace_bytes(5, 4, 100, 6, 4, 512) == 0  # heads not a multiple of kv_heads
    assert kime.kime_attn_workspace_bytes(5, 4, 100, 6, 3, 0) == 0    # no cache rows
    assert kime.kime_attn_workspace_bytes(0, -1, 10) == 0
    assert kime.kime_attn_workspace_bytes(9, 4, 100) == 0
    assert kime.kime_attn_workspace_bytes(1, 128, 0, 9, 3, 8192) > 0
